"""dflash_draft_block_noalloc against dflash_draft_block.

The no-alloc variant serves callers that must not allocate device memory while
drafting: a decode loop recorded by stream capture in global mode (where an
allocation call is an error and breaks the capture), or a process that carves
its device memory once at start-up.  Its attention split-KV scratch lives in a
static 8 MiB device array, and when the split count a draft would choose does
not fit that array it runs with fewer splits, so its results must agree with
the regular draft's on the same state within the bf16 parity tolerance (they
differ only in the fp32 summation order of the split merge), call after call.
A draft that would need a context workspace to grow is refused, not allocated.
This file is collected last.
"""
import numpy as np
import pytest

from synth import CONFIGS, make_weights
from tests.helpers import feats_block, row_rel_err, to_device, top2_gap, upload_weights

pytestmark = pytest.mark.gpu

TOL = 2e-2   # per-row relative logit tolerance of the bf16 parity tests


def _drafter(shape, ctx):
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    W = upload_weights(make_weights(shape))
    dr = DFlashDrafter(DrafterConfig.from_shape(shape), W, shape.batch)
    f = feats_block(shape, ctx, max(ctx), "prefill")
    dr.ctx_append(to_device(f), max(ctx), rows=np.array(ctx, np.int32))
    return dr, W


def _check_against_regular(dr, s, anchors_np, calls=2, capture=False):
    """Draft once with dflash_draft_block, then `calls` times with the no-alloc
    variant on the same state; compare ids and logits, device memory and the
    launch count (the same launches means the split-KV merge ran in every
    layer, i.e. the static scratch was used)."""
    torch = pytest.importorskip("torch")
    B, K = s.batch, s.K
    anchors = to_device(anchors_np)
    d_ref = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    z_ref = torch.zeros((B, K, s.vocab), dtype=torch.float32, device="cuda")
    # a first draft takes the one-time work out of the count (the fp16 weight
    # copies of a draft of 33+ rows)
    dr.draft_block(K, anchor_ids=anchors, draft_ids=d_ref, logits=z_ref)
    n0 = dr.launch_count()
    dr.draft_block(K, anchor_ids=anchors, draft_ids=d_ref, logits=z_ref)
    torch.cuda.synchronize()
    n_regular = dr.launch_count() - n0
    zr = z_ref.cpu().numpy()
    dref = d_ref.cpu().numpy()
    d = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    z = torch.zeros((B, K, s.vocab), dtype=torch.float32, device="cuda")
    free0 = None
    graph = None
    for call in range(calls):
        d.fill_(-1)
        z.zero_()
        n0 = dr.launch_count()
        if capture and call > 0:
            if graph is None:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, capture_error_mode="global"):
                    dr.draft_block_noalloc(K, anchor_ids=anchors, draft_ids=d, logits=z,
                                           stream=torch.cuda.current_stream().cuda_stream)
                d.fill_(-1)
                z.zero_()
            graph.replay()
        else:
            dr.draft_block_noalloc(K, anchor_ids=anchors, draft_ids=d, logits=z)
            assert dr.launch_count() - n0 == n_regular, "the no-alloc draft skipped the split-KV merge"
        torch.cuda.synchronize()
        # the first call on the device looks up the static array, which (with lazy
        # module loading) brings its 8 MiB into existence; later calls take nothing
        if free0 is None:
            free0 = torch.cuda.mem_get_info()[0]
        elif not capture:
            assert torch.cuda.mem_get_info()[0] == free0
        zn = z.cpu().numpy()
        dn = d.cpu().numpy()
        for b in range(B):
            assert row_rel_err(zn[b], zr[b]).max() <= TOL
            # the two differ only in fp32 rounding: every id whose top-2 gap is not
            # itself at rounding level must agree
            ok = top2_gap(zr[b]) > 1e-4 * np.abs(zr[b]).max(axis=-1)
            assert np.array_equal(dn[b][ok], dref[b][ok])
    assert dr.query_state()["flags"] == 0


def test_noalloc_draft_matches_draft_block_twice():
    pytest.importorskip("torch")
    # head_dim 128 selects the tensor-core attention; a 2048-slot context gives several KV splits
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256,
                                  n_layers=2, batch=2, K=15, K_max=15, seed=31)
    dr, _ = _drafter(s, [2048, 700])
    _check_against_regular(dr, s, np.array([11, 12], np.int32), calls=3)


def test_noalloc_draft_of_a_batch_of_ragged_sequences():
    """16+ sequences: the persistent attention, its partials in the static array."""
    pytest.importorskip("torch")
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256,
                                  n_layers=2, batch=18, K=15, K_max=15, seed=33)
    ctx = [3000, 1, 64, 65, 2047, 300, 9, 1200, 4100, 129, 700, 2, 128, 1500, 63, 2500, 800, 5000]
    dr, _ = _drafter(s, ctx)
    _check_against_regular(dr, s, np.arange(5, 5 + s.batch, dtype=np.int32), calls=2)


def test_noalloc_qwen3_4b_attention_shape():
    """32 query / 8 KV heads of 128, a 2048-token context, K = 16: the regular
    draft picks 17 KV splits (8 x 17 x 128 x 129 floats, more than the static
    array), so the no-alloc draft runs with the 15 that fit."""
    pytest.importorskip("torch")
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=32, n_kv_heads=8, hidden=512,
                                  intermediate=1024, n_layers=2, batch=1, K=16, K_max=16, vocab=2048, seed=33)
    dr, _ = _drafter(s, [2048])
    _check_against_regular(dr, s, np.array([5], np.int32), calls=2)


def test_noalloc_draft_under_global_stream_capture():
    """One eager call (it looks up the static array), then the same call recorded
    by stream capture in global mode -- where any allocation is an error -- and
    replayed: the replays must match the regular draft."""
    pytest.importorskip("torch")
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256,
                                  n_layers=2, batch=2, K=15, K_max=15, seed=34)
    dr, _ = _drafter(s, [1500, 333])
    _check_against_regular(dr, s, np.array([3, 4], np.int32), calls=3, capture=True)


def test_noalloc_refuses_a_draft_that_needs_a_larger_workspace():
    torch = pytest.importorskip("torch")
    from block_diffusion_speculative_dflash_gb300 import DflashError
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256,
                                  n_layers=1, batch=2, K=15, K_max=15, seed=32)
    # a short context keeps the append's GEMM workspace small; a draft of 3
    # masks then sizes it for 8 rows, and 15 masks need about four times more
    dr, _ = _drafter(s, [8, 4])
    dr.draft_block(3, anchor_ids=np.array([1, 2], np.int32))
    with pytest.raises(DflashError) as e:
        dr.draft_block_noalloc(15)
    assert e.value.code == 3            # DFLASH_ERR_CAPACITY
    torch.cuda.synchronize()
    assert dr.query_state()["flags"] == 0
