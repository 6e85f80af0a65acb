"""GPU: the optional execution paths selected at context creation give the
default path's results on the same state -- the mma.sync attention kernel
instead of the tcgen05 one (DFLASH_ATTN_UMMA=0, the kernel of head counts whose
group size does not divide 128), the LM head as one GEMM with the argmax in its
epilogue (DFLASH_LM_FUSED=1) -- and the default path (partial-store LM-head
GEMM + argmax kernel) stays within the oracle's bf16 tolerance; loops with the
appends' K/V projected inside the next draft's QKV GEMMs (DFLASH_FUSE_APPEND=1)
match the oracle."""
import os

import numpy as np
import pytest

import oracle as orc
from synth import CONFIGS, make_weights
from tests.helpers import feats_block, row_rel_err, to_device, upload_weights

pytestmark = pytest.mark.gpu


def _run(s, Wd, ctx, env):
    import torch
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    saved = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, s.batch)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    f = feats_block(s, ctx, max(ctx), "prefill")
    dr.ctx_append(to_device(f), max(ctx), rows=np.array(ctx, np.int32))
    d = torch.zeros((s.batch, s.K), dtype=torch.int32, device="cuda")
    z = torch.zeros((s.batch, s.K, s.vocab), dtype=torch.float32, device="cuda")
    anchors = np.arange(7, 7 + s.batch, dtype=np.int32)
    dr.draft_block(s.K, anchor_ids=anchors, draft_ids=d, logits=z)
    torch.cuda.synchronize()
    st = dr.query_state()
    dr.close()
    return d.cpu().numpy(), z.cpu().numpy(), st, f, anchors


@pytest.mark.parametrize("env", [{"DFLASH_ATTN_UMMA": "0"}, {"DFLASH_LM_FUSED": "1"}])
def test_optional_path_matches_default(env):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=384,
                                  intermediate=768, n_layers=2, batch=2, K=16, K_max=16, seed=51)
    Wn = make_weights(s)
    Wd = upload_weights(Wn)
    ctx = [3000, 1500]   # long enough for several KV splits
    d0, z0, st0, f, anchors = _run(s, Wd, ctx, {})
    d1, z1, st1, _, _ = _run(s, Wd, ctx, env)
    # against the oracle (exact definition) within the bf16 tolerance
    o = orc.OracleDrafter(s, Wn, s.batch)
    for b in range(s.batch):
        o.ctx_append(b, f[b, :ctx[b]])
    od, oz = o.draft(s.K, anchors=list(anchors))
    for z in (z0, z1):
        assert max(row_rel_err(z[b], oz[b]).max() for b in range(s.batch)) <= 2e-2
    # the two paths agree to bf16 accuracy, and on ids where the gap is clear of it
    err = np.stack([row_rel_err(z1[b], z0[b]) for b in range(s.batch)])
    assert err.max() <= 2e-2
    srt = np.sort(z0, axis=-1)
    ok = (srt[..., -1] - srt[..., -2]) > 2 * err * np.max(np.abs(z0), axis=-1)
    assert np.array_equal(d0[ok], d1[ok])
    assert np.array_equal(d1, np.argmax(z1, axis=-1))
    for k in ("ctx_len", "kv_len", "flags"):
        assert np.array_equal(st0[k], st1[k])


@pytest.mark.parametrize("shape_kw,ctx,K", [
    (dict(dtype="bf16", head_dim=128), [64], 15),
    (dict(dtype="bf16", head_dim=128, n_q_heads=8, n_kv_heads=2, hidden=256, n_layers=2, seed=44),
     [700, 5, 1300], 12),
])
def test_fused_append_loop_matches_oracle(shape_kw, ctx, K):
    """DFLASH_FUSE_APPEND=1: each append of <= 128 rows leaves its K/V projection
    to the next draft's QKV GEMMs (the rows ride along as a second token tile).
    Draft + verify + append loops against the oracle: logits, ids where
    decidable, accept lengths and state."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from tests.helpers import SideBySide
    s = CONFIGS["tiny_f32"].with_(K=K, K_max=K, batch=len(ctx), **shape_kw)
    Wn = make_weights(s)
    old = os.environ.get("DFLASH_FUSE_APPEND")
    os.environ["DFLASH_FUSE_APPEND"] = "1"
    try:
        sb = SideBySide(s, Wn, upload_weights(Wn), K=K, ctx=ctx, iterations=4)
    finally:
        if old is None:
            os.environ.pop("DFLASH_FUSE_APPEND", None)
        else:
            os.environ["DFLASH_FUSE_APPEND"] = old
    sb.prefill(list(range(3, 3 + s.batch)))
    for it in range(4):
        sb.step(it, 2e-2)
