"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle.

Tolerances (the drafter's specification, with the reading taken for bf16):
  * logits: per-row ||gpu - oracle||_inf / ||oracle||_inf <= 1e-4 (fp32) or 2e-2 (bf16);
  * the greedy argmax is a decision taken in floating point, so it is checked
    bit-exactly where both sides take it in the same precision: the fused
    LM-head argmax must equal argmax of the kernel's own fp32 logits;
  * end to end, draft ids equal the oracle's wherever its top-2 logit gap
    exceeds 1e-2 and twice that row's measured logit error (bf16 activations
    and a bf16 KV cache carry ~1.5% relative logit error, so a 1e-2 gap alone
    cannot decide a bf16 argmax; in fp32 the error term is ~1e-6); the rows in
    between are counted and reported;
  * accepted lengths, next anchors and state offsets bit-exact;
  * the context KV cache element-wise against the exact oracle, within the
    bound of its bf16 storage;
  * exact ties of the greedy argmax resolve to the lowest token id.
"""
import numpy as np
import pytest

from synth import CONFIGS, context_lengths, make_weights
from tests.helpers import SideBySide, to_device, upload_weights

pytestmark = pytest.mark.gpu

RTOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


_W = {}


def weights(name, torch_cuda):
    if name not in _W:
        _W.clear()
        torch_cuda.cuda.empty_cache()
        s = CONFIGS[name]
        Wn = make_weights(s)
        _W[name] = (Wn, upload_weights(Wn))
    return _W[name]


def test_tiny_f32_loop(torch_cuda):
    s = CONFIGS["tiny_f32"]
    Wn, Wd = weights("tiny_f32", torch_cuda)
    sb = SideBySide(s, Wn, Wd, K=s.K, iterations=6)
    sb.prefill([17])
    for it in range(6):
        sb.step(it, RTOL["f32"], device_rows=(it % 2 == 0))


def test_tiny_f32_batch_ragged(torch_cuda):
    s = CONFIGS["tiny_f32"].with_(batch=5)
    Wn, Wd = weights("tiny_f32", torch_cuda)
    sb = SideBySide(s, Wn, Wd, K=7, ctx=[1, 64, 33, 200, 5], iterations=3)
    sb.prefill([1, 2, 3, 4, 1000])
    for it in range(3):
        sb.step(it, RTOL["f32"])


def test_tiny_bf16_loop(torch_cuda):
    """The tensor-core path on the tiny shape (all GEMMs on tcgen05)."""
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", batch=3, head_dim=128)
    Wn = make_weights(s)
    Wd = upload_weights(Wn)
    sb = SideBySide(s, Wn, Wd, K=15, ctx=[64, 3, 130], iterations=3)
    sb.prefill([17, 5, 900])
    for it in range(3):
        sb.step(it, RTOL["bf16"])


@pytest.mark.parametrize("K,ctx,n_q,n_kv", [
    (15, [2048], 8, 2),                 # one query tile, many KV splits
    (40, [1, 300, 5000], 4, 1),         # G*R = 164 rows -> two query tiles; ragged batch
    (7, [63, 64, 65, 129], 16, 8),      # tile-boundary contexts, GQA group 2
    # 16+ sequences: the persistent kernel on the device-planned schedule (per-sequence
    # splits, one-split sequences written directly, the rest merged)
    (15, [1, 2, 63, 64, 65, 127, 128, 129, 300, 700, 1000, 1500, 2047, 2048, 3000, 4097, 5000, 9000], 8, 2),
    (40, [5000, 1, 64, 300, 2100, 17, 900, 129, 63, 4000, 2, 1200, 700, 65, 3333, 128], 4, 1),   # two query tiles
])
def test_tensor_core_attention_shapes(torch_cuda, K, ctx, n_q, n_kv):
    """bf16, head_dim 128: the tensor-core attention (split-KV and merge) against the oracle."""
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", head_dim=128, n_q_heads=n_q, n_kv_heads=n_kv, hidden=256,
                                  n_layers=2, batch=len(ctx), K=K, K_max=K, seed=21)
    Wn = make_weights(s)
    Wd = upload_weights(Wn)
    sb = SideBySide(s, Wn, Wd, K=K, ctx=ctx, iterations=2)
    sb.prefill(list(range(3, 3 + len(ctx))))
    for it in range(2):
        sb.step(it, RTOL["bf16"])


@pytest.mark.parametrize("shape_kw,ctx,K", [
    (dict(dtype="bf16", batch=3, head_dim=128), [64, 3, 130], 15),
    (dict(dtype="bf16", head_dim=128, n_q_heads=4, n_kv_heads=1, hidden=256, n_layers=2, batch=3, seed=21),
     [1, 300, 5000], 40),
    (dict(dtype="f32", batch=2), [100, 7], 15),
])
def test_kv_cache_matches_oracle(torch_cuda, shape_kw, ctx, K):
    """Context append (fc, RMSNorm, every layer's K/V, RoPE), element by element
    against the exact fp64 oracle's KV cache.  fp32: 1e-5 relative.  bf16: every
    element g of a K or V row within the bound of its storage,

        |g - e| <= 2^-8 |e| + (1 + 2^-8) 2^-13 A,

    e the exact value, A = sum_i |W_ji| |u_i| (for K the sum of the two rotated
    partners' A): the cache row is rounded once to bf16 (RNE, at most half an
    ulp, 2^-8 relative), and before that the value carries the error of its
    inputs -- the context feature u stored as a bf16 pair hi + lo (2^-16 relative
    per element) and fp32 accumulation of the fc and K/V products -- which the
    2^-13 A term bounds with room to spare."""
    import oracle as orc
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    from tests.helpers import feats_block
    s = CONFIGS["tiny_f32"].with_(K=K, K_max=K, **shape_kw)
    Wn = make_weights(s)
    dr = DFlashDrafter(DrafterConfig.from_shape(s), upload_weights(Wn), s.batch)
    f = feats_block(s, ctx, max(ctx), "prefill")
    dr.ctx_append(to_device(f), max(ctx), rows=np.array(ctx, np.int32))
    o = orc.OracleDrafter(s, Wn, s.batch)
    for b in range(s.batch):
        o.ctx_append(b, f[b, :ctx[b]])
    dr.draft_block(K, anchor_ids=np.arange(1, s.batch + 1, dtype=np.int32))
    torch_cuda.cuda.synchronize()
    worst = 0.0
    d2 = s.head_dim // 2
    for b in range(s.batch):
        if s.dtype == "bf16":
            x = orc.decode(f[b, :ctx[b]], np.float64)
            u = orc.rms_norm(x @ o.w("w_fc").T, o.w("fc_norm"), s.rms_eps)
        for l in range(s.n_layers):
            for kind in (0, 1):
                g = dr.read_kv(b, l, kind, 0, ctx[b])
                ref = (o.seqs[b].k if kind == 0 else o.seqs[b].v)[l].transpose(1, 0, 2)
                if s.dtype == "f32":
                    np.testing.assert_allclose(g, ref, rtol=1e-5, atol=1e-6)
                    continue
                W = o.w(f"layers.{l}." + ("wk" if kind == 0 else "wv"))
                A = (np.abs(u) @ np.abs(W).T).reshape(ctx[b], s.n_kv_heads, s.head_dim).transpose(1, 0, 2)
                if kind == 0:   # rotate-half: output i mixes inputs i and i +- d/2
                    A = A + np.concatenate([A[..., d2:], A[..., :d2]], axis=-1)
                bound = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * 2.0 ** -13 * A
                err = np.abs(g.astype(np.float64) - ref)
                ratio = err / np.maximum(bound, 1e-300)
                worst = max(worst, float(ratio.max()))
                assert (err <= bound).all(), (
                    f"seq {b} layer {l} {'KV'[kind]}: {(err > bound).sum()} elements past the storage bound "
                    f"(worst ratio {ratio.max():.2f})")
    print(f"KV cache: worst error / storage bound = {worst:.3f}")


def test_qwen3_4b_shape(torch_cuda):
    s = CONFIGS["qwen3_4b"]
    Wn, Wd = weights("qwen3_4b", torch_cuda)
    sb = SideBySide(s, Wn, Wd, K=s.K, iterations=2)
    sb.prefill([12345])
    for it in range(2):
        rep = sb.step(it, RTOL["bf16"])
        assert rep["ids_compared"] >= 3      # rows whose gap exceeds twice the bf16 logit error


def test_accept_bit_exact_on_arbitrary_targets(torch_cuda):
    """verify_accept on random target rows (not planted): bit-exact vs the literal rule."""
    import oracle as orc
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    s = CONFIGS["tiny_f32"].with_(batch=64, vocab=1024)
    Wn, Wd = weights("tiny_f32", torch_cuda)
    dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, s.batch)
    rng = np.random.default_rng(9)
    f = np.zeros((s.batch, 4, s.feat_dim), np.float32)
    dr.ctx_append(to_device(f), 4)
    K = 6
    d = np.zeros((s.batch, K), np.int32)
    dr.draft_block(K, anchor_ids=rng.integers(0, s.vocab, s.batch).astype(np.int32), draft_ids=d)
    torch_cuda.cuda.synchronize()
    g = rng.integers(0, s.vocab, size=(s.batch, K + 1)).astype(np.int32)
    # force a spread of prefix lengths
    for b in range(s.batch):
        n = b % (K + 1)
        g[b, :n] = d[b, :n]
        if n < K and g[b, n] == d[b, n]:
            g[b, n] = (d[b, n] + 1) % s.vocab
    acc = np.zeros(s.batch, np.int32)
    nxt = np.zeros(s.batch, np.int32)
    dr.verify_accept(g, accept_len=acc, next_anchor=nxt)
    torch_cuda.cuda.synchronize()
    for b in range(s.batch):
        assert (acc[b], nxt[b]) == orc.accept_prefix(d[b], g[b])
    st = dr.query_state()
    assert np.array_equal(st["ctx_len"], 4 + acc + 1)
    assert np.array_equal(st["anchor"], nxt)


def test_plant_kernel_matches_generator(torch_cuda):
    from block_diffusion_speculative_dflash_gb300 import plant_targets as plant_gpu
    from synth import plant_targets
    rng = np.random.default_rng(4)
    B, K, V = 33, 9, 500
    d = rng.integers(0, V, (B, K)).astype(np.int32)
    L = rng.integers(0, K + 1, B).astype(np.int32)
    fill = rng.integers(0, V, (B, K + 1)).astype(np.int32)
    out = torch_cuda.empty((B, K + 1), dtype=torch_cuda.int32, device="cuda")
    plant_gpu(to_device(d), to_device(L), to_device(fill), B, K, V, out)
    assert np.array_equal(out.cpu().numpy(), plant_targets(d, L, fill, V))


def test_growth_and_reserve_give_identical_results(torch_cuda):
    """Capacity (power-of-two growth with copy vs one large reservation) does not change results."""
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    from tests.helpers import feats_block
    s = CONFIGS["tiny_f32"].with_(batch=2)
    Wn, Wd = weights("tiny_f32", torch_cuda)
    outs = []
    for reserve in (0, 4096):
        dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, s.batch)
        if reserve:
            dr.reserve(reserve)
        caps = []
        for step, rows in enumerate((40, 30, 50, 20)):      # crosses 64 -> 128 -> 256
            f = feats_block(s, [rows, rows // 2], rows, f"grow{step}")
            dr.ctx_append(to_device(f), rows, rows=np.array([rows, rows // 2], np.int32))
            caps.append(dr.query_state()["capacity"].copy())
        z = torch_cuda.empty((2, 5, s.vocab), dtype=torch_cuda.float32, device="cuda")
        dr.draft_block(5, anchor_ids=np.array([3, 4], np.int32), logits=z)
        outs.append(z.cpu().numpy())
        if not reserve:
            assert caps[0].tolist() == [64, 64] and caps[-1].tolist() == [256, 128]
    assert np.array_equal(outs[0], outs[1])


def test_device_faults_are_latched_not_trapped(torch_cuda):
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DflashError, DrafterConfig
    from block_diffusion_speculative_dflash_gb300.binding import FLAG_BAD_TOKEN, FLAG_NOT_CONSUMED
    s = CONFIGS["tiny_f32"]
    Wn, Wd = weights("tiny_f32", torch_cuda)
    dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, 1)
    dr.ctx_append(to_device(np.zeros((1, 8, s.feat_dim), np.float32)), 8)
    with pytest.raises(DflashError):
        dr.draft_block(s.K + 1)                                  # K beyond k_max: host check
    with pytest.raises(DflashError):
        dr.draft_block(4, anchor_ids=np.array([s.vocab], np.int32))   # host-checked id
    dr.draft_block(4, anchor_ids=to_device(np.array([s.vocab + 5], np.int32)))  # device-side id
    st = dr.query_state(raise_on_flags=False)
    assert st["flags"] & FLAG_BAD_TOKEN
    dr.verify_accept(np.zeros(5, np.int32))
    dr.draft_block(4)                                            # accepted rows not appended
    st = dr.query_state(raise_on_flags=False)
    assert st["flags"] & FLAG_NOT_CONSUMED
    assert dr.query_state()["flags"] == 0                        # cleared by the read


def test_cuda_graph_replay_matches_eager(torch_cuda):
    """A captured append+draft+verify iteration replays to the eager results."""
    torch = torch_cuda
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    from tests.helpers import feats_block
    s = CONFIGS["tiny_f32"].with_(dtype="bf16", batch=2, head_dim=128)
    Wn = make_weights(s)
    Wd = upload_weights(Wn)
    K = 8
    res = []
    for mode in ("eager", "graph"):
        dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, 2)
        f0 = feats_block(s, [20, 9], 20, "prefill")
        dr.ctx_append(to_device(f0), 20, rows=np.array([20, 9], np.int32))
        dr.reserve(256)
        anchors = to_device(np.array([5, 6], np.int32))
        d = torch.zeros((2, K), dtype=torch.int32, device="cuda")
        g = to_device(np.array([[1] * (K + 1), [2] * (K + 1)], np.int32))
        acc = torch.zeros(2, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(2, dtype=torch.int32, device="cuda")
        rows = torch.zeros(2, dtype=torch.int32, device="cuda")
        fs = to_device(feats_block(s, [K + 1, K + 1], K + 1, "step"))
        dr.draft_block(K, anchor_ids=anchors, draft_ids=d)

        def it():
            dr.verify_accept(g, accept_len=acc, next_anchor=nxt)
            torch.add(acc, 1, out=rows)
            dr.ctx_append(fs, K + 1, rows=rows)
            dr.draft_block(K, draft_ids=d)

        if mode == "eager":
            for _ in range(3):
                it()
        else:
            it()  # warm-up sizes every workspace
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                it()
            graph.replay()
            graph.replay()
        torch.cuda.synchronize()
        st = dr.query_state()
        res.append((d.cpu().numpy(), st["ctx_len"].copy(), st["kv_len"].copy()))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1]) and np.array_equal(res[0][2], res[1][2])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_exact_ties_take_the_lowest_id(torch_cuda, dtype):
    """The greedy argmax breaks exact ties towards the lowest token id (KCH
    system architecture with GDB's greedy decoding; reading R8).  LM-head rows
    2i and 2i+1 are made identical, so every logit is tied with its pair bit for
    bit on the GPU (same inputs, same summation): every drafted id must be even,
    and equal to the oracle's wherever the best pair leads the next one by more
    than 1e-2 and twice the row's logit error."""
    import oracle as orc
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    from tests.helpers import feats_block, row_rel_err, top2_gap
    kw = dict(dtype=dtype, batch=2, seed=41)
    if dtype == "bf16":
        kw["head_dim"] = 128
    s = CONFIGS["tiny_f32"].with_(**kw)
    Wn = make_weights(s)
    lm = Wn["lm_head"].copy()
    lm[1::2] = lm[0::2]
    Wn["lm_head"] = lm
    dr = DFlashDrafter(DrafterConfig.from_shape(s), upload_weights(Wn), s.batch)
    ctx = [64, 30]
    f = feats_block(s, ctx, max(ctx), "prefill")
    dr.ctx_append(to_device(f), max(ctx), rows=np.array(ctx, np.int32))
    o = orc.OracleDrafter(s, Wn, s.batch)
    for b in range(s.batch):
        o.ctx_append(b, f[b, :ctx[b]])
    K = s.K
    anchors = np.array([3, 8], np.int32)
    d = torch_cuda.zeros((s.batch, K), dtype=torch_cuda.int32, device="cuda")
    z = torch_cuda.zeros((s.batch, K, s.vocab), dtype=torch_cuda.float32, device="cuda")
    dr.draft_block(K, anchor_ids=anchors, draft_ids=d, logits=z)
    od, oz = o.draft(K, anchors=list(anchors))
    torch_cuda.cuda.synchronize()
    dg, zg = d.cpu().numpy(), z.cpu().numpy()
    assert np.all(dg % 2 == 0), f"odd ids drafted on exact ties: {dg[dg % 2 == 1]}"
    assert np.all(od % 2 == 0)
    # the pairs are bit-identical on the GPU too
    assert np.array_equal(zg[..., 0::2], zg[..., 1::2])
    for b in range(s.batch):
        assert row_rel_err(zg[b], oz[b]).max() <= RTOL[dtype]
        pair_gap = top2_gap(oz[b][:, 0::2])
        row_err = np.max(np.abs(zg[b] - oz[b]), axis=-1)
        ok = pair_gap > np.maximum(1e-2, 2.0 * row_err)
        assert ok.sum() >= K // 2
        assert np.array_equal(dg[b][ok], od[b][ok])
