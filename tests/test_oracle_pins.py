"""Pins of the CPU oracle against things other than itself.

Closed forms, invariants, special cases that reduce to library routines
(torch CPU fp64), brute force on tiny inputs and hand-worked cases.  Each
check is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, index or position, a transposed operand, context injected into the
wrong layer) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as orc
from synth import DrafterShape, make_features, make_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_forms():
    # constant vector a*1: mean square a^2
    x = np.full((1, 6), 3.0)
    g = np.full(6, 2.0)
    out = orc.rms_norm(x, g, 1e-6)
    np.testing.assert_allclose(out, 2.0 * 3.0 / math.sqrt(9.0 + 1e-6), rtol=0, atol=1e-15)
    # [3, 4]: rms = sqrt(12.5)
    out = orc.rms_norm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    np.testing.assert_allclose(out, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=1e-15)
    # normalisation is per row (last axis), gain is per column
    x = np.array([[1.0, 1.0], [10.0, 10.0]])
    out = orc.rms_norm(x, np.array([1.0, 3.0]), 0.0)
    np.testing.assert_allclose(out, [[1.0, 3.0], [1.0, 3.0]], rtol=1e-15)


def test_rms_norm_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((4, 16))
    g = rng.standard_normal(16)
    np.testing.assert_allclose(orc.rms_norm(7.5 * x, g, 0.0), orc.rms_norm(x, g, 0.0), rtol=1e-13)


# ---------------------------------------------------------------- RoPE

def test_rope_d2_by_hand():
    # d = 2: one pair, frequency theta^0 = 1; position 1 rotates by 1 radian.
    x = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    out = orc.apply_rope(x, np.array([1, 1]), theta=1e4)
    c, s = math.cos(1.0), math.sin(1.0)
    np.testing.assert_allclose(out[0, 0], [c, s], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[1, 0], [-s, c], rtol=0, atol=1e-15)


def test_rope_d4_pairs_and_frequencies_by_hand():
    # d = 4: pairs (0, 2) at frequency 1 and (1, 3) at theta^(-1/2).
    theta = 100.0
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    out = orc.apply_rope(x, np.array([2]), theta)
    ang = 2 * theta ** -0.5  # 0.2 rad
    np.testing.assert_allclose(out[0, 0], [0.0, math.cos(ang), 0.0, math.sin(ang)], atol=1e-15)
    x = np.array([[[0.0, 0.0, 1.0, 0.0]]])
    out = orc.apply_rope(x, np.array([2]), theta)
    np.testing.assert_allclose(out[0, 0], [-math.sin(2.0), 0.0, math.cos(2.0), 0.0], atol=1e-15)
    np.testing.assert_allclose(orc.rope_inv_freq(4, theta), [1.0, 0.1], rtol=1e-15)


def test_rope_relative_and_norm_preserving():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((1, 1, 16))
    dots = []
    for m in (3, 10, 1000):
        qm = orc.apply_rope(q, np.array([m]), 1e4)
        kn = orc.apply_rope(k, np.array([m - 2]), 1e4)
        dots.append(float(np.sum(qm * kn)))
        np.testing.assert_allclose(np.linalg.norm(qm), np.linalg.norm(q), rtol=1e-13)
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


# ---------------------------------------------------------------- attention

def test_attention_single_key_returns_value_exactly():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((3, 4, 8))
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    out = orc.attention(q, k, v)
    for h in range(4):
        assert np.array_equal(out[:, h, :], np.repeat(v[:, h // 2, :], 3, axis=0))


def test_attention_zero_query_is_mean_of_values():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((7, 1, 4))
    v = rng.standard_normal((7, 1, 4))
    out = orc.attention(np.zeros((2, 2, 4)), k, v)
    np.testing.assert_allclose(out[0, 1], v[:, 0].mean(axis=0), rtol=1e-14)


def test_attention_matches_torch_sdpa_gqa():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(4)
    for (Rq, T, nq, nkv, d) in [(5, 9, 4, 2, 8), (17, 33, 8, 2, 16), (1, 1, 2, 1, 4)]:
        q = rng.standard_normal((Rq, nq, d))
        k = rng.standard_normal((T, nkv, d))
        v = rng.standard_normal((T, nkv, d))
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q).permute(1, 0, 2)[None], torch.from_numpy(k).permute(1, 0, 2)[None],
            torch.from_numpy(v).permute(1, 0, 2)[None], is_causal=False, enable_gqa=True)
        np.testing.assert_allclose(orc.attention(q, k, v), ref[0].permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-13)


def test_attention_key_permutation_invariance():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 2, 8))
    k = rng.standard_normal((11, 1, 8))
    v = rng.standard_normal((11, 1, 8))
    perm = rng.permutation(11)
    np.testing.assert_allclose(orc.attention(q, k, v), orc.attention(q, k[perm], v[perm]), rtol=1e-12)


# ---------------------------------------------------------------- MLP, argmax

def test_silu_and_swiglu_closed_forms():
    assert orc.silu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(orc.silu(np.array(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(orc.silu(np.array(-2.0)), -2.0 / (1.0 + math.exp(2.0)), rtol=1e-15)
    x = np.array([[0.5, -1.0, 2.0]])
    eye = np.eye(3)
    np.testing.assert_allclose(orc.swiglu(x, eye, eye, eye), orc.silu(x) * x, rtol=1e-15)
    # gate and up are distinct operands: swapping them changes the result
    wg = np.diag([1.0, 2.0, 3.0])
    np.testing.assert_allclose(orc.swiglu(x, wg, eye, eye), orc.silu(x * [1, 2, 3]) * x, rtol=1e-15)
    # down projection maps the inner size back: [out, in] layout
    wd = np.array([[1.0, 0.0, 0.0]])
    np.testing.assert_allclose(orc.swiglu(x, eye, eye, wd), (orc.silu(x) * x)[:, :1], rtol=1e-15)


def test_greedy_argmax_lowest_index_on_ties():
    z = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [0.0, -1.0, 0.5, 0.5]])
    assert orc.greedy_argmax(z).tolist() == [1, 0, 2]


# ---------------------------------------------------------------- accept rule

def _golden_accept_cases():
    cases = []
    with open(os.path.join(GOLDEN, "accept_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            d, g, n, bonus = [p.strip() for p in line.split("|")]
            cases.append(([int(t) for t in d.split()], [int(t) for t in g.split()], int(n), int(bonus)))
    return cases


@pytest.mark.parametrize("case", _golden_accept_cases())
def test_accept_hand_worked(case):
    d, g, n, bonus = case
    assert orc.accept_prefix(d, g) == (n, bonus)


def test_accept_brute_force_v2_k3():
    # every draft in {0,1}^3 against every target row in {0,1}^4, checked
    # against the set definition n = max{ n <= K : d_j == g_{j-1} for all j <= n }
    K = 3
    for d in itertools.product((0, 1), repeat=K):
        for g in itertools.product((0, 1), repeat=K + 1):
            valid = [n for n in range(K + 1) if all(d[j] == g[j] for j in range(n))]
            n = max(valid)
            assert orc.accept_prefix(d, g) == (n, g[n])


# ---------------------------------------------------------------- full drafter

def _tiny(shape, **kw):
    return shape.with_(**kw)


def _drafter(shape, weights=None, batch=1, **kw):
    weights = make_weights(shape) if weights is None else weights
    return orc.OracleDrafter(shape, weights, batch, **kw), weights


def _prefill(dr, shape, rows, b=0, tag="prefill"):
    f = make_features(shape, rows, tag=tag, batch_index=b)
    dr.ctx_append(b, f)
    return f


def test_drafter_matches_torch_encoder_without_context(tiny_shape):
    """c = 0 and no RoPE: the drafter is a pre-norm bidirectional encoder with
    GQA attention and a SwiGLU MLP followed by a final norm and the LM head --
    built here from torch library routines (rms_norm, sdpa, silu, linear)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    s = _tiny(tiny_shape, n_layers=2)
    dr, W = _drafter(s, use_rope=False)
    dr.set_anchor(0, 7)
    K = 4
    drafts, logits = dr.draft(K)

    t = {k: torch.from_numpy(orc.decode(v)) for k, v in W.items()}
    ids = torch.tensor([7] + [s.mask_token_id] * K)
    h = t["embed"][ids]
    for l in range(s.n_layers):
        p = f"layers.{l}."
        x = F.rms_norm(h, (s.hidden,), t[p + "attn_norm"], eps=s.rms_eps)
        q = F.linear(x, t[p + "wq"]).view(K + 1, s.n_q_heads, s.head_dim).transpose(0, 1)
        k = F.linear(x, t[p + "wk"]).view(K + 1, s.n_kv_heads, s.head_dim).transpose(0, 1)
        v = F.linear(x, t[p + "wv"]).view(K + 1, s.n_kv_heads, s.head_dim).transpose(0, 1)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], enable_gqa=True)[0]
        h = h + F.linear(o.transpose(0, 1).reshape(K + 1, -1), t[p + "wo"])
        x = F.rms_norm(h, (s.hidden,), t[p + "mlp_norm"], eps=s.rms_eps)
        h = h + F.linear(F.silu(F.linear(x, t[p + "w_gate"])) * F.linear(x, t[p + "w_up"]),
                         t[p + "w_down"])
    z = F.linear(F.rms_norm(h[1:], (s.hidden,), t["final_norm"], eps=s.rms_eps), t["lm_head"])
    np.testing.assert_allclose(logits[0], z.numpy(), rtol=1e-11, atol=1e-12)
    assert drafts[0].tolist() == torch.argmax(z, dim=-1).tolist()


def test_block_is_permutation_equivariant_without_rope(tiny_shape):
    s = _tiny(tiny_shape, n_layers=2)
    dr, W = _drafter(s, use_rope=False)
    _prefill(dr, s, 5)
    rng = np.random.default_rng(6)
    K = 5
    emb = rng.standard_normal((1, K + 1, s.hidden))
    perm = np.concatenate([[0], 1 + rng.permutation(K)])
    _, z0 = dr.draft(K, block_embeds=emb)
    _, z1 = dr.draft(K, block_embeds=emb[:, perm])
    np.testing.assert_allclose(z1[0], z0[0][perm[1:] - 1], rtol=1e-11, atol=1e-12)


def test_mask_rows_identical_without_rope(tiny_shape):
    dr, _ = _drafter(tiny_shape, use_rope=False)
    _prefill(dr, tiny_shape, 6)
    dr.set_anchor(0, 3)
    _, z = dr.draft(4)
    for j in range(1, 4):
        np.testing.assert_allclose(z[0, j], z[0, 0], rtol=1e-13, atol=1e-14)


def test_mask_rows_differ_with_rope(tiny_shape):
    dr, _ = _drafter(tiny_shape)
    _prefill(dr, tiny_shape, 6)
    _, z = dr.draft(4)
    assert np.max(np.abs(z[0, 1] - z[0, 0])) > 1e-5     # vs ~1e-14 without RoPE


def test_relative_position_invariance(tiny_shape):
    s = _tiny(tiny_shape, n_layers=2)
    W = make_weights(s)
    feats = make_features(s, 9)
    outs = []
    for off in (0, 37, 1000):
        dr = orc.OracleDrafter(s, W, 1, pos_offset=off)
        dr.ctx_append(0, feats)
        dr.set_anchor(0, 5)
        outs.append(dr.draft(5)[1])
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-9, atol=1e-10)
    # but the absolute placement of the block relative to the context matters
    dr = orc.OracleDrafter(s, W, 1)
    dr.ctx_append(0, feats)
    dr.set_anchor(0, 5)
    dr.seqs[0].ctx_len += 3
    dr.seqs[0].kv_len += 3     # block shifted away from the context
    assert np.max(np.abs(dr.draft(5)[1] - outs[0])) > 1e-4


def test_chunked_append_equals_single_append(tiny_shape):
    s = _tiny(tiny_shape, n_layers=2)
    W = make_weights(s)
    feats = make_features(s, 14)
    a, _ = _drafter(s, W)
    a.ctx_append(0, feats)
    b, _ = _drafter(s, W)
    lo = 0
    for n in (1, 3, 7, 3):
        b.ctx_append(0, feats[lo:lo + n])
        lo += n
    for l in range(s.n_layers):
        np.testing.assert_allclose(b.seqs[0].k[l], a.seqs[0].k[l], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(b.seqs[0].v[l], a.seqs[0].v[l], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b.draft(5)[1], a.draft(5)[1], rtol=1e-11, atol=1e-12)


def test_context_row_equals_block_row_in_one_layer(tiny_shape):
    """KV injection pin (1 draft layer).  With W_fc selecting the first target
    feature and unit gains, a context row whose first feature is E[t] yields the
    same K/V as a block row holding token t at that position.  So drafting with
    context t_0..t_{c-1} and anchor t_c equals drafting with context
    t_0..t_{c-2} and the block [t_{c-1}, t_c, masks] one position earlier."""
    s = tiny_shape
    W = make_weights(s)
    H, Lt = s.hidden, s.n_target_layers
    W = dict(W)
    W["w_fc"] = np.concatenate([np.eye(H, dtype=np.float32),
                                np.zeros((H, (Lt - 1) * H), np.float32)], axis=1)
    E = orc.decode(W["embed"])
    rng = np.random.default_rng(7)
    c = 6
    toks = rng.integers(0, s.vocab - 1, size=c + 1)
    feats = np.zeros((c, Lt * H), np.float32)
    feats[:, :H] = E[toks[:c]]
    feats[:, H:] = rng.standard_normal((c, (Lt - 1) * H))   # ignored by this W_fc
    K = 4

    a = orc.OracleDrafter(s, W, 1)
    a.ctx_append(0, feats)
    a.set_anchor(0, int(toks[c]))
    _, za = a.draft(K)

    b = orc.OracleDrafter(s, W, 1)
    b.ctx_append(0, feats[:c - 1])
    emb = np.concatenate([E[toks[c - 1]][None], E[toks[c]][None],
                          np.repeat(E[s.mask_token_id][None], K, 0)])[None]
    _, zb = b.draft(K + 1, block_embeds=emb)
    np.testing.assert_allclose(zb[0, 1:], za[0], rtol=1e-10, atol=1e-11)


def test_context_is_injected_into_every_layer(tiny_shape):
    """With layer 0's output projections zeroed, a 2-layer drafter equals the
    1-layer drafter made of layer 1 -- which still sees the context, through
    layer 1's own K/V projections of the context feature."""
    s2 = _tiny(tiny_shape, n_layers=2)
    W2 = dict(make_weights(s2))
    W2["layers.0.wo"] = np.zeros_like(W2["layers.0.wo"])
    W2["layers.0.w_down"] = np.zeros_like(W2["layers.0.w_down"])
    s1 = _tiny(tiny_shape, n_layers=1)
    W1 = {k: v for k, v in W2.items() if not k.startswith("layers.")}
    for k, v in W2.items():
        if k.startswith("layers.1."):
            W1["layers.0." + k[len("layers.1."):]] = v
    feats = make_features(s2, 8)
    outs = []
    for s, W in ((s2, W2), (s1, W1)):
        dr = orc.OracleDrafter(s, W, 1)
        dr.ctx_append(0, feats)
        dr.set_anchor(0, 9)
        outs.append(dr.draft(5)[1])
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-12, atol=1e-13)
    # and the context matters there
    dr = orc.OracleDrafter(s1, W1, 1)
    dr.ctx_append(0, make_features(s2, 8, tag="other"))
    dr.set_anchor(0, 9)
    assert np.max(np.abs(dr.draft(5)[1] - outs[1])) > 1e-3


def test_verify_advances_state_by_accepted_count_only(tiny_shape):
    dr, W = _drafter(tiny_shape)
    _prefill(dr, tiny_shape, 6)
    dr.set_anchor(0, 3)
    K = 5
    drafts, _ = dr.draft(K)
    targets = np.array([[drafts[0, 0], drafts[0, 1], 0, 0, 0, 0]])
    targets[0, 2] = (drafts[0, 2] + 1) % tiny_shape.vocab
    n, bonus = dr.verify(drafts, targets)
    assert n.tolist() == [2] and bonus.tolist() == [int(targets[0, 2])]
    st = dr.seqs[0]
    assert st.ctx_len == 6 + 3 and st.kv_len == 6 and st.anchor == bonus[0]
    with pytest.raises(ValueError):
        dr.draft(K)                       # the accepted rows were not appended yet
    dr.ctx_append(0, make_features(tiny_shape, 3, tag="step1"))
    assert st.kv_len == st.ctx_len == 9
    dr.draft(K)


def test_fp32_mode_close_to_fp64(tiny_shape):
    W = make_weights(tiny_shape)
    feats = make_features(tiny_shape, 6)
    z = []
    for dt in (np.float64, np.float32):
        dr = orc.OracleDrafter(tiny_shape, W, 1, dtype=dt)
        dr.ctx_append(0, feats)
        z.append(dr.draft(5)[1])
    assert z[1].dtype == np.float32
    np.testing.assert_allclose(z[1], z[0], rtol=1e-4, atol=1e-5)


# ---------------------------------------------------------------- bf16 storage mode

def test_round_bf16_by_hand():
    # representable values are kept; 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    x = np.array([1.0, -2.5, 3.140625, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)])
    assert orc.round_bf16(x).tolist() == [1.0, -2.5, 3.140625, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0]
    r = np.random.default_rng(8).standard_normal(5000)
    rel = np.abs(orc.round_bf16(r) - r.astype(np.float32)) / np.abs(r)
    assert rel.max() <= 2 ** -8 + 1e-7
    assert np.array_equal(orc.round_bf16(orc.round_bf16(r)), orc.round_bf16(r))   # idempotent
