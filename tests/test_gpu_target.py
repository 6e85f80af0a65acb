"""GPU: the target-side verify forward (dflash_target_*) against the oracle's
causal decoder -- a prefill forward kept to ragged lengths, then verify blocks
of R tokens with partial commits (accepted + 1 rows); logits, greedy ids (where
the oracle's top-2 gap decides them) and the exported features."""
import numpy as np
import pytest

from oracle import OracleTarget
from synth import CONFIGS, make_weights
from tests.helpers import greedy_ids, row_rel_err, to_device, top2_gap, upload_weights

pytestmark = pytest.mark.gpu


def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


def _shape(**kw):
    return CONFIGS["tiny_f32"].with_(**{**dict(dtype="bf16", head_dim=128, n_layers=2, seed=48), **kw})


@pytest.mark.parametrize("shape_kw,B", [
    (dict(), 3),
    (dict(n_layers=3, n_q_heads=8, n_kv_heads=2), 3),
    (dict(n_q_heads=8, n_kv_heads=2), 17),   # 16+ sequences: the persistent causal attention
])
def test_target_forward_matches_oracle(shape_kw, B):
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DFlashTarget, TargetConfig
    s = _shape(**shape_kw)
    W = make_weights(s)
    r_max = 64
    feat = [0, s.n_layers - 1]
    tg = DFlashTarget(TargetConfig.from_shape(s, r_max, feat_layers=feat), upload_weights(W), B)
    orc = OracleTarget(s, W, B, feat_layers=feat)
    rng = np.random.default_rng(5)
    rtol = 2e-2

    def run(R, keep, device_keep=False):
        toks = rng.integers(0, s.vocab, size=(B, R)).astype(np.int32)
        ids = torch.empty((B, R), dtype=torch.int32, device="cuda")
        z = torch.empty((B, R, s.vocab), dtype=torch.float32, device="cuda")
        f = torch.empty((B, R, len(feat) * s.hidden), dtype=torch.bfloat16, device="cuda")
        tg.forward(to_device(toks), ids, logits=z, feats=f)
        torch.cuda.synchronize()
        ig, zg, fg = ids.cpu().numpy(), z.cpu().numpy(), f.float().cpu().numpy()
        compared = 0
        for b in range(B):
            io, zo, fo = orc.forward(b, toks[b])
            err = row_rel_err(zg[b], zo)
            assert err.max() <= rtol, f"seq {b} R {R}: logits rel err {err.max():.3e}"
            assert np.array_equal(ig[b], greedy_ids(zg[b])), "fused argmax != argmax(logits)"
            row_err = np.max(np.abs(zg[b] - zo), axis=-1)
            ok = top2_gap(zo) > np.maximum(1e-2, 2.0 * row_err)
            compared += int(ok.sum())
            assert np.array_equal(ig[b][ok], io[ok]), f"seq {b} R {R}: ids differ where the gap decides"
            ferr = row_rel_err(fg[b], fo)
            assert ferr.max() <= rtol, f"seq {b} R {R}: features rel err {ferr.max():.3e}"
            orc.commit(b, int(keep[b]))
        assert compared > 0   # (a single-row block of one sequence may have no decidable row)
        tg.commit(to_device(keep.astype(np.int32)) if device_keep else keep.astype(np.int32))
        np.testing.assert_array_equal(tg.query(), np.array(orc.len, np.int32))

    run(37, np.resize(np.array([37, 5, 20, 1, 30, 12]), B))   # prefill, kept to ragged lengths
    for it, R in enumerate([17, 11, 40, 3, 1, 60]):   # verify blocks (60 rows: 180 GEMM rows, plain bf16 operands)
        run(R, rng.integers(1, R + 1, size=B), device_keep=it % 2 == 1)


def test_target_checks_its_arguments():
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DFlashTarget, DflashError, TargetConfig
    s = _shape()
    W = upload_weights(make_weights(s))
    B, r_max = 2, 8
    with pytest.raises(DflashError):                # a feature layer outside the model
        DFlashTarget(TargetConfig.from_shape(s, r_max, feat_layers=[0, s.n_layers]), W, B)
    tg = DFlashTarget(TargetConfig.from_shape(s, r_max), W, B)
    ids = torch.empty((B, r_max + 1), dtype=torch.int32, device="cuda")
    with pytest.raises(DflashError) as e:           # R past r_max
        tg.forward(torch.zeros((B, r_max + 1), dtype=torch.int32, device="cuda"), ids)
    assert e.value.code == 1
    toks = torch.ones((B, 4), dtype=torch.int32, device="cuda")
    ids = torch.empty((B, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(DflashError):                # features without feature layers
        tg.forward(toks, ids, feats=torch.empty((B, 4, s.hidden), dtype=torch.bfloat16, device="cuda"))
    tg.forward(toks, ids)
    with pytest.raises(DflashError):                # keep past the forward's rows
        tg.commit(np.array([5, 1], np.int32))
    tg.commit(np.array([4, 2], np.int32))
    np.testing.assert_array_equal(tg.query(), [4, 2])
