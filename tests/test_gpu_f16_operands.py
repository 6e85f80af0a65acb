"""GPU: fp16 token operands.  From 33 GEMM rows a bf16 draft stores every
projection's token operand as one fp16 plane and multiplies it with fp16
copies of the weights, instead of split bf16 (two planes, twice the tensor
work).  The drafts must still meet the logit tolerance against the oracle;
the mode must engage from 33 rows (the logits differ from the split ones)
and nowhere else (bit-identical at 32 rows or fewer)."""
import numpy as np
import pytest

from synth import CONFIGS, make_weights
from tests.helpers import SideBySide, feats_block, row_rel_err, to_device, upload_weights

pytestmark = pytest.mark.gpu


def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


def _shape(batch, K, **kw):
    return CONFIGS["tiny_f32"].with_(**{**dict(dtype="bf16", head_dim=128, n_layers=2, K=K, K_max=K, batch=batch,
                                               seed=57), **kw})


def test_f16_operand_drafts_match_the_oracle():
    _cuda()
    s = _shape(12, 15)                                     # 192 GEMM rows
    W = make_weights(s)
    ctx = np.array([5, 300, 17, 64, 129, 1, 90, 200, 33, 250, 8, 150], np.int32)
    sb = SideBySide(s, W, upload_weights(W), s.K, ctx=ctx, iterations=3)
    sb.prefill(np.arange(12, dtype=np.int32) * 7 % s.vocab)
    for it in range(3):
        sb.step(it, rtol=2e-2)


def _draft(torch, s, W_dev, ctx):
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    B, K = s.batch, s.K
    dr = DFlashDrafter(DrafterConfig.from_shape(s), W_dev, B)
    rmax = int(ctx.max())
    dr.ctx_append(to_device(feats_block(s, ctx, rmax, "prefill")), rmax, rows=ctx.copy())
    d = torch.empty((B, K), dtype=torch.int32, device="cuda")
    z = torch.empty((B, K, s.vocab), dtype=torch.float32, device="cuda")
    dr.draft_block(K, anchor_ids=to_device(np.arange(B, dtype=np.int32) + 3), draft_ids=d, logits=z)
    torch.cuda.synchronize()
    out = z.cpu().numpy()
    dr.close()
    return out


@pytest.mark.parametrize("batch,K,engaged", [(12, 15, True), (3, 10, True), (2, 15, False), (1, 16, False)])
def test_f16_operands_engage_from_33_rows_only(monkeypatch, batch, K, engaged):
    torch = _cuda()
    s = _shape(batch, K)
    W_dev = upload_weights(make_weights(s))
    ctx = (np.arange(batch, dtype=np.int32) * 37 % 200 + 4).astype(np.int32)
    z_default = _draft(torch, s, W_dev, ctx)
    monkeypatch.setenv("DFLASH_F16_OPS", "0")
    z_split = _draft(torch, s, W_dev, ctx)
    if engaged:
        assert not np.array_equal(z_default, z_split), f"fp16 operands did not engage at {batch * (K + 1)} rows"
        assert row_rel_err(z_default.reshape(-1, s.vocab), z_split.reshape(-1, s.vocab)).max() <= 2e-2
    else:
        assert np.array_equal(z_default, z_split), f"the operand format changed at {batch * (K + 1)} rows"
