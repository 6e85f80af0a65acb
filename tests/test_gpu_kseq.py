"""GPU: a block length per sequence (dflash_draft_block_k).  Sequence b drafts
its own K_b masks -- its block rows see its K_b + 1 block keys only -- in a
batch padded to K + 1 rows; loops of draft -> verify -> append against the
oracle's per-sequence drafts (each its own forward), on the fp32 and bf16
paths, the persistent engine and the mma.sync attention."""
import os

import numpy as np
import pytest

from synth import CONFIGS, make_weights
from tests.helpers import SideBySide, to_device, upload_weights

pytestmark = pytest.mark.gpu


def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


def _with_env(env, fn):
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return fn()
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("shape_kw,env", [
    (dict(), {}),
    (dict(dtype="bf16", head_dim=128), {}),
    (dict(dtype="bf16", head_dim=128), {"DFLASH_ATTN_UMMA": "0"}),
])
def test_per_sequence_k_loop_matches_oracle(shape_kw, env):
    _cuda()
    K, ctx = 12, [64, 5, 300]
    s = CONFIGS["tiny_f32"].with_(K=K, K_max=K, batch=len(ctx), seed=46, **shape_kw)
    Wn = make_weights(s)
    sb = _with_env(env, lambda: SideBySide(s, Wn, upload_weights(Wn), K=K, ctx=ctx, iterations=4))
    sb.prefill([3, 4, 5])
    rng = np.random.default_rng(7)
    rtol = 2e-2 if s.dtype == "bf16" else 1e-4
    for it in range(4):
        ks = rng.integers(1, K + 1, size=len(ctx)).astype(np.int32)
        ks[it % len(ctx)] = K if it % 2 else 1          # the extremes
        sb.step(it, rtol, ks=ks)


def test_per_sequence_k_checks_its_argument():
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DflashError
    from block_diffusion_speculative_dflash_gb300.binding import FLAG_BAD_K
    K = 6
    s = CONFIGS["tiny_f32"].with_(K=K, K_max=K, batch=2, dtype="bf16", head_dim=128)
    sb = SideBySide(s, make_weights(s), upload_weights(make_weights(s)), K=K, ctx=[20, 20], iterations=1)
    sb.prefill([3, 4])
    d = torch.zeros((2, K), dtype=torch.int32, device="cuda")
    with pytest.raises(DflashError) as e:          # host values are checked before any launch
        sb.gpu.draft_block(K, draft_ids=d, k_seq=np.array([0, 3], np.int32))
    assert e.value.code == 1
    with pytest.raises(DflashError):
        sb.gpu.draft_block(K, draft_ids=d, k_seq=np.array([2, K + 1], np.int32))
    # a device array is clamped to [1, K] and latches DFLASH_FLAG_BAD_K
    sb.gpu.draft_block(K, draft_ids=d, k_seq=to_device(np.array([K + 5, 2], np.int32)))
    torch.cuda.synchronize()
    dg = d.cpu().numpy()
    assert np.all(dg[0] >= 0) and np.all(dg[1, 2:] == -1)
    with pytest.raises(DflashError) as e:
        sb.gpu.query_state()
    assert e.value.code == 5 and "0x20" in str(e.value)
