"""GPU: failure detection without a GPU fault.

Every wait in the kernels is bounded by the context's wait limit; a wait that
runs out latches DFLASH_FLAG_WAIT_TIMEOUT and its kernel returns, so the
context stays usable.  A device allocation that fails (injected on the host)
returns DFLASH_ERR_OOM and leaves the context as it was; so does an exhausted
KV pool.  An fp16 GEMM operand outside +-65504 latches DFLASH_FLAG_F16_RANGE.
Nothing here faults, traps or hangs the GPU: the one wait made to run out is
on an mbarrier no one arrives at, with a 1 ms limit.
"""
import time

import numpy as np
import pytest

from synth import CONFIGS, make_weights
from tests.helpers import SideBySide, feats_block, to_device, upload_weights

pytestmark = pytest.mark.gpu

FLAG_WAIT_TIMEOUT, FLAG_F16_RANGE = 0x8, 0x40


def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


def _bf16(**kw):
    return CONFIGS["tiny_f32"].with_(**{**dict(dtype="bf16", head_dim=128, n_layers=2, seed=61), **kw})


def test_wait_timeout_selftest_latches_the_flag_and_the_context_recovers():
    torch = _cuda()
    s = _bf16(batch=1)
    W = make_weights(s)
    sb = SideBySide(s, W, upload_weights(W), s.K, ctx=np.array([70], np.int32), iterations=2)
    sb.prefill([9])
    sb.gpu.set_wait_limit(1_000_000)                    # 1 ms
    t0 = time.perf_counter()
    sb.gpu.selftest_wait()
    st = sb.gpu.query_state(raise_on_flags=False)       # synchronises the stream
    dt = time.perf_counter() - t0
    assert st["flags"] & FLAG_WAIT_TIMEOUT, f"flags {st['flags']:#x}"
    assert dt < 1.0, f"the 1 ms wait took {dt:.3f} s"
    assert sb.gpu.query_state()["flags"] == 0           # returned once, then cleared
    # with the default limit back, the context drafts as before
    sb.gpu.set_wait_limit(0)
    for it in range(2):
        sb.step(it, 2e-2)
    torch.cuda.synchronize()


def test_injected_allocation_failure_at_create():
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DflashError, DrafterConfig, inject_alloc_failure
    s = _bf16(batch=2)
    Wd = upload_weights(make_weights(s))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for after in (0, 3, 9):
            assert inject_alloc_failure(after) == -1
            with pytest.raises(DflashError) as e:
                DFlashDrafter(DrafterConfig.from_shape(s), Wd, s.batch)
            assert e.value.code == 2                    # DFLASH_ERR_OOM
            assert inject_alloc_failure(-1) == -1       # spent: it fails once
            torch.cuda.synchronize()
            # everything the failed create had taken was given back
            assert abs(torch.cuda.mem_get_info()[0] - free0) <= (64 << 20)
    finally:
        inject_alloc_failure(-1)
    dr = DFlashDrafter(DrafterConfig.from_shape(s), Wd, s.batch)
    f = feats_block(s, [40, 12], 40, "prefill")
    dr.ctx_append(to_device(f), 40, rows=np.array([40, 12], np.int32))
    dr.draft_block(s.K, anchor_ids=np.array([1, 2], np.int32))
    assert dr.query_state()["flags"] == 0
    dr.close()


def test_injected_allocation_failure_on_workspace_growth():
    """The draft that needs a larger workspace fails with OOM and leaves the
    context consistent; the same draft succeeds once allocation works again."""
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DflashError, inject_alloc_failure
    s = _bf16(batch=2, K=15, K_max=15)
    W = make_weights(s)
    sb = SideBySide(s, W, upload_weights(W), s.K, ctx=np.array([8, 4], np.int32), iterations=2)
    sb.prefill([3, 4])
    st0 = sb.gpu.query_state()
    sb.gpu.draft_block(3, anchor_ids=np.array([3, 4], np.int32))   # workspace sized for 8 rows
    try:
        inject_alloc_failure(0)
        with pytest.raises(DflashError) as e:
            sb.gpu.draft_block(15)                      # needs about four times more
        assert e.value.code == 2
    finally:
        inject_alloc_failure(-1)
    st = sb.gpu.query_state()
    for k in ("ctx_len", "kv_len", "capacity"):
        assert np.array_equal(st[k], st0[k])
    for it in range(2):                                 # the loop against the oracle, as if nothing happened
        sb.step(it, 2e-2)
    torch.cuda.synchronize()


def test_exhausted_kv_pool_returns_oom_and_keeps_the_state():
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DflashError, DrafterConfig
    s = _bf16(batch=2, K=15, K_max=15)
    W = make_weights(s)
    # 256 token slots: two sequences of 100 rows take 128 each; growing one to 256 cannot fit
    dr = DFlashDrafter(DrafterConfig.from_shape(s, kv_pool_tokens=256), upload_weights(W), s.batch)
    f = feats_block(s, [100, 100], 100, "prefill")
    dr.ctx_append(to_device(f), 100, rows=np.array([100, 100], np.int32))
    st0 = dr.query_state()
    assert list(st0["capacity"]) == [128, 128]
    f2 = feats_block(s, [60, 0], 60, "more")
    with pytest.raises(DflashError) as e:
        dr.ctx_append(to_device(f2), 60, rows=np.array([60, 0], np.int32))
    assert e.value.code == 2                            # DFLASH_ERR_OOM: KV arena full
    st = dr.query_state()
    for k in ("ctx_len", "kv_len", "capacity"):
        assert np.array_equal(st[k], st0[k])
    # the context still drafts (both sequences fit their capacity)
    d = torch.zeros((2, s.K), dtype=torch.int32, device="cuda")
    dr.draft_block(s.K, anchor_ids=np.array([5, 6], np.int32), draft_ids=d)
    assert dr.query_state()["flags"] == 0
    dr.check_guards()
    dr.close()


def test_f16_operand_out_of_range_latches_the_flag():
    """Above 128 GEMM rows the token operands are fp16: a norm gain of 2^17
    pushes the normalised rows past 65504, and the draft reports it."""
    torch = _cuda()
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig
    s = _bf16(batch=9, K=15, K_max=15)                  # 144 GEMM rows
    W = make_weights(s)
    g = W["layers.0.attn_norm"].copy()
    g[:] = np.uint16(0x4800)                            # bf16 2^17
    W["layers.0.attn_norm"] = g
    dr = DFlashDrafter(DrafterConfig.from_shape(s), upload_weights(W), s.batch)
    ctx = [30] * s.batch
    f = feats_block(s, ctx, 30, "prefill")
    dr.ctx_append(to_device(f), 30, rows=np.array(ctx, np.int32))
    dr.draft_block(s.K, anchor_ids=np.arange(1, s.batch + 1, dtype=np.int32))
    st = dr.query_state(raise_on_flags=False)
    assert st["flags"] & FLAG_F16_RANGE, f"flags {st['flags']:#x}"
    dr.close()
    torch.cuda.synchronize()
