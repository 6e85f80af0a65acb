"""The bench's roofline numerators on CPU: the algorithmic bytes of one draft +
accept step and of one append, checked against the byte counts worked out by
hand from the Qwen3-4B-shaped drafter's matrices, and the rule that a committed
ncu traffic figure is used only while it was taken on the current sources."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_step_bytes_qwen3_4b_by_hand():
    import bench
    from synth import CONFIGS
    s = CONFIGS["qwen3_4b"]
    draft, append = bench.step_bytes(s, [2048], 16)
    # one draft layer, bf16: W_q 4096x2560, W_k and W_v 1024x2560 each, W_o 2560x4096,
    # W_gate and W_up 9728x2560 each, W_down 2560x9728
    layer = 2 * (10_485_760 + 2 * 2_621_440 + 10_485_760 + 2 * 24_903_680 + 24_903_680)
    assert layer == 201_850_880
    lm_head = 2 * 151_936 * 2560                      # 777,912,320
    kv = (2048 + 17) * 5 * 2 * 1024 * 2               # K and V of 2065 slots in 5 layers
    assert draft == 5 * layer + lm_head + kv == 1_829_457_920
    # append: W_fc (2560 x 5*2560 target features) + every layer's [W_k; W_v]
    assert append == 2 * (2560 * 12_800 + 5 * 2 * 1024 * 2560) == 117_964_800


def test_step_bytes_conditioning_variants():
    import bench
    from synth import CONFIGS
    s = CONFIGS["qwen3_4b"]
    kv_draft, _ = bench.step_bytes(s, [2048, 100], 16)
    in_draft, in_append = bench.step_bytes(s, [2048, 100], 16, conditioning="input")
    none_draft, none_append = bench.step_bytes(s, [2048, 100], 16, conditioning="none")
    per_slot = 5 * 2 * 1024 * 2
    # without context K/V only the block's own 17 slots per sequence are read
    assert kv_draft - in_draft == (2048 + 100) * per_slot
    assert in_draft == none_draft
    assert in_append == 2 * 2560 * 12_800 and none_append == 0


def test_lm_traffic_only_for_current_sources(monkeypatch):
    import bench

    class Shape:
        name = "qwen3_4b"

    v = bench.lm_traffic(Shape, 16)
    if v is None:
        pytest.skip("the committed LM-head capture predates the current kernel sources")
    assert v > 778_000_000   # at least the LM head's weights
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.lm_traffic(Shape, 16) is None
    monkeypatch.undo()
    assert bench.lm_traffic(Shape, 32) is None   # another workload
