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


def test_other_config_summary_reads_the_childs_last_line():
    import json

    import bench
    line = {"metric": "m", "value": 8367.5, "ms_per_step": 0.9561, "clocks": {"sm_mhz": 2070.0},
            "config": {"workload": "llama31_8b: ..."}}
    out = "warming up\n" + json.dumps({"value": 1.0}) + "\n" + json.dumps(line) + "\n"
    r = bench.other_config_summary("llama31_8b", 0, out)
    assert r["us_per_step"] == pytest.approx(956.1) and r["blocks_per_s"] == 8367.5
    assert r["workload"] == "llama31_8b: ..." and r["clocks"] == {"sm_mhz": 2070.0}
    assert r["command"].startswith("python bench.py --config llama31_8b ")
    # a failed child or one without a result line is reported, not raised
    assert "error" in bench.other_config_summary("x", 1, json.dumps(line), "Traceback\nRuntimeError: boom")
    assert "boom" in bench.other_config_summary("x", 1, "", "Traceback\nRuntimeError: boom")["error"]
    assert "error" in bench.other_config_summary("x", 0, "no json here\n{not json")


def test_other_config_cmd_runs_no_nested_extras():
    import bench
    cmd = bench.other_config_cmd("qwen3_4b_serving")
    assert cmd[1].endswith("bench.py") and cmd[cmd.index("--config") + 1] == "qwen3_4b_serving"
    for flag in ("--no-cpu-baseline", "--no-e2e", "--k-sweep=", "--other-configs="):
        assert flag in cmd
    assert int(cmd[cmd.index("--warmup") + 1]) >= 3
