"""The C-ABI library builds for sm_103a, loads, and exports every declared symbol.

No compute call is made here (no GPU needed): only argument validation paths
that return before touching the device.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from block_diffusion_speculative_dflash_gb300 import load_library
    return load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("dflash_create", "dflash_destroy", "dflash_ctx_append", "dflash_draft_block",
              "dflash_verify_accept", "dflash_query_state", "dflash_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dflash_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    from block_diffusion_speculative_dflash_gb300.binding import EXPORTS
    assert set(EXPORTS) == set(declared_functions())


def test_struct_layouts_match_binding(tmp_path):
    """sizeof/offsetof of the C structs (compiled with gcc) equal the ctypes mirrors."""
    from block_diffusion_speculative_dflash_gb300.binding import Config, LayerWeights, TargetConfigC, Weights
    src = tmp_path / "probe.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "dflash.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(dflash_config),"
        " sizeof(dflash_layer_weights),"
        " sizeof(dflash_weights), offsetof(dflash_config, kv_pool_tokens), offsetof(dflash_config, dtype),"
        " offsetof(dflash_weights, layers), sizeof(dflash_target_config),"
        " offsetof(dflash_target_config, feat_layers), offsetof(dflash_target_config, kv_pool_tokens)); return 0;}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals == [ctypes.sizeof(Config), ctypes.sizeof(LayerWeights), ctypes.sizeof(Weights),
                    Config.kv_pool_tokens.offset, Config.dtype.offset, Weights.layers.offset,
                    ctypes.sizeof(TargetConfigC), TargetConfigC.feat_layers.offset,
                    TargetConfigC.kv_pool_tokens.offset]


def test_invalid_arguments_return_status_without_device(lib):
    from block_diffusion_speculative_dflash_gb300.binding import Config, Weights
    h = ctypes.c_void_p()
    assert lib.dflash_create(None, None, 1, ctypes.byref(h)) == 1
    assert b"null" in lib.dflash_last_error()
    c, w = Config(), Weights()
    assert lib.dflash_create(ctypes.byref(c), ctypes.byref(w), 0, ctypes.byref(h)) == 1
    assert lib.dflash_destroy(None) == 1
    assert lib.dflash_ctx_append(None, None, 0, None, None) == 1
    assert lib.dflash_draft_block(None, None, 1, None, None, None) == 1
    assert lib.dflash_verify_accept(None, None, None, None, None) == 1
    assert lib.dflash_plant_targets(None, None, None, 1, 1, 1, None, None, 1, None) == 1


def test_build_is_sm103a_only():
    from block_diffusion_speculative_dflash_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_alloc_failure_injection_hook(lib):
    """The host hook behind DFLASH_ERR_OOM injection: a process-wide counter,
    set and read back without touching a device."""
    from block_diffusion_speculative_dflash_gb300 import inject_alloc_failure
    try:
        assert inject_alloc_failure(-1) == -1      # off by default
        assert inject_alloc_failure(5) == -1
        assert inject_alloc_failure(2) == 5
        assert inject_alloc_failure(-7) == 2       # any negative value turns it off
        assert inject_alloc_failure(-1) == -1
    finally:
        inject_alloc_failure(-1)

