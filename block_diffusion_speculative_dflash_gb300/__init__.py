"""GB300-native DFlash drafter hot path: C-ABI library (libdflash.so) + ctypes binding.

    ctx_append     project concatenated target features into every draft layer's KV
    draft_block    one non-causal forward over [anchor ; K masks] -> greedy drafts
    verify_accept  longest matching prefix vs the target's argmax; state advance
    DFlashTarget   the target model's causal verify forward (ids, features) + commit
"""
from .binding import (  # noqa: F401
    DFlashDrafter,
    DFlashTarget,
    DflashError,
    DrafterConfig,
    EXPORTS,
    inject_alloc_failure,
    load_library,
    plant_targets,
    ptr,
    TargetConfig,
)
from ._build import build  # noqa: F401
