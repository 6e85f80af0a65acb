"""Thin ctypes binding of libdflash.so: argument marshalling only.

Every step of the drafter runs in the library's CUDA kernels; this module only
turns tensors / arrays into pointers and status codes into exceptions.  There
is no fallback: if the library cannot be built or loaded, importing the
drafter fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np

from . import _build

MAX_LAYERS = 32
DTYPES = {"f32": 0, "bf16": 1}
CONDITIONING = {"kv": 0, "input": 1, "none": 2}   # dflash_conditioning

STATUS = {0: "DFLASH_OK", 1: "DFLASH_ERR_INVALID", 2: "DFLASH_ERR_OOM", 3: "DFLASH_ERR_CAPACITY",
          4: "DFLASH_ERR_CUDA", 5: "DFLASH_ERR_DEVICE_FLAG", 6: "DFLASH_ERR_UNSUPPORTED"}
FLAG_BAD_TOKEN, FLAG_NOT_CONSUMED, FLAG_CAPACITY, FLAG_WAIT_TIMEOUT, FLAG_BAD_ROWS, FLAG_BAD_K = 1, 2, 4, 8, 16, 32
FLAG_F16_RANGE = 64

EXPORTS = ("dflash_create", "dflash_destroy", "dflash_reserve", "dflash_ctx_append", "dflash_draft_block",
           "dflash_verify_accept", "dflash_query_state", "dflash_last_error", "dflash_plant_targets",
           "dflash_trace_enable", "dflash_trace_read", "dflash_launch_count", "dflash_read_kv",
           "dflash_draft_block_noalloc", "dflash_reserve_headroom", "dflash_draft_block_k",
           "dflash_target_create", "dflash_target_destroy", "dflash_target_forward", "dflash_target_commit",
           "dflash_target_query", "dflash_graph_replays", "dflash_set_wait_limit", "dflash_selftest_wait",
           "dflash_inject_alloc_failure", "dflash_check_guards")
TRACE_GEMM, TRACE_APPEND, TRACE_DRAFT, TRACE_VERIFY, TRACE_ENGINE = 0, 1, 2, 3, 4


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_target_layers", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("mask_token_id", ctypes.c_int32), ("k_max", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("kv_pool_tokens", ctypes.c_int64), ("conditioning", ctypes.c_int32)]


class TargetConfigC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("r_max", ctypes.c_int32), ("n_feat", ctypes.c_int32), ("feat_layers", ctypes.c_int32 * 8),
                ("kv_pool_tokens", ctypes.c_int64)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("w_fc", ctypes.c_void_p), ("fc_norm", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", LayerWeights * MAX_LAYERS)]


_lib = None


def load_library(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libdflash.so (building it in-tree first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_needed and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libdflash.so not built ({_build.LIB}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_build.LIB)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.dflash_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i32, ctypes.POINTER(vp)]
    lib.dflash_destroy.argtypes = [vp]
    lib.dflash_reserve.argtypes = [vp, i32, vp]
    lib.dflash_reserve_headroom.argtypes = [vp, i32, vp]
    lib.dflash_ctx_append.argtypes = [vp, vp, i32, vp, vp]
    lib.dflash_draft_block.argtypes = [vp, vp, i32, vp, vp, vp]
    lib.dflash_draft_block_k.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.dflash_verify_accept.argtypes = [vp, vp, vp, vp, vp]
    lib.dflash_query_state.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dflash_last_error.argtypes = []
    lib.dflash_last_error.restype = ctypes.c_char_p
    lib.dflash_plant_targets.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i32, vp]
    lib.dflash_trace_enable.argtypes = [vp, i32]
    lib.dflash_trace_read.argtypes = [vp, i32, vp, vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.dflash_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
    lib.dflash_graph_replays.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
    lib.dflash_read_kv.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp]
    lib.dflash_draft_block_noalloc.argtypes = [vp, vp, i32, vp, vp, vp]
    lib.dflash_target_create.argtypes = [ctypes.POINTER(TargetConfigC), ctypes.POINTER(Weights), i32,
                                         ctypes.POINTER(vp)]
    lib.dflash_target_destroy.argtypes = [vp]
    lib.dflash_target_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.dflash_target_commit.argtypes = [vp, vp, vp]
    lib.dflash_target_query.argtypes = [vp, vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dflash_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
    lib.dflash_selftest_wait.argtypes = [vp, vp]
    lib.dflash_inject_alloc_failure.argtypes = [ctypes.c_int64]
    lib.dflash_check_guards.argtypes = [vp, vp]
    for name in EXPORTS:
        if name not in ("dflash_last_error", "dflash_inject_alloc_failure"):
            getattr(lib, name).restype = ctypes.c_int
    lib.dflash_inject_alloc_failure.restype = ctypes.c_int64
    _lib = lib
    return lib


def _check(code: int) -> None:
    if code != 0:
        msg = _lib.dflash_last_error().decode(errors="replace")
        raise DflashError(code, msg)


def ptr(x) -> Optional[int]:
    """Raw address of a contiguous torch tensor / numpy array (host or device), or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy array must be C-contiguous")
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class DrafterConfig:
    hidden: int
    n_target_layers: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rope_theta: float
    rms_eps: float
    mask_token_id: int
    k_max: int
    dtype: str = "bf16"
    kv_pool_tokens: int = 0
    conditioning: str = "kv"   # "kv" (context K/V injection), "input" (input fusion), "none"

    @classmethod
    def from_shape(cls, s, **kw) -> "DrafterConfig":
        vals = dict(hidden=s.hidden, n_target_layers=s.n_target_layers, n_layers=s.n_layers,
                    n_q_heads=s.n_q_heads, n_kv_heads=s.n_kv_heads, head_dim=s.head_dim,
                    intermediate=s.intermediate, vocab=s.vocab, rope_theta=s.rope_theta, rms_eps=s.rms_eps,
                    mask_token_id=s.mask_token_id, k_max=getattr(s, "k_max", getattr(s, "K_max", None)),
                    dtype=s.dtype)
        vals.update(kw)
        return cls(**vals)

    def to_c(self) -> Config:
        return Config(self.hidden, self.n_target_layers, self.n_layers, self.n_q_heads, self.n_kv_heads,
                      self.head_dim, self.intermediate, self.vocab, float(self.rope_theta), float(self.rms_eps),
                      self.mask_token_id, self.k_max, DTYPES[self.dtype], int(self.kv_pool_tokens),
                      CONDITIONING[self.conditioning])


class DFlashDrafter:
    """One proposer context (libdflash ``dflash_ctx``) over `batch` sequences.

    `weights` maps the names ``embed, w_fc, fc_norm, final_norm, lm_head`` and
    ``layers.<l>.{wq,wk,wv,wo,w_gate,w_up,w_down,attn_norm,mlp_norm}`` to
    contiguous device tensors (fp32, or bf16 for dtype "bf16"); they are
    borrowed and kept alive by this object.
    """

    def __init__(self, cfg: DrafterConfig, weights: Dict[str, object], batch: int):
        self.lib = load_library()
        self.cfg = cfg
        self.batch = int(batch)
        self._weights = weights
        w = Weights()
        w.embed, w.w_fc, w.fc_norm = ptr(weights["embed"]), ptr(weights["w_fc"]), ptr(weights["fc_norm"])
        w.final_norm, w.lm_head = ptr(weights["final_norm"]), ptr(weights["lm_head"])
        for l in range(cfg.n_layers):
            lw = w.layers[l]
            for f in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm"):
                setattr(lw, f, ptr(weights[f"layers.{l}.{f}"]))
        c = cfg.to_c()
        h = ctypes.c_void_p()
        _check(self.lib.dflash_create(ctypes.byref(c), ctypes.byref(w), self.batch, ctypes.byref(h)))
        self.handle = h

    # -- the three calls of the hot path ----------------------------------
    def ctx_append(self, feats, rows_max: int, rows=None, stream=None) -> None:
        _check(self.lib.dflash_ctx_append(self.handle, ptr(feats), int(rows_max), ptr(rows), _stream(stream)))

    def draft_block(self, K: int, anchor_ids=None, draft_ids=None, logits=None, stream=None, k_seq=None) -> None:
        """k_seq: optional int32 [B] block length per sequence (each in [1, K]); ids past it are -1."""
        if k_seq is None:
            _check(self.lib.dflash_draft_block(self.handle, ptr(anchor_ids), int(K), ptr(draft_ids), ptr(logits),
                                               _stream(stream)))
        else:
            _check(self.lib.dflash_draft_block_k(self.handle, ptr(anchor_ids), int(K), ptr(k_seq), ptr(draft_ids),
                                                 ptr(logits), _stream(stream)))

    def draft_block_noalloc(self, K: int, anchor_ids=None, draft_ids=None, logits=None, stream=None) -> None:
        """draft_block without any device allocation (static split-KV scratch; frozen workspaces)."""
        _check(self.lib.dflash_draft_block_noalloc(self.handle, ptr(anchor_ids), int(K), ptr(draft_ids),
                                                   ptr(logits), _stream(stream)))

    def verify_accept(self, target_ids, accept_len=None, next_anchor=None, stream=None) -> None:
        _check(self.lib.dflash_verify_accept(self.handle, ptr(target_ids), ptr(accept_len), ptr(next_anchor),
                                             _stream(stream)))

    # -- state -------------------------------------------------------------------
    def reserve(self, min_capacity: int, stream=None) -> None:
        _check(self.lib.dflash_reserve(self.handle, int(min_capacity), _stream(stream)))

    def reserve_headroom(self, headroom: int, stream=None) -> None:
        """Grow each sequence's KV capacity to its own context + headroom slots."""
        _check(self.lib.dflash_reserve_headroom(self.handle, int(headroom), _stream(stream)))

    def query_state(self, stream=None, raise_on_flags: bool = True) -> dict:
        B = self.batch
        out = {k: np.zeros(B, np.int32) for k in ("ctx_len", "kv_len", "capacity", "anchor")}
        flags = ctypes.c_uint32(0)
        code = self.lib.dflash_query_state(self.handle, _stream(stream), ptr(out["ctx_len"]), ptr(out["kv_len"]),
                                           ptr(out["capacity"]), ptr(out["anchor"]), ctypes.byref(flags))
        out["flags"] = int(flags.value)
        if code != 0 and (code != 5 or raise_on_flags):
            _check(code)
        return out

    # -- tracing -----------------------------------------------------------------
    def trace_enable(self, n_pairs: int) -> None:
        _check(self.lib.dflash_trace_enable(self.handle, int(n_pairs)))

    def trace_read(self, max_entries: int = 65536):
        kind = np.zeros(max_entries, np.int32)
        ms = np.zeros(max_entries, np.float32)
        nbytes = np.zeros(max_entries, np.float64)
        n = ctypes.c_int32(0)
        _check(self.lib.dflash_trace_read(self.handle, int(max_entries), ptr(kind), ptr(ms), ptr(nbytes),
                                          ctypes.byref(n)))
        k = n.value
        return kind[:k], ms[:k], nbytes[:k]

    def read_kv(self, seq: int, layer: int, kind: int, slot0: int, n_slots: int, stream=None) -> np.ndarray:
        """KV rows [n_kv_heads, n_slots, head_dim] (fp32 values; bf16 contexts are widened)."""
        c = self.cfg
        bf16 = c.dtype == "bf16"
        out = np.zeros((c.n_kv_heads, n_slots, c.head_dim), np.uint16 if bf16 else np.float32)
        _check(self.lib.dflash_read_kv(self.handle, int(seq), int(layer), int(kind), int(slot0), int(n_slots),
                                       ptr(out), _stream(stream)))
        if bf16:
            return (out.astype(np.uint32) << np.uint32(16)).view(np.float32)
        return out

    def launch_count(self) -> int:
        v = ctypes.c_int64(0)
        _check(self.lib.dflash_launch_count(self.handle, ctypes.byref(v)))
        return int(v.value)

    def graph_replays(self) -> int:
        """Drafts served by replaying the recorded graph."""
        v = ctypes.c_int64(0)
        _check(self.lib.dflash_graph_replays(self.handle, ctypes.byref(v)))
        return int(v.value)

    # -- failure detection ----------------------------------------------------
    def set_wait_limit(self, limit_ns: int) -> None:
        """Time limit of every bounded device wait of this context (0: the 2 s default)."""
        _check(self.lib.dflash_set_wait_limit(self.handle, int(limit_ns)))

    def selftest_wait(self, stream=None) -> None:
        """One kernel whose wait nothing ends: it runs out and latches FLAG_WAIT_TIMEOUT."""
        _check(self.lib.dflash_selftest_wait(self.handle, _stream(stream)))

    def check_guards(self, stream=None) -> None:
        """Raise DflashError if a guard band around the KV arena was written."""
        _check(self.lib.dflash_check_guards(self.handle, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.dflash_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def inject_alloc_failure(after: int) -> int:
    """Make the after-th next device allocation of the library fail once (after < 0: off).
    Returns the previous setting."""
    return int(load_library().dflash_inject_alloc_failure(int(after)))


def plant_targets(draft_ids, accept_len_plan, fill, batch: int, K: int, vocab: int, target_ids,
                  step_counter=None, n_plans: int = 1, stream=None) -> None:
    """Synthetic-input harness kernel: target ids that force planted accept lengths."""
    lib = load_library()
    _check(lib.dflash_plant_targets(ptr(draft_ids), ptr(accept_len_plan), ptr(fill), int(batch), int(K),
                                    int(vocab), ptr(target_ids), ptr(step_counter), int(n_plans), _stream(stream)))


@dataclass
class TargetConfig:
    """Shape of the target model whose verify forward dflash_target_* runs."""
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rope_theta: float
    rms_eps: float
    r_max: int
    feat_layers: Tuple[int, ...] = ()
    kv_pool_tokens: int = 0

    @classmethod
    def from_shape(cls, s, r_max: int, feat_layers=(), **kw) -> "TargetConfig":
        vals = dict(hidden=s.hidden, n_layers=s.n_layers, n_q_heads=s.n_q_heads, n_kv_heads=s.n_kv_heads,
                    head_dim=s.head_dim, intermediate=s.intermediate, vocab=s.vocab, rope_theta=s.rope_theta,
                    rms_eps=s.rms_eps, r_max=r_max, feat_layers=tuple(feat_layers))
        vals.update(kw)
        return cls(**vals)

    def to_c(self) -> TargetConfigC:
        c = TargetConfigC()
        for f in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab", "r_max"):
            setattr(c, f, int(getattr(self, f)))
        c.rope_theta, c.rms_eps = float(self.rope_theta), float(self.rms_eps)
        c.n_feat = len(self.feat_layers)
        for i, l in enumerate(self.feat_layers):
            c.feat_layers[i] = int(l)
        c.kv_pool_tokens = int(self.kv_pool_tokens)
        return c


class DFlashTarget:
    """The target model's verify forward (libdflash ``dflash_target``) over `batch`
    sequences; `weights` as for DFlashDrafter (bf16 device tensors; w_fc and
    fc_norm are not needed)."""

    def __init__(self, cfg: TargetConfig, weights: Dict[str, object], batch: int):
        self.lib = load_library()
        self.cfg = cfg
        self.batch = int(batch)
        self._weights = weights
        w = Weights()
        w.embed, w.final_norm, w.lm_head = ptr(weights["embed"]), ptr(weights["final_norm"]), ptr(weights["lm_head"])
        for l in range(cfg.n_layers):
            lw = w.layers[l]
            for f in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "mlp_norm"):
                setattr(lw, f, ptr(weights[f"layers.{l}.{f}"]))
        c = cfg.to_c()
        h = ctypes.c_void_p()
        _check(self.lib.dflash_target_create(ctypes.byref(c), ctypes.byref(w), self.batch, ctypes.byref(h)))
        self.handle = h

    def forward(self, tokens, ids, logits=None, feats=None, stream=None) -> None:
        """tokens: int32 [batch, R] device; ids out [batch, R]; logits [batch, R, V]
        float32 and feats [batch, R, n_feat * hidden] bf16 (device) or None."""
        R = int(tokens.shape[1])
        _check(self.lib.dflash_target_forward(self.handle, ptr(tokens), R, ptr(ids), ptr(logits), ptr(feats),
                                              _stream(stream)))

    def commit(self, keep, stream=None) -> None:
        """keep: int32 [batch] (host numpy or device) rows of the last forward to keep."""
        if isinstance(keep, np.ndarray):
            keep = np.ascontiguousarray(keep, np.int32)
        _check(self.lib.dflash_target_commit(self.handle, ptr(keep), _stream(stream)))

    def query(self, stream=None) -> np.ndarray:
        ln = np.zeros(self.batch, np.int32)
        flags = ctypes.c_uint32(0)
        _check(self.lib.dflash_target_query(self.handle, _stream(stream), ptr(ln), ctypes.byref(flags)))
        return ln

    # -- failure detection ----------------------------------------------------
    def set_wait_limit(self, limit_ns: int) -> None:
        """Time limit of every bounded device wait of this context (0: the 2 s default)."""
        _check(self.lib.dflash_set_wait_limit(self.handle, int(limit_ns)))

    def selftest_wait(self, stream=None) -> None:
        """One kernel whose wait nothing ends: it runs out and latches FLAG_WAIT_TIMEOUT."""
        _check(self.lib.dflash_selftest_wait(self.handle, _stream(stream)))

    def check_guards(self, stream=None) -> None:
        """Raise DflashError if a guard band around the KV arena was written."""
        _check(self.lib.dflash_check_guards(self.handle, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.lib.dflash_target_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

