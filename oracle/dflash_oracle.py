"""CPU oracle of the DFlash drafter hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The library path never calls it, and it
shares no code with the CUDA kernels: it receives the same seeded input bits
(from ``synth``) and computes the plain definitions below with numpy, in fp64
by default (fp32 only for the timed CPU baseline).  Nothing is blocked, fused
or reordered beyond what the definitions state: attention is the matrix form
softmax(Q K^T / sqrt(d)) V per sequence and head, with no online softmax and no
KV splitting; the accept rule is a literal loop.

Pages followed (web write-ups of DFlash; cited by title and section):
  [GDB] "在谷歌TPU上实现3倍加速：UCSD利用扩散式推测解码优化LLM推理"
        (AI translation of the Google Developers Blog post on DFlash on TPU)
  [KCH] "D-Flash：扩散草稿让大模型推理提速3.5倍的秘密" (summary of the DFlash paper)
  [UPJ] upppp.jp summary "DFlash（Block Diffusion for Flash Speculative Decoding）"

What each function computes, and where the pages leave a step open, the
reading taken (all readings are listed in the design notes):
  * ctx_append  -- [KCH §系统架构]: features of several target layers are
    concatenated and projected by a light fc layer into one target context
    feature; [KCH §创新二]: that feature goes through every draft layer's K and
    V projections and is stored as a persistent, reused KV cache.  Reading: an
    RMSNorm follows fc; each layer applies its own W_k / W_v to the normalised
    feature directly (no per-layer input norm); K gets RoPE at the token's
    absolute position.  [GDB §智能上下文管理]: the proposer tracks exactly how
    much context it has consumed (``kv_len`` here).
  * draft       -- [KCH §系统架构, §创新一]: the known token (anchor) and K mask
    tokens enter the draft layers together and all masks are predicted in one
    forward; draft layers are bidirectional attention + MLP; the target's LM
    head yields the logits.  [GDB §用于注意力机制的“双缓存”方案]: block
    attention is non-causal.  Readings: pre-norm decoder layers with RMSNorm,
    GQA, rotate-half RoPE, SwiGLU MLP, a final RMSNorm before the LM head; no
    attention mask at all (every block row sees all context keys and all block
    keys); block row j sits at position ctx_len + j; drafts come from the K
    mask rows; greedy argmax with the lowest index on ties ([GDB] Table 2
    caption: greedy decoding).
  * verify      -- [GDB §克服自回归瓶颈]: the target verifies the drafts in one
    parallel forward and keeps the correct ones; [KCH §系统架构]: the final
    result is decided by the target.  Reading: accept the longest prefix of
    drafts equal to the target's argmax; the bonus token is the target's argmax
    after the last accepted draft.  [GDB §弥合 TPU 推理中的元数据鸿沟] and
    [UPJ メタデータの同期]: the context buffer, KV positions and RoPE offset
    advance by the truly accepted count, never by the verified block length.

Parity status: each function is pinned by the CPU tests (closed forms,
invariants, library routines on special cases, brute force on tiny inputs).
The full drafter's logits have no worked example on the pages, so the complete
forward is pinned only through those internal checks.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# storage decoding

def decode(a: np.ndarray, dtype=np.float64) -> np.ndarray:
    """bf16 bit patterns (uint16) or fp32 values -> floating array of `dtype`."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        f = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
        return f.astype(dtype)
    return a.astype(dtype)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    bf16 keeps the top 16 bits of an IEEE fp32 word; rounding adds half a unit
    of the dropped 16 bits (0x7FFF, plus 1 when the kept part is odd) before
    truncating.  Values are first rounded to fp32 (exact for what the kernels
    store, which is computed in fp32 or finer).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# building blocks (plain definitions)

def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def rope_inv_freq(head_dim: int, theta: float, dtype=np.float64) -> np.ndarray:
    """Rotary frequencies theta^(-2i/d), i = 0 .. d/2-1."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return (float(theta) ** (-2.0 * i / head_dim)).astype(dtype)


def apply_rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  x: [n, heads, d]; pos: [n] absolute positions.

    Pair (i, i + d/2) of each head is rotated by the angle pos * theta^(-2i/d):
    (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin).
    """
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, theta)[None, :]
    cos = np.cos(ang).astype(x.dtype)[:, None, :]
    sin = np.sin(ang).astype(x.dtype)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def softmax(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Unmasked (bidirectional) grouped-query attention.

    q: [Rq, n_q, d]; k, v: [T, n_kv, d].  Query head h reads KV head
    h // (n_q / n_kv); scores are scaled by d^-1/2; every query sees every key.
    Returns [Rq, n_q, d].
    """
    n_q, d = q.shape[1], q.shape[2]
    n_kv = k.shape[1]
    group = n_q // n_kv
    out = np.empty_like(q)
    scale = 1.0 / np.sqrt(d)
    for h in range(n_q):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        p = softmax((q[:, h, :] @ kh.T) * scale)
        out[:, h, :] = p @ vh
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """SwiGLU MLP: W_down (silu(W_gate x) * (W_up x)); weights are [out, in]."""
    return (silu(x @ w_gate.T) * (x @ w_up.T)) @ w_down.T


def greedy_argmax(z: np.ndarray) -> np.ndarray:
    """Argmax over the last axis; np.argmax returns the first (lowest) index of ties."""
    return np.argmax(z, axis=-1).astype(np.int32)


def accept_prefix(drafts: Sequence[int], targets: Sequence[int]) -> Tuple[int, int]:
    """Greedy verify of one sequence.

    drafts: d_1..d_K; targets: g_0..g_K, g_{j-1} being the target's argmax at
    the position where d_j was proposed.  Returns (n, bonus) with n the length
    of the longest prefix where d_j == g_{j-1} and bonus = g_n.
    """
    K = len(drafts)
    n = 0
    while n < K and int(drafts[n]) == int(targets[n]):
        n += 1
    return n, int(targets[n])


# ----------------------------------------------------------------------------
# the stateful drafter

@dataclass
class SeqState:
    ctx_len: int = 0      # committed tokens = absolute position of the anchor
    kv_len: int = 0       # context rows whose K/V are stored ("consumed")
    anchor: int = 0
    k: List[np.ndarray] = field(default_factory=list)   # per layer [kv_len, n_kv, d]
    v: List[np.ndarray] = field(default_factory=list)
    u_last: Optional[np.ndarray] = None                  # input fusion: context feature of the last row


class OracleDrafter:
    """Plain numpy drafter: ctx_append / draft / verify over B sequences.

    `weights` maps the names produced by synth.inputs.weight_shapes to arrays
    (bf16 bits or fp32); `shape` is a synth DrafterShape (or anything with the
    same attributes).  `dtype` is the arithmetic type (fp64 for parity).
    """

    # How the target context conditions the draft ("KCH" page, sections on the
    # target-feature KV injection and on the ablations):
    #   "kv"    -- the context feature of every consumed row is projected by each
    #              draft layer's W_k / W_v into that layer's KV cache (the method);
    #   "input" -- input fusion, the ablation's EAGLE-style alternative: the
    #              context feature is fused into the draft's input embeddings once
    #              and no layer sees context keys.  Reading taken here: the context
    #              feature u of the sequence's most recent consumed row is added to
    #              the embedding of every block row (same u = RMSNorm(W_fc f), same
    #              shape as an embedding; the pages give no formula);
    #   "none"  -- all target context removed: the block attends only to itself.
    CONDITIONING = ("kv", "input", "none")

    def __init__(self, shape, weights: Dict[str, np.ndarray], batch: int,
                 dtype=np.float64, pos_offset: int = 0, use_rope: bool = True, conditioning: str = "kv"):
        if conditioning not in self.CONDITIONING:
            raise ValueError(conditioning)
        self.cond = conditioning
        self.s = shape
        self.raw = weights
        self.dtype = dtype
        self.pos_offset = int(pos_offset)   # test hook: shifts every RoPE position
        self.use_rope = use_rope            # test hook: RoPE off for equivariance checks
        self.seqs = [SeqState(k=[np.zeros((0, shape.n_kv_heads, shape.head_dim), dtype)
                                 for _ in range(shape.n_layers)],
                              v=[np.zeros((0, shape.n_kv_heads, shape.head_dim), dtype)
                                 for _ in range(shape.n_layers)])
                     for _ in range(batch)]
        self._cache: Dict[str, np.ndarray] = {}

    # -- weights ---------------------------------------------------------
    def w(self, name: str) -> np.ndarray:
        a = self._cache.get(name)
        if a is None:
            a = decode(self.raw[name], self.dtype)
            if a.size <= (1 << 27):       # keep all but the two vocab-sized tables
                self._cache[name] = a
        return a

    def _norm_proj(self, h: np.ndarray, gain: np.ndarray, mats):
        """[RMSNorm(h) W^T for W in mats]."""
        x = rms_norm(h, gain, self.s.rms_eps)
        return [x @ W.T for W in mats]

    def _rope(self, x: np.ndarray, pos: np.ndarray) -> np.ndarray:
        if not self.use_rope:
            return x
        return apply_rope(x, pos + self.pos_offset, self.s.rope_theta)

    # -- context append ----------------------------------------------------
    def ctx_append(self, b: int, feats: np.ndarray) -> None:
        """Project `rows` target feature rows of sequence b into every layer's KV.

        feats: [rows, L_t * H] (the L_t features of a token back to back).
        Rows land at positions kv_len .. kv_len + rows - 1.
        """
        s = self.s
        st = self.seqs[b]
        x = decode(feats, self.dtype)
        rows = x.shape[0]
        if rows == 0:
            return
        if self.cond != "kv":   # the rows are consumed, but no layer stores context K/V
            if self.cond == "input":
                y = x[-1:] @ self.w("w_fc").T
                st.u_last = rms_norm(y, self.w("fc_norm"), s.rms_eps)[0]
            st.kv_len += rows
            st.ctx_len = max(st.ctx_len, st.kv_len)
            return
        y = x @ self.w("w_fc").T
        pos = np.arange(st.kv_len, st.kv_len + rows)
        for l in range(s.n_layers):
            p = f"layers.{l}."
            k, v = self._norm_proj(y, self.w("fc_norm"), [self.w(p + "wk"), self.w(p + "wv")])
            k = k.reshape(rows, s.n_kv_heads, s.head_dim)
            v = v.reshape(rows, s.n_kv_heads, s.head_dim)
            st.k[l] = np.concatenate([st.k[l], self._rope(k, pos)], axis=0)
            st.v[l] = np.concatenate([st.v[l], v], axis=0)
        st.kv_len += rows
        st.ctx_len = max(st.ctx_len, st.kv_len)

    def set_anchor(self, b: int, token: int) -> None:
        self.seqs[b].anchor = int(token)

    # -- one block-diffusion draft ----------------------------------------------
    def draft(self, K: int, anchors: Optional[Sequence[int]] = None,
              block_embeds: Optional[np.ndarray] = None, seqs: Optional[Sequence[int]] = None,
              want_logits: bool = True, want_hidden: bool = False):
        """One non-causal forward over [anchor ; K masks] for the selected sequences.

        Returns (drafts int32 [B', K], logits [B', K, V] or None[, final hidden]).
        `block_embeds` ([B', K+1, H]) replaces the embedding lookup (test hook).
        """
        s = self.s
        seqs = list(range(len(self.seqs))) if seqs is None else list(seqs)
        Bs, R, H = len(seqs), K + 1, s.hidden
        for b in seqs:
            st = self.seqs[b]
            if st.kv_len != st.ctx_len:
                raise ValueError(f"sequence {b}: context not consumed "
                                 f"(kv_len {st.kv_len} != ctx_len {st.ctx_len})")
        if block_embeds is None:
            E = self.raw["embed"]
            h = np.empty((Bs, R, H), self.dtype)
            for i, b in enumerate(seqs):
                a = self.seqs[b].anchor if anchors is None else int(anchors[i])
                h[i, 0] = decode(E[a], self.dtype)
                h[i, 1:] = decode(E[s.mask_token_id], self.dtype)[None, :]
        else:
            h = np.array(block_embeds, dtype=self.dtype)
        if self.cond == "input":   # input fusion: the last context feature on every block row
            for i, b in enumerate(seqs):
                u = self.seqs[b].u_last
                if u is not None:
                    h[i] = h[i] + u[None, :]

        for l in range(s.n_layers):
            p = f"layers.{l}."
            q, k, v = self._norm_proj(h, self.w(p + "attn_norm"),
                                      [self.w(p + "wq"), self.w(p + "wk"), self.w(p + "wv")])
            q = q.reshape(Bs, R, s.n_q_heads, s.head_dim)
            k = k.reshape(Bs, R, s.n_kv_heads, s.head_dim)
            v = v.reshape(Bs, R, s.n_kv_heads, s.head_dim)
            o = np.empty((Bs, R, s.q_dim), self.dtype)
            for i, b in enumerate(seqs):
                st = self.seqs[b]
                pos = st.ctx_len + np.arange(R)
                qb = self._rope(q[i], pos)
                kb = self._rope(k[i], pos)
                if self.cond == "kv":
                    keys = np.concatenate([st.k[l], kb], axis=0)
                    vals = np.concatenate([st.v[l], v[i]], axis=0)
                else:   # no context keys: the block attends to itself only
                    keys, vals = kb, v[i]
                o[i] = attention(qb, keys, vals).reshape(R, s.q_dim)
            h = h + o @ self.w(p + "wo").T
            x = rms_norm(h, self.w(p + "mlp_norm"), s.rms_eps)
            h = h + swiglu(x, self.w(p + "w_gate"), self.w(p + "w_up"), self.w(p + "w_down"))

        hm = h[:, 1:, :].reshape(Bs * K, H)   # the K mask rows
        xf = rms_norm(hm, self.w("final_norm"), s.rms_eps)
        logits = self.lm_head(xf).reshape(Bs, K, s.vocab)
        xf = xf.reshape(Bs, K, H)
        drafts = greedy_argmax(logits)
        out = (drafts, logits if want_logits else None)
        return out + (xf,) if want_hidden else out

    def draft_k(self, ks: Sequence[int], anchors: Optional[Sequence[int]] = None,
                seqs: Optional[Sequence[int]] = None, want_logits: bool = True):
        """A block length per sequence: sequence seqs[i] drafts ks[i] masks, i.e.
        its own forward over [anchor ; ks[i] masks] (the block is non-causal, so a
        shorter block is a different forward, not a truncated one).  Returns ids
        [B', max ks] padded with -1 and logits [B', max ks, V] padded with NaN."""
        seqs = list(range(len(self.seqs))) if seqs is None else list(seqs)
        Kmax = int(max(ks))
        ids = np.full((len(seqs), Kmax), -1, np.int32)
        logits = np.full((len(seqs), Kmax, self.s.vocab), np.nan, self.dtype) if want_logits else None
        for i, b in enumerate(seqs):
            k = int(ks[i])
            a = None if anchors is None else [int(anchors[i])]
            d, z = self.draft(k, anchors=a, seqs=[b], want_logits=want_logits)
            ids[i, :k] = d[0]
            if want_logits:
                logits[i, :k] = z[0]
        return ids, logits

    def lm_head(self, x: np.ndarray, chunk: int = 32768) -> np.ndarray:
        """logits = x W_lm^T, evaluated over vocabulary chunks to bound memory."""
        W = self.raw["lm_head"]
        out = np.empty((x.shape[0], W.shape[0]), self.dtype)
        for lo in range(0, W.shape[0], chunk):
            out[:, lo:lo + chunk] = x @ decode(W[lo:lo + chunk], self.dtype).T
        return out

    # -- greedy verify and state advance -------------------------------------
    def verify(self, drafts: np.ndarray, targets: np.ndarray,
               seqs: Optional[Sequence[int]] = None,
               ks: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
        """Accept the longest matching prefix per sequence and advance the state
        (ks: each sequence's own block length, default the drafts' width).

        ctx_len (the RoPE offset / KV position of the next anchor) moves by the
        accepted count n plus the anchor itself; the bonus g_n becomes the next
        anchor.  kv_len is left for the next ctx_append of those n + 1 rows.
        """
        seqs = list(range(len(self.seqs))) if seqs is None else list(seqs)
        n_out = np.zeros(len(seqs), np.int32)
        a_out = np.zeros(len(seqs), np.int32)
        for i, b in enumerate(seqs):
            k = len(drafts[i]) if ks is None else int(ks[i])   # the sequence's own block length
            n, bonus = accept_prefix(drafts[i][:k], targets[i][:k + 1])
            st = self.seqs[b]
            st.ctx_len += n + 1
            st.anchor = bonus
            n_out[i], a_out[i] = n, bonus
        return n_out, a_out
