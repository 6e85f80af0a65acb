// Epilogue helpers of the tensor-core GEMMs, run by a group of four warps
// (128 threads, epilogue thread r = TMEM lane r = weight-tile row r) that meet
// on named barrier 1: split-K reduction in split order, the folded RMSNorm row
// scale, RoPE + KV-slot writes, residual + sums of squares, SwiGLU, and the
// bounded cross-CTA counter waits.  Shared by the tensor-core GEMM kernel's
// instances.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr int kEpiChunk = 32;                 // tokens per epilogue shared-memory chunk
constexpr int kEpiLd = kTileRows + 1;         // padded row of the epilogue chunk

// named barrier of the four epilogue warps
__device__ __forceinline__ void epi_bar(int id = 1) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
// both epilogue halves of a direct GEMM CTA (256 threads)
__device__ __forceinline__ void epi_pair_bar() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// acc[i] += sum over splits s0 .. s0+NS-1 (< S), in split order, of the
// partials of tokens t0 + i (i < n <= TN) in column b.  Every load is issued
// before the first is used (indices clamped to valid ones, the surplus masked
// when summing: adding 0 leaves a sum unchanged), so a batch costs one L2 round
// trip; NS * TN = 32 loads per batch whatever the token count.
constexpr int kRedTok = 8;
template <int NS, int TN>
__device__ __forceinline__ void red_batch(const float* b, size_t stride, size_t ld, int s0, int S, int n,
                                          float (&acc)[kRedTok]) {
  float v[NS][TN];
#pragma unroll
  for (int sp = 0; sp < NS; ++sp)
#pragma unroll
    for (int i = 0; i < TN; ++i) v[sp][i] = __ldcg(b + (size_t)min(s0 + sp, S - 1) * stride + (size_t)min(i, n - 1) * ld);
#pragma unroll
  for (int sp = 0; sp < NS; ++sp)
#pragma unroll
    for (int i = 0; i < TN; ++i) acc[i] += (s0 + sp < S && i < n) ? v[sp][i] : 0.f;
}
template <int NS, int TN>
__device__ __forceinline__ void red_batches(const float* b, size_t stride, size_t ld, int S, int n,
                                            float (&acc)[kRedTok]) {
  for (int s0 = 0; s0 < S; s0 += NS) red_batch<NS, TN>(b, stride, ld, s0, S, n, acc);
}
// acc[i] = sum over every split, in split order, of the partials of tokens
// t0 + i (i < n <= kRedTok) in column col: the batch shape follows n so that
// the few tokens of a small slice take all splits in one round trip.
__device__ __forceinline__ void red_tokens(const EpiArgs& p, int t0, int n, int col, float (&acc)[kRedTok]) {
  const size_t stride = (size_t)p.M * p.N, ld = (size_t)p.N;
  const float* b = p.ws + (size_t)t0 * p.N + col;
  const int S = p.splits;
#pragma unroll
  for (int i = 0; i < kRedTok; ++i) acc[i] = 0.f;
  if (n > 4)
    red_batches<4, 8>(b, stride, ld, S, n, acc);
  else if (n > 2)
    red_batches<8, 4>(b, stride, ld, S, n, acc);
  else if (n > 1)
    red_batches<16, 2>(b, stride, ld, S, n, acc);
  else
    red_batches<32, 1>(b, stride, ld, S, n, acc);
}
// the same for two columns at once (the gate and up halves of a SwiGLU pair):
// both columns' loads of a batch in flight together
template <int NS, int TN>
__device__ __forceinline__ void red_batches2(const float* b0, const float* b1, size_t stride, size_t ld, int S, int n,
                                             float (&a0)[kRedTok], float (&a1)[kRedTok]) {
  for (int s0 = 0; s0 < S; s0 += NS) {
    float v0[NS][TN], v1[NS][TN];
#pragma unroll
    for (int sp = 0; sp < NS; ++sp)
#pragma unroll
      for (int i = 0; i < TN; ++i) {
        const size_t off = (size_t)min(s0 + sp, S - 1) * stride + (size_t)min(i, n - 1) * ld;
        v0[sp][i] = __ldcg(b0 + off);
        v1[sp][i] = __ldcg(b1 + off);
      }
#pragma unroll
    for (int sp = 0; sp < NS; ++sp)
#pragma unroll
      for (int i = 0; i < TN; ++i) {
        const bool m = s0 + sp < S && i < n;
        a0[i] += m ? v0[sp][i] : 0.f;
        a1[i] += m ? v1[sp][i] : 0.f;
      }
  }
}
__device__ __forceinline__ void red_tokens2(const EpiArgs& p, int t0, int n, int col0, int col1, float (&a0)[kRedTok],
                                            float (&a1)[kRedTok]) {
  const size_t stride = (size_t)p.M * p.N, ld = (size_t)p.N;
  const float* b0 = p.ws + (size_t)t0 * p.N + col0;
  const float* b1 = p.ws + (size_t)t0 * p.N + col1;
  const int S = p.splits;
#pragma unroll
  for (int i = 0; i < kRedTok; ++i) a0[i] = a1[i] = 0.f;
  if (n > 4)
    red_batches2<2, 8>(b0, b1, stride, ld, S, n, a0, a1);
  else if (n > 2)
    red_batches2<4, 4>(b0, b1, stride, ld, S, n, a0, a1);
  else if (n > 1)
    red_batches2<8, 2>(b0, b1, stride, ld, S, n, a0, a1);
  else
    red_batches2<16, 1>(b0, b1, stride, ld, S, n, a0, a1);
}

// Split-K sums of this thread's output column(s), token by token:
// red(which, t0, n, acc) sums tokens t0 .. t0+n-1 of tile `which` (0, or 1 for
// the up half of a gate/up pair) over every split, in split order.

// partials in global memory, ws[split][t][n]
struct GlobalRed {
  static constexpr bool kTmem = false;
  const EpiArgs* p;
  int col[2];
  __device__ __forceinline__ void operator()(int which, int t0, int n, float (&acc)[kRedTok]) const {
    red_tokens(*p, t0, n, col[which], acc);
  }
  __device__ __forceinline__ void pair(int t0, int n, float (&a0)[kRedTok], float (&a1)[kRedTok]) const {
    red_tokens2(*p, t0, n, col[0], col[1], a0, a1);
  }
};

// A tile with a single split: its sums are the CTA's own accumulator in
// tensor memory (thread r = lane r), read straight from there -- no partials
// leave the SM.  Token t = n0 + i * bn + c (token tile i of the CTA) is column
// i * (bn + lo) + c, its lo-plane half `lo` columns further for a split operand
// (lo = bn; 0 for a plain one); the up half of a gate/up pair computed by the
// same CTA starts `up` columns further.  Callers pass groups of 8 tokens that
// start on a multiple of 8 from n0 (bn is one too), so a group never straddles
// two tiles.  Every call is warp-uniform.
struct TmemRed {
  static constexpr bool kTmem = true;
  uint32_t taddr;   // column 0 of this warp's 32 lanes
  int n0, bn, lo, up;
  // tokens t0 .. t0 + T - 1 (those below t0 + n) of tile `which` in one batch of
  // loads and one wait; groups past n are not read (acc 0)
  template <int T>
  __device__ __forceinline__ void chunk(int which, int t0, int n, float (&acc)[T]) const {
    static_assert(T % 8 == 0, "groups of 8 columns");
    uint32_t h[T], l[T];
#pragma unroll
    for (int i = 0; i < T; ++i) h[i] = l[i] = 0u;
#pragma unroll
    for (int g = 0; g < T / 8; ++g) {
      if (g * 8 < n) {   // warp-uniform
        const int d = t0 - n0 + g * 8;
        const uint32_t a = taddr + (uint32_t)(d + (d / bn) * lo + which * up);
        tmem_ld8_issue(a, h + g * 8);
        if (lo != 0) tmem_ld8_issue(a + (uint32_t)lo, l + g * 8);
      }
    }
    tmem_wait_ld_all();
#pragma unroll
    for (int g = 0; g < T / 8; ++g) {
      tmem_hold8(h + g * 8);
      tmem_hold8(l + g * 8);
    }
#pragma unroll
    for (int i = 0; i < T; ++i) acc[i] = __uint_as_float(h[i]) + (lo != 0 ? __uint_as_float(l[i]) : 0.f);
  }
  __device__ __forceinline__ void operator()(int which, int t0, int n, float (&acc)[kRedTok]) const {
    static_assert(kRedTok == 8, "one 8-column tensor-memory load per call");
    const int d = t0 - n0;
    const uint32_t a = taddr + (uint32_t)(d + (d / bn) * lo + which * up);
    tmem_ld8(a, acc);
    if (lo != 0) {
      float w[8];
      tmem_ld8(a + (uint32_t)lo, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += w[i];
    }
  }
  __device__ __forceinline__ void pair(int t0, int n, float (&a0)[kRedTok], float (&a1)[kRedTok]) const {
    (*this)(0, t0, n, a0);
    (*this)(1, t0, n, a1);
  }
};

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* a) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// Arrival on a counter that publishes the CTA's earlier writes: the caller
// first meets the other epilogue threads on a CTA barrier, then one thread
// performs the release (cheaper than a sequentially consistent fence per warp).
__device__ __forceinline__ void red_release_add(unsigned int* a, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_acq_rel_add(unsigned int* a, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// Row scales 1/sqrt(mean square + eps) of tokens [t_lo, t_lo + n) into sc[0..n)
// (1 when the token operand is not normalised); run by the 128 epilogue threads.
__device__ void row_scales(const EpiArgs& p, int r, int t_lo, int n, float* sc) {
  const float inv_dim = 1.0f / (float)(p.nkb * kTileK);
  const int half = p.M >> 1;   // fuse_ctx: block rows in [0, half), context rows in [half, M)
  for (int i = r; i < n; i += 128) {
    const int t = t_lo + i;
    const float* src = p.ss_in;
    int ld = p.ss_ld, row = t;
    bool valid = t < p.M;
    if (p.fuse_ctx) {
      if (t < half) {
        valid = t < p.m_blk;
      } else {
        src = p.ss_ctx;
        ld = p.ss_ctx_ld;
        row = t - half;
        valid = row < p.m_ctx;
      }
    }
    float v = 1.0f;
    if (src != nullptr && valid) {
      float ss = 0.f;
      for (int q0 = 0; q0 < p.n_ss; q0 += 8) {   // 8 unconditional loads in flight, summed in tile order
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __ldcg(src + (size_t)min(q0 + j, p.n_ss - 1) * ld + row);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += q0 + j < p.n_ss ? x[j] : 0.f;
      }
      v = 1.0f / sqrtf(ss * inv_dim + p.eps);
    }
    sc[i] = v;
  }
  epi_bar();
}

// Bounded wait until *cnt >= expected (the other CTAs of the tile arrived).
__device__ bool wait_count(const unsigned int* cnt, unsigned int expected, const uint32_t* gflags) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(cnt) >= expected) return true;
    __nanosleep(64);
    if ((it & 63u) == 63u) {
      uint32_t fl;
      uint64_t limit;
      ld_flags_limit(gflags, &fl, &limit);
      if (fl & DFLASH_FLAG_WAIT_TIMEOUT) return false;
      if (globaltimer_ns() - t0 > limit) return false;
    }
  }
}

// Bounded wait of the whole epilogue group (threads 0..127) on one phase: thread
// 0 waits, the result is shared through `flag`, and on success every thread
// re-checks the (completed) phase for its own acquire.  The answer is uniform,
// so the group's named barriers never split.
__device__ __forceinline__ bool group_wait(int r, uint64_t* bar, uint32_t parity, volatile int* abort,
                                           const uint32_t* gflags, volatile int* flag) {
  if (r == 0) *flag = mbar_wait(bar, parity, abort, gflags) ? 1 : 0;
  epi_bar();
  const bool okw = *flag != 0;
  epi_bar();   // everyone has read the flag before it can be rewritten
  if (okw) (void)mbar_wait(bar, parity, nullptr);
  return okw;
}

// ---------------------------------------------------------------- epilogues
// Run by the 128 epilogue threads of a CTA on its slice of a tile's tokens;
// thread r owns tile row r (output column gcol = seg_col0[seg] + row0 + r).

// Per token t = c0 + i (i < cn <= kEpiChunk) of a QKV or context-K/V tile: its
// RoPE position and destination row (q row, or KV arena row; -1: padding row
// of an append, or over capacity), looked up in parallel by threads i < cn.
// Reads only the sequence state, so it may run before the tile's sums exist.
__device__ __forceinline__ void rope_kv_stage(const EpiArgs& p, int r, int seg, int row0, int c0, int cn, bool ctx,
                                              int* tpos, long long* tdst) {
  if (r >= cn) return;
  const int head = row0 / kTileRows;
  const bool is_q = !ctx && seg == 0;
  const bool is_v = ctx ? (seg & 1) : (seg == 2);
  const int layer = ctx ? (seg >> 1) : p.layer;
  const int t = c0 + r;
  int b = 0, pos = 0, slot = 0;
  bool valid = true, is_q_row = is_q;
  // a fused append's context rows (token tile 1) take the context-row path
  const bool ctx_row = ctx || (p.fuse_ctx && t >= (p.M >> 1));
  if (ctx_row) {
    const int flat = ctx ? p.t0 + t : t - (p.M >> 1);
    const int fl = min(flat, p.m_ctx > 0 ? p.m_ctx - 1 : flat);
    b = fl / p.rows_max;
    const int rr = fl % p.rows_max;
    valid = rr < p.rows[b] && (ctx || flat < p.m_ctx);   // else a padding row of the append
    slot = p.st.pend_base[b] + rr;                       // the append is committed before its K/V
    pos = slot;
    if (is_q) {   // context rows have no query
      valid = false;
      is_q_row = false;
    }
  } else {
    if (p.fuse_ctx) valid = t < p.m_blk;   // padding of the block tile
    const int tb = valid ? t : 0;
    b = tb / p.R;
    const int j = tb % p.R;
    pos = p.st.ctx_len[b] + j;
    slot = block_base(p.st, b) + j;
    if (!is_q && j >= p.st.rblk[b]) valid = false;   // beyond this sequence's K_b + 1 block rows: no K/V
  }
  long long dst = -1;
  if (is_q_row) {
    if (valid) dst = t;
  } else if (valid) {
    const int cap = p.st.cap[b];
    if (slot < cap)
      dst = kv_row(p.kv, p.st.kv_base[b], cap, layer, is_v ? 1 : 0, head, slot);
    else
      set_flag(p.flags, DFLASH_FLAG_CAPACITY);
  }
  tpos[r] = pos;
  tdst[r] = dst;
}

// QKV (segments q, k, v) or context K/V (segments (W_k^l, W_v^l) = (2l, 2l+1)):
// rotate-half RoPE on q and k (pairs r, r + 64 of the head, exchanged through
// shared memory), then q to q_out and k, v to their KV slots.  staged: 0 --
// tpos / tdst hold kEpiChunk entries, filled here chunk by chunk; 1 -- the
// same, rope_kv_stage already filled them for the first chunk (tokens n0 ..)
// and the group has met since; 2 -- they hold every token of [n0, t_hi) at
// index t - n0, all staged before (no per-chunk lookups of the sequence state).
template <class Red>
__device__ void epi_rope_kv(const EpiArgs& p, const Red& red, int r, int seg, int row0, int n0, int t_hi, float* sm,
                            const float* sc, bool ctx, int* tpos, long long* tdst, int staged, int bar = 1) {
  const int head = row0 / kTileRows;
  const bool is_q = !ctx && seg == 0;
  const bool is_v = ctx ? (seg & 1) : (seg == 2);
  __nv_bfloat16* arena = reinterpret_cast<__nv_bfloat16*>(p.kv.base);
  const int pi = r & 63;
  const uint64_t f = p.rope_turns[pi];
  for (int c0 = n0; c0 < t_hi; c0 += kEpiChunk) {
    const int cn = min(kEpiChunk, t_hi - c0);
    if (staged == 0 || (staged == 1 && c0 != n0)) rope_kv_stage(p, r, seg, row0, c0, cn, ctx, tpos, tdst);
    const int* cpos = staged == 2 ? tpos + (c0 - n0) : tpos;
    const long long* cdst = staged == 2 ? tdst + (c0 - n0) : tdst;
    if constexpr (Red::kTmem) {   // the chunk's sums in one batch of tensor-memory loads
      float acc[kEpiChunk];
      red.template chunk<kEpiChunk>(0, c0, cn, acc);
#pragma unroll
      for (int i = 0; i < kEpiChunk; ++i)
        if (i < cn) sm[i * kEpiLd + r] = acc[i] * sc[c0 + i - n0];
    } else {
      for (int i0 = 0; i0 < cn; i0 += kRedTok) {
        float acc[kRedTok];
        red(0, c0 + i0, min(kRedTok, cn - i0), acc);
#pragma unroll
        for (int i = 0; i < kRedTok; ++i)
          if (i0 + i < cn) sm[(i0 + i) * kEpiLd + r] = acc[i] * sc[c0 + i0 + i - n0];
      }
    }
    epi_bar(bar);
    if constexpr (Red::kTmem) {
      // four tokens at a time with no early exit: their RoPE angles are
      // independent chains the scheduler can overlap (one warp per scheduler here)
      for (int i = 0; i < cn; i += 4) {
        float y[4];
        long long dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ii = min(i + u, cn - 1);
          dst[u] = i + u < cn ? cdst[ii] : -1;
          y[u] = sm[ii * kEpiLd + r];
          if (!is_v) {
            float c, s;
            rope_cs_fast(cpos[ii], f, &c, &s);
            const float x1 = sm[ii * kEpiLd + pi], x2 = sm[ii * kEpiLd + pi + 64];
            y[u] = r < 64 ? x1 * c - x2 * s : x2 * c + x1 * s;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (dst[u] < 0) continue;
          if (is_q)
            p.q_out[(size_t)dst[u] * p.seg_rows[0] + head * kTileRows + r] = __float2bfloat16_rn(y[u]);
          else
            arena[dst[u] * kTileRows + r] = __float2bfloat16_rn(y[u]);
        }
      }
    } else {
      for (int i = 0; i < cn; ++i) {
        const long long dst = cdst[i];
        if (dst < 0) continue;
        float y = sm[i * kEpiLd + r];
        if (!is_v) {
          float c, s;
          rope_cs_fast(cpos[i], f, &c, &s);
          const float x1 = sm[i * kEpiLd + pi], x2 = sm[i * kEpiLd + pi + 64];
          y = r < 64 ? x1 * c - x2 * s : x2 * c + x1 * s;
        }
        if (is_q)
          p.q_out[(size_t)dst * p.seg_rows[0] + head * kTileRows + r] = __float2bfloat16_rn(y);
        else
          arena[dst * kTileRows + r] = __float2bfloat16_rn(y);
      }
    }
    epi_bar(bar);
  }
}

// EPI_RESID (h += y) and EPI_Y_SS (v = y), then the tile's sum of squares per
// token (warp butterflies, then the four warps in order: deterministic) and,
// for the RMSNorm that follows, v * gain in bf16.
template <class Red>
__device__ void epi_resid(const EpiArgs& p, const Red& red, int r, int tile, int seg, int row0, int n0, int t_hi,
                          float* sm, bool add, int bar = 1) {
  static_assert(kRedTok == 8 && kEpiChunk % kRedTok == 0, "groups of 8 tokens (warp_sum8)");
  // tensor-memory sums (a whole tile per CTA): a 32-token chunk at a time, its
  // residual loads and accumulator loads all in flight together, the squares
  // summed 8 tokens per warp_sum8; partials in memory (a few tokens per CTA):
  // 8 tokens at a time
  const int warp = r >> 5, lane = r & 31;
  const int gcol = p.seg_col0[seg] + row0 + r;
  const float gain = p.xn_out != nullptr ? __bfloat162float(p.xn_gain[gcol]) : 0.f;
  const int slot = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);   // warp_sum8's slot
  if constexpr (Red::kTmem) {
    for (int c0 = n0; c0 < t_hi; c0 += kEpiChunk) {
      const int cn = min(kEpiChunk, t_hi - c0);
      bool bad = false;      // an fp16 operand out of range in this chunk
      float hv[kEpiChunk];   // the chunk's residual rows, every load in flight at once
      if (add) {
#pragma unroll
        for (int i = 0; i < kEpiChunk; ++i) hv[i] = i < cn ? __ldcg(p.h + (size_t)(c0 + i) * p.N + gcol) : 0.f;
      }
      float acc[kEpiChunk];   // the chunk's sums in one batch of tensor-memory loads
      red.template chunk<kEpiChunk>(0, c0, cn, acc);
#pragma unroll
      for (int g = 0; g < kEpiChunk / kRedTok; ++g) {
        const int i0 = g * kRedTok;
        if (i0 >= cn) break;
        const int n = min(kRedTok, cn - i0);
        float sq[kRedTok];
#pragma unroll
        for (int i = 0; i < kRedTok; ++i) {
          const int t = c0 + i0 + i;
          const float v = add ? acc[i0 + i] + hv[i0 + i] : acc[i0 + i];
          if (i < n) {
            if (p.h != nullptr) p.h[(size_t)t * p.N + gcol] = v;
            if (p.xn_out != nullptr)
              put_op_acc(v * gain, p.xn_out + (size_t)t * p.N + gcol, p.op16 ? kF16Plane : (size_t)p.M * p.N, bad);
          }
          sq[i] = v * v;   // slots past n are summed but never stored
        }
        const float ss = warp_sum8(sq, lane);
        if ((lane & 3) == 0 && slot < n) sm[warp * kEpiChunk + i0 + slot] = ss;
      }
      if (bad) set_flag(p.flags, DFLASH_FLAG_F16_RANGE);
      epi_bar(bar);
      if (r < cn) {
        const float ss = sm[r] + sm[kEpiChunk + r] + sm[2 * kEpiChunk + r] + sm[3 * kEpiChunk + r];
        p.ss_out[(size_t)tile * p.M + c0 + r] = ss;
      }
      epi_bar(bar);
    }
  } else {
    for (int c0 = n0; c0 < t_hi; c0 += kEpiChunk) {
      const int cn = min(kEpiChunk, t_hi - c0);
      bool bad = false;
      for (int i0 = 0; i0 < cn; i0 += kRedTok) {
        const int n = min(kRedTok, cn - i0);
        float acc[kRedTok], hv[kRedTok];
        if (add) {
#pragma unroll
          for (int i = 0; i < kRedTok; ++i) hv[i] = __ldcg(p.h + (size_t)(c0 + i0 + min(i, n - 1)) * p.N + gcol);
        }
        red(0, c0 + i0, n, acc);
#pragma unroll
        for (int i = 0; i < kRedTok; ++i) {
          if (i >= n) break;
          const int t = c0 + i0 + i;
          const float v = add ? acc[i] + hv[i] : acc[i];
          if (p.h != nullptr) p.h[(size_t)t * p.N + gcol] = v;
          if (p.xn_out != nullptr)
            put_op_acc(v * gain, p.xn_out + (size_t)t * p.N + gcol, p.op16 ? kF16Plane : (size_t)p.M * p.N, bad);
          const float sq = warp_sum(v * v);
          if (lane == 0) sm[warp * kEpiChunk + i0 + i] = sq;
        }
      }
      if (bad) set_flag(p.flags, DFLASH_FLAG_F16_RANGE);
      epi_bar(bar);
      if (r < cn) {
        const float ss = sm[r] + sm[kEpiChunk + r] + sm[2 * kEpiChunk + r] + sm[3 * kEpiChunk + r];
        p.ss_out[(size_t)tile * p.M + c0 + r] = ss;
      }
      epi_bar(bar);
    }
  }
}

// Maxima of 16 packed keys over the 32 lanes at once (k[j] of every lane ->
// slot j): lane l returns the maximum of slot 8 b4 + 4 b3 + 2 b2 + b1 (b_k = bit
// k of l), in 16 shuffles of 64 bits instead of 16 x 5.  A maximum is exact, so
// the result equals any other reduction order.
__device__ __forceinline__ unsigned long long warp_max16_u64(const unsigned long long (&k)[16], int lane) {
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0, b1 = (lane & 2) != 0;
  unsigned long long a[8], c[4], d[2];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const unsigned long long keep = b4 ? k[8 + i] : k[i], send = b4 ? k[i] : k[8 + i];
    a[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned long long keep = b3 ? a[4 + i] : a[i], send = b3 ? a[i] : a[4 + i];
    c[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const unsigned long long keep = b2 ? c[2 + i] : c[i], send = b2 ? c[i] : c[2 + i];
    d[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  unsigned long long e = max(b1 ? d[1] : d[0], __shfl_xor_sync(0xffffffffu, b1 ? d[0] : d[1], 2));
  return max(e, __shfl_xor_sync(0xffffffffu, e, 1));
}

// Draft index of token t (mask row j = t % R of sequence t / R: (t / R) (R - 1)
// + j - 1), or -1 for an anchor row, of tokens n0 + i (i < n) into kx[i]; run
// by the 128 threads of one epilogue group while the weights stream.
__device__ __forceinline__ void argmax_stage(const EpiArgs& p, int r, int n0, int n, int* kx) {
  for (int i = r; i < n; i += 128) {
    const int t = n0 + i;
    const int jb = p.R > 0 ? t % p.R : 1;
    kx[i] = jb == 0 ? -1 : p.R > 0 ? (t / p.R) * (p.R - 1) + jb - 1 : t;
  }
}

// EPI_ARGMAX from tensor memory, tokens [lo, hi) of a CTA whose tokens start at
// n0 (NT of them): per 16 tokens, each thread's packed (logit, id) keys of its
// vocabulary row, the maximum over the warp's 32 rows (warp_max16_u64), the
// four lane quadrants' maxima in wkeys[quadrant][token]; after the group meets,
// one atomicMax per token into one of kKeySlots slots (anchor rows skipped).
// Optional fp32 logits of the mask rows.  sc: row scales and kx: draft indices
// (argmax_stage), both from token n0.
__device__ void epi_argmax(const EpiArgs& p, const TmemRed& red, int r, int gcol, bool rvalid, int n0, int NT, int lo,
                           int hi, const float* sc, const int* kx, unsigned long long* wkeys, int tile, int bar) {
  const int quad = r >> 5, lane = r & 31;
  const int slot = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
  // the 16 columns of the next chunk are loaded while this one is reduced
  // (the wait at the top of a step covers only the chunk issued before it);
  // two named buffers, alternating, so that every index is static
  uint32_t h0[16], l0[16], h1[16], l1[16];
  auto issue = [&](int t0, uint32_t (&h)[16], uint32_t (&l)[16]) {
    const int n = min(16, hi - t0);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      if (g * 8 < n) {   // warp-uniform
        const int d = t0 - n0 + g * 8;
        const uint32_t a = red.taddr + (uint32_t)(d + (d / red.bn) * red.lo);
        tmem_ld8_issue(a, h + g * 8);
        if (red.lo != 0) tmem_ld8_issue(a + (uint32_t)red.lo, l + g * 8);
      }
    }
  };
  auto step = [&](int t0, uint32_t (&h)[16], uint32_t (&l)[16], uint32_t (&hn)[16], uint32_t (&ln)[16]) {
    const int n = min(16, hi - t0);
    tmem_wait_ld_all();
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      tmem_hold8(h + g * 8);
      tmem_hold8(l + g * 8);
    }
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(h[i]) + (red.lo != 0 ? __uint_as_float(l[i]) : 0.f);
    if (t0 + 16 < hi) issue(t0 + 16, hn, ln);
    unsigned long long k[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int ti = min(t0 + i, hi - 1) - n0;
      const int kidx = kx[ti];
      const bool live = rvalid && i < n && kidx >= 0;
      const float z = v[i] * sc[ti];
      if (live && p.logits != nullptr) p.logits[(size_t)kidx * p.N + gcol] = z;
      k[i] = live ? argmax_key(z, (uint32_t)gcol) : 0ull;
    }
    const unsigned long long kk = warp_max16_u64(k, lane);
    if ((lane & 1) == 0 && slot < n) wkeys[quad * NT + (t0 - n0) + slot] = kk;
  };
#pragma unroll
  for (int i = 0; i < 16; ++i) h0[i] = l0[i] = h1[i] = l1[i] = 0u;
  if (lo < hi) issue(lo, h0, l0);
  for (int t0 = lo; t0 < hi; t0 += 32) {
    step(t0, h0, l0, h1, l1);
    if (t0 + 16 < hi) step(t0 + 16, h1, l1, h0, l0);
  }
  epi_bar(bar);
  for (int t = lo + r; t < hi; t += 128) {
    const int kidx = kx[t - n0];
    if (kidx < 0) continue;
    unsigned long long key = wkeys[t - n0];
#pragma unroll
    for (int w = 1; w < 4; ++w) key = max(key, wkeys[w * NT + t - n0]);
    atomicMax(p.argmax_keys + ((size_t)kidx * kKeySlots + (tile % kKeySlots)) * kKeyStride, key);
  }
}

// EPI_SILU: gate tile `pair` and up tile pair + half_tiles -> a = silu(gate) * up
template <class Red>
__device__ void epi_silu(const EpiArgs& p, const Red& red, int r, int pair, int n0, int t_hi, const float* sc) {
  const int I = p.seg_rows[0];
  const int f = pair * kTileRows + r;
  bool bad = false;   // an fp16 operand out of range, latched once at the end
  if constexpr (Red::kTmem) {   // gate and up sums of 16 tokens in one batch of loads
    for (int t0 = n0; t0 < t_hi; t0 += 16) {
      const int n = min(16, t_hi - t0);
      float g[16], u[16];
      red.template chunk<16>(0, t0, n, g);
      red.template chunk<16>(1, t0, n, u);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i >= n) break;
        const float gs = g[i] * sc[t0 + i - n0], us = u[i] * sc[t0 + i - n0];
        put_op_acc(__fdividef(gs, 1.0f + __expf(-gs)) * us, p.a_out + (size_t)(t0 + i) * I + f,
                   p.op16 ? kF16Plane : (size_t)p.M * I, bad);
      }
    }
  } else {
    for (int t0 = n0; t0 < t_hi; t0 += kRedTok) {
      const int n = min(kRedTok, t_hi - t0);
      float g[kRedTok], u[kRedTok];
      red.pair(t0, n, g, u);
#pragma unroll
      for (int i = 0; i < kRedTok; ++i) {
        if (i >= n) break;
        const float gs = g[i] * sc[t0 + i - n0], us = u[i] * sc[t0 + i - n0];
        put_op_acc(__fdividef(gs, 1.0f + __expf(-gs)) * us, p.a_out + (size_t)(t0 + i) * I + f,
                   p.op16 ? kF16Plane : (size_t)p.M * I, bad);
      }
    }
  }
  if (bad) set_flag(p.flags, DFLASH_FLAG_F16_RANGE);
}

}  // namespace
}  // namespace dfl
