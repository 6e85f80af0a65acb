// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05, sm_103a),
// with the drafter's normalisations and epilogues folded in.
//
//   Y[t][n] = sum_k X[t][k] * W[n][k]      (W: weights [N, K], X: tokens [M, K], bf16)
//
// At drafting time M = batch * (K+1) is small, so every projection is bound by
// streaming W from HBM.  The weights sit on the MMA's M side ("swap AB"): one
// CTA owns a 128-row weight tile and a K range; a producer warp streams
// 128 x 64 weight boxes and the matching BN x 64 token boxes with TMA into a
// ring of shared-memory stages (128-byte swizzle) -- the first weight boxes
// before waiting for the previous kernel, since weights never depend on it.
// One thread issues tcgen05.mma (M=128, N=BN, K=16) into a TMEM accumulator;
// the four epilogue warps read it back with tcgen05.ld and store fp32 partial
// sums [split][t][n].  The CTAs of a tile then meet on a counter, and each
// sums the partials of its own slice of tokens in split order -- so results do
// not depend on scheduling -- and applies the epilogue: RoPE and KV-slot
// writes, residual add, SwiGLU on gate/up tile pairs, or the greedy argmax of
// the LM head.
//
// RMSNorm is folded into the GEMMs on either side of it.  A residual epilogue
// leaves, next to the fp32 rows, the per-tile sums of squares and the rows
// times the next norm's gain in bf16 -- the next GEMM's token operand; that
// GEMM multiplies its reduced outputs by each row's 1/sqrt(mean square + eps).
// RMSNorm(h) W^T = diag(1/rms(h)) (h * g) W^T, so this is the same product
// with the row scale applied after the sum instead of before it.
//
// Roles (192 threads): warps 0-3 epilogue (TMEM lanes 32w..32w+31), warp 4 TMA
// producer, warp 5 TMEM owner and MMA issuer; the single-split (direct)
// instances have 320: eight epilogue warps, then the producer and the MMA issuer.
#include <algorithm>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dfl {

namespace {

// tokens of a CTA whose RoPE positions and KV destinations a direct epilogue
// stages before its accumulator is ready (TT * BN <= 256)
constexpr int kStageTok = 256;

__host__ __device__ __forceinline__ uint32_t tmem_cols_for(int BN) {
  return BN <= 32 ? 32u : (BN <= 64 ? 64u : (BN <= 128 ? 128u : (BN <= 256 ? 256u : 512u)));
}

// TT token tiles of BN per CTA (1, or 2 for wide split operands); the one-tile
// instance is the common drafting case and fits two CTAs per SM.  DIRECT: the
// tiles have one split and the epilogue reads the accumulator in place (its own
// instances, so that the split-K instances carry none of that code).  E: the
// epilogue (a GemmEpi) compiled in, or -1 for the one in the parameters; the
// split-K one-tile instance, on every drafting step's critical path, has one
// instance per epilogue so that each carries only its own code.
template <int TT, bool DIRECT, int E>
__global__ void __launch_bounds__(DIRECT ? 320 : 192, TT == 1 && !DIRECT ? 2 : 1)
    gemm_tc_kernel(const __grid_constant__ TcGemmParams p) {
  constexpr int EW = DIRECT ? 8 : 4;   // epilogue warps; warp EW: TMA producer, EW + 1: MMA issuer
  const int epi = E >= 0 ? E : p.epi;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  const int S = p.stages, BN = p.BN;
  const uint32_t w_box = kTileRows * kTileK * 2;                        // one weight box: 16 KB
  const int W = DIRECT && p.wpair ? 2 : 1;                              // weight boxes per stage
  const uint32_t a_bytes = w_box * (uint32_t)W;
  const int XP = p.x_planes;                                            // token planes (1, or 2: hi + lo)
  const int NT = TT * BN;                                               // tokens per CTA
  const uint32_t box_bytes = (uint32_t)BN * kTileK * 2;                 // one bf16 token box
  const uint32_t tb_bytes = box_bytes * (uint32_t)XP;                   // one token tile's B operand
  const uint32_t b_bytes = tb_bytes * (uint32_t)TT;                     // all token tiles of a stage
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)S * a_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)S * b_bytes);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* wait_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
  float* row_sc = reinterpret_cast<float*>(tmem_slot + 4);   // [NT] row scales of the folded RMSNorm
  long long* tdst = reinterpret_cast<long long*>(row_sc + 256);   // [kStageTok] RoPE/KV destinations
  int* tpos = reinterpret_cast<int*>(tdst + kStageTok);            // [kStageTok] RoPE positions

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!p.late_trigger) pdl_trigger();   // (else after the dependency wait)

  // weight tile -> segment
  // grid (token tiles, weight tiles, splits): the token tiles of one weight tile
  // are adjacent in launch order, so they run together and share its boxes in L2
  const int tile = blockIdx.y;
  int seg = 0, row0;
  if (W == 2) {   // gate rows 128 * tile.. (segment 0) and the same up rows (segment 1)
    row0 = tile * kTileRows;
  } else if (p.interleave2) {
    seg = tile & 1;
    row0 = (tile >> 1) * kTileRows;
  } else {
    while (seg + 1 < p.nseg && tile >= p.seg_tile0[seg + 1]) ++seg;
    row0 = (tile - p.seg_tile0[seg]) * kTileRows;
  }
  const int split = blockIdx.z;
  const int kb0 = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.nkb - kb0);
  const int n0 = blockIdx.x * NT;
  const uint32_t ncols = tmem_cols_for(TT * XP * BN * W);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == EW + 1) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  int issued = 0;   // producer: k-blocks whose loads were issued
  if (warp == EW) {
    if (lane == 0) {
      // Weights do not depend on the previous kernel: stream the first S
      // weight boxes before waiting for it (their barriers only expect the
      // bytes; the arrival comes with the token box after the wait).
      const int pre = min(S, nkb);
      const uint64_t pol = l2_evict_first_policy();   // weights are read once
      tma_prefetch_desc(&p.tm_w[seg]);
      if (W == 2) tma_prefetch_desc(&p.tm_w[1]);
      for (int kb = 0; kb < pre; ++kb) {
        mbar_expect_tx(&full[kb], a_bytes);
        for (int w = 0; w < W; ++w)
          tma_load_2d_hint(sA + (size_t)kb * a_bytes + w * w_box, &p.tm_w[seg + w], (kb0 + kb) * kTileK, row0,
                           &full[kb], pol);
      }
      issued = pre;
      pdl_wait_release(p.late_trigger);
      tma_prefetch_desc(&p.tm_x);
      if (TT == 2 && p.fuse_ctx) tma_prefetch_desc(&p.tm_x2);
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % S;
        const int kc = (kb0 + kb) * kTileK;
        if (kb >= pre) {
          const uint32_t ph = (uint32_t)(kb / S) & 1u;
          if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.flags)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], a_bytes + b_bytes);
          for (int w = 0; w < W; ++w)
            tma_load_2d_hint(sA + (size_t)st * a_bytes + w * w_box, &p.tm_w[seg + w], kc, row0, &full[st], pol);
          issued = kb + 1;
        } else {
          mbar_arrive_expect_tx(&full[st], b_bytes);
        }
        for (int i = 0; i < TT; ++i) {
          // a fused append's context rows are token tile 1, from their own map
          const bool ctx_tile = TT == 2 && i == 1 && p.fuse_ctx;
          for (int pl = 0; pl < XP; ++pl)
            tma_load_3d(sB + (size_t)st * b_bytes + (size_t)(i * XP + pl) * box_bytes, ctx_tile ? &p.tm_x2 : &p.tm_x,
                        kc, ctx_tile ? 0 : n0 + i * BN, pl, &full[st]);
        }
      }
    } else {
      pdl_wait_release(p.late_trigger);
    }
  } else if (warp == EW + 1) {
    pdl_wait_release(p.late_trigger);
    if (lane == 0) {
      // fp16 token operands go with the fp16 weight copies (A and B of one type)
      const uint32_t idesc = p.op16 ? umma_idesc_f16(kTileRows, XP * BN) : umma_idesc_bf16(kTileRows, XP * BN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int st = kb % S;
        const uint32_t ph = (uint32_t)(kb / S) & 1u;
        if (!mbar_wait(&full[st], ph, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int w = 0; w < W; ++w) {   // each weight box of the stage (gate, up of a pair)
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + (size_t)st * a_bytes + w * w_box));
          for (int i = 0; i < TT; ++i) {   // against each token tile
            const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + (size_t)st * b_bytes + (size_t)i * tb_bytes));
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k) {
              // advance 16 bf16 = 32 bytes along K inside the swizzled row: +2 in 16-byte units
              umma_bf16(tmem + (uint32_t)((w * TT + i) * XP * BN), ad + 2u * k, bd + 2u * k, idesc,
                        (kb | k) != 0 ? 1u : 0u);
            }
          }
        }
        umma_commit(&empty[st]);  // frees the stage once these MMAs have read it
      }
      umma_commit(accum);         // accumulator complete (tracks every MMA issued above)
    }
  } else if constexpr (DIRECT) {
    // One split: the sums are this CTA's accumulator, read in place.  Eight
    // epilogue warps, two per tensor-memory lane quadrant (warp w reads lanes
    // 32 (w % 4) ..): half h = w / 4 finishes its own contiguous run of whole
    // token chunks, on its own named barrier and scratch.
    pdl_wait_release(p.late_trigger);
    const int half = warp >> 2;
    const int r = threadIdx.x & 127;   // tile row = tensor-memory lane
    const int t_end = min(n0 + NT, p.M);
    if (half == 0) {
      // while the weights stream: the folded-norm row scales and every token's
      // RoPE position and destination (<= kStageTok tokens, 128 per pass)
      if (n0 < t_end) {
        if (epi == EPI_QKV || epi == EPI_CTXKV)
          for (int c = n0; c < t_end; c += 128)
            rope_kv_stage(p, r, seg, row0, c, min(128, t_end - c), epi == EPI_CTXKV, tpos + (c - n0), tdst + (c - n0));
        if (epi == EPI_ARGMAX) argmax_stage(p, r, n0, t_end - n0, tpos);   // draft index per token
        if (epi == EPI_QKV || epi == EPI_CTXKV || epi == EPI_SILU || epi == EPI_ARGMAX)
          row_scales(p, r, n0, t_end - n0, row_sc);
        epi_bar();
      }
      if (ok && !group_wait(r, accum, 0u, abort_flag, p.flags, wait_flag)) ok = false;
    }
    epi_pair_bar();   // both halves: staging done, accumulator verdict in *wait_flag
    if (half == 1) {
      ok = ok && *wait_flag != 0;
      if (ok) (void)mbar_wait(accum, 0u, nullptr);
    }
    if (ok) {
      tc_fence_after();
      const int nch = (t_end - n0 + kEpiChunk - 1) / kEpiChunk;
      const int mid = min(t_end, n0 + kEpiChunk * ((nch + 1) / 2));
      const int lo = half ? mid : n0, hi = half ? t_end : mid;
      float* sm = reinterpret_cast<float*>(sA) + half * kEpiChunk * kEpiLd;   // the stage ring is idle now
      const TmemRed red{tmem + ((uint32_t)((warp & 3) * 32) << 16), n0, BN, XP == 2 ? BN : 0, XP * BN};
      const int bar = 1 + half;
      const int off = lo - n0;
      if (lo < hi) {
        switch (epi) {
          case EPI_QKV:
            epi_rope_kv(p, red, r, seg, row0, lo, hi, sm, row_sc + off, false, tpos + off, tdst + off, 2, bar);
            break;
          case EPI_CTXKV:
            epi_rope_kv(p, red, r, seg, row0, lo, hi, sm, row_sc + off, true, tpos + off, tdst + off, 2, bar);
            break;
          case EPI_RESID: epi_resid(p, red, r, tile, seg, row0, lo, hi, sm, true, bar); break;
          case EPI_Y_SS: epi_resid(p, red, r, tile, seg, row0, lo, hi, sm, false, bar); break;
          case EPI_SILU: epi_silu(p, red, r, tile, lo, hi, row_sc + off); break;
          case EPI_ARGMAX:   // keys in the idle stage ring, [quadrant][NT]
            epi_argmax(p, red, r, p.seg_col0[seg] + row0 + r, row0 + r < p.seg_rows[seg], n0, NT, lo, hi, row_sc,
                       tpos, reinterpret_cast<unsigned long long*>(sA), tile, bar);
            break;
          default: break;
        }
      }
    }
    if (epi == EPI_ARGMAX) {
      // every key of the CTA is in its slots: the last CTA to finish turns the
      // slots into draft ids (half 0)
      epi_pair_bar();
      if (half == 0) {
        if (r == 0) {
          const unsigned int prev = atom_acq_rel_add(p.counters, 1u);
          const int last = prev == gridDim.x * gridDim.y * gridDim.z - 1;
          if (last) p.counters[0] = 0u;
          *last_flag = ok && last;
        }
        epi_bar();
        if (*last_flag) {
          const int nk = p.R > 0 ? (p.M / p.R) * (p.R - 1) : p.M;
          for (int k = r; k < nk; k += 128) {
            unsigned long long* a = p.argmax_keys + (size_t)k * kKeySlots * kKeyStride;
            unsigned long long v[kKeySlots];   // every slot's load in flight at once
#pragma unroll
            for (int sl = 0; sl < kKeySlots; ++sl) v[sl] = __ldcg(a + (size_t)sl * kKeyStride);
            unsigned long long key = 0ull;
#pragma unroll
            for (int sl = 0; sl < kKeySlots; ++sl) {
              key = max(key, v[sl]);
              a[(size_t)sl * kKeyStride] = 0ull;   // every CTA has arrived: no atomic can still target it
            }
            p.ids[k] = (int32_t)argmax_key_index(key);
          }
        }
      }
    }
  } else {
    pdl_wait_release(p.late_trigger);
    const int tid = threadIdx.x;   // 0..127
    // While the weights stream: everything of the epilogue that does not depend
    // on this tile's sums -- the folded-norm row scales and the RoPE positions
    // and KV destinations of the tokens this CTA finishes -- so that only the
    // split-K reduction itself is left after the last CTA of the tile arrives.
    if (epi == EPI_ARGMAX) {
      row_scales(p, tid, n0, NT, row_sc);
    } else if (epi != EPI_PARTIAL) {
      const int members = (epi == EPI_SILU ? 2 : 1) * p.splits;
      const int member = (epi == EPI_SILU ? (tile & 1) * p.splits : 0) + split;
      const int t_end = min(n0 + NT, p.M);
      const int per = (t_end - n0 + members - 1) / members;
      const int lo = min(t_end, n0 + member * per), hi = min(t_end, lo + per);
      if (lo < hi) {
        if (epi == EPI_QKV || epi == EPI_CTXKV)
          rope_kv_stage(p, tid, seg, row0, lo, min(kEpiChunk, hi - lo), epi == EPI_CTXKV, tpos, tdst);
        if (epi == EPI_QKV || epi == EPI_CTXKV || epi == EPI_SILU) row_scales(p, tid, lo, hi - lo, row_sc);
        epi_bar();
      }
    }
    // epilogue: warp w reads TMEM lanes 32w..32w+31 = weight rows row0+32w..
    if (ok && !group_wait(tid, accum, 0u, abort_flag, p.flags, wait_flag)) ok = false;
    if (ok) {
      tc_fence_after();
      const int grow = row0 + warp * 32 + lane;
      const bool rvalid = grow < p.seg_rows[seg];
      const int gcol = p.seg_col0[seg] + grow;
      const bool argmax = epi == EPI_ARGMAX;
      float* out = p.ws + (size_t)split * p.M * p.N;
      unsigned long long* wkeys = reinterpret_cast<unsigned long long*>(sA);   // [4][NT], ring idle now
      for (int i = 0; i < TT; ++i) {      // token tile i: columns i * XP * BN .., tokens n0 + i * BN ..
        const uint32_t col0 = (uint32_t)(i * XP * BN);
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + col0 + (uint32_t)c, v);
          if (XP == 2) {   // token t's product = hi-plane column t + lo-plane column BN + t
            float w2[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + col0 + (uint32_t)(BN + c), w2);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += w2[j];
          }
          const int tc = i * BN + c;   // token of v[0] within the CTA
          if (!argmax) {
            if (rvalid) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {   // columns past BN belong to the lo plane
                const int t = n0 + tc + j;
                if (c + j < BN && t < p.M) out[(size_t)t * p.N + gcol] = v[j];
              }
            }
          } else {
            // greedy argmax over this warp's 32 vocabulary rows: packed (logit, lowest id) keys;
            // token t = b*R + j, anchor rows (j = 0) carry no draft
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c + j >= BN) break;
              const int t = n0 + tc + j;
              const float z = v[j] * row_sc[tc + j];
              const int jb = p.R > 0 ? t % p.R : 1;
              const int kidx = p.R > 0 ? (t / p.R) * (p.R - 1) + jb - 1 : t;
              if (rvalid && p.logits != nullptr && t < p.M && jb != 0) p.logits[(size_t)kidx * p.N + gcol] = z;
              unsigned long long key = rvalid ? argmax_key(z, (uint32_t)gcol) : 0ull;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
                key = other > key ? other : key;
              }
              if (lane == 0) wkeys[warp * NT + tc + j] = key;
            }
          }
        }
      }
      if (argmax) {
        // one atomic per token and CTA, into one of kKeySlots slots per token
        // (each on its own 128-byte line) so that few CTAs share a line
        epi_bar();
        for (int i = tid; i < NT; i += 128) {
          const int t = n0 + i;
          const int jb = p.R > 0 ? t % p.R : 1;
          if (t >= p.M || jb == 0) continue;
          const int kidx = p.R > 0 ? (t / p.R) * (p.R - 1) + jb - 1 : t;
          unsigned long long key = wkeys[i];
#pragma unroll
          for (int w = 1; w < 4; ++w) key = max(key, wkeys[w * NT + i]);
          atomicMax(p.argmax_keys + ((size_t)kidx * kKeySlots + (tile % kKeySlots)) * kKeyStride, key);
        }
      }
      if (epi != EPI_PARTIAL) {
        epi_bar();   // every epilogue thread's partial sums (or keys) are written
        float* sm = reinterpret_cast<float*>(sA);   // the stage ring is idle now
        if (argmax) {
          // the last CTA to finish turns the keys into draft ids
          if (tid == 0) {
            const unsigned int prev = atom_acq_rel_add(p.counters, 1u);
            const int last = prev == gridDim.x * gridDim.y * gridDim.z - 1;
            if (last) p.counters[0] = 0u;
            *last_flag = last;
          }
          epi_bar();
          if (*last_flag) {
            const int nk = p.R > 0 ? (p.M / p.R) * (p.R - 1) : p.M;
            for (int k = tid; k < nk; k += 128) {
              unsigned long long key = 0ull;
              for (int sl = 0; sl < kKeySlots; ++sl) {
                unsigned long long* a = p.argmax_keys + ((size_t)k * kKeySlots + sl) * kKeyStride;
                key = max(key, __ldcg(a));
                *a = 0ull;   // every CTA has arrived: no atomic can still target it
              }
              p.ids[k] = (int32_t)argmax_key_index(key);
            }
          }
        } else {
          // all CTAs of the tile (or gate/up pair) meet, then each finishes a slice of tokens
          const bool pair = epi == EPI_SILU;
          const int unit = pair ? tile >> 1 : tile;
          const unsigned int idx = (unsigned)(unit * gridDim.x + blockIdx.x);
          const int expected = (pair ? 2 : 1) * p.splits;
          const int member = (pair ? (tile & 1) * p.splits : 0) + split;
          if (tid == 0) {
            red_release_add(p.counters + 2 * idx, 1u);
            *last_flag = wait_count(p.counters + 2 * idx, (unsigned)expected, p.flags) ? 1 : 0;
          }
          epi_bar();
          if (!*last_flag) {
            ok = false;
          } else {
            const int t_end = min(n0 + NT, p.M);
            const int per = (t_end - n0 + expected - 1) / expected;
            const int lo = min(t_end, n0 + member * per), hi = min(t_end, lo + per);
            if (lo < hi) {   // row scales and the first chunk's RoPE table were staged above
              const int gcol = p.seg_col0[seg] + row0 + tid;
              const GlobalRed red{&p, {pair ? unit * kTileRows + tid : gcol, pair ? p.seg_rows[0] + unit * kTileRows + tid : gcol}};
              switch (epi) {
                case EPI_QKV: epi_rope_kv(p, red, tid, seg, row0, lo, hi, sm, row_sc, false, tpos, tdst, 1); break;
                case EPI_CTXKV: epi_rope_kv(p, red, tid, seg, row0, lo, hi, sm, row_sc, true, tpos, tdst, 1); break;
                case EPI_RESID: epi_resid(p, red, tid, tile, seg, row0, lo, hi, sm, true); break;
                case EPI_Y_SS: epi_resid(p, red, tid, tile, seg, row0, lo, hi, sm, false); break;
                case EPI_SILU: epi_silu(p, red, tid, unit, lo, hi, row_sc); break;
                default: break;
              }
            }
            epi_bar();
            if (tid == 0) {
              const unsigned int prev = atomicAdd(p.counters + 2 * idx + 1, 1u);
              if (prev == (unsigned)expected - 1) {   // every member is done: reset for the next launch
                p.counters[2 * idx] = 0u;
                p.counters[2 * idx + 1] = 0u;
              }
            }
          }
        }
      }
    }
  }

  if (!ok) {
    *abort_flag = 1;
    set_flag(p.flags, DFLASH_FLAG_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted && warp == EW && lane == 0) {
    // let every load still in flight land before the CTA's shared memory goes away
    for (int kb = max(0, issued - S); kb < issued; ++kb) {
      (void)mbar_wait(&full[kb % S], (uint32_t)(kb / S) & 1u, nullptr);
    }
  }
  if (warp == EW + 1) {
    if (aborted && lane == 0) (void)mbar_wait(accum, 0u, nullptr);  // MMAs done before TMEM is freed
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// Persistent direct GEMM for grids of more tiles than SMs (large M, plain fp16
// token operands, one token tile per CTA and one split): one CTA per SM walks
// the tiles blockIdx.x, blockIdx.x + gridDim.x, ... (token tiles of a weight
// tile adjacent, so concurrent CTAs share its boxes in L2).  The producer runs
// the stage ring on across tiles, the MMA issuer alternates between two TMEM
// accumulators, and the eight epilogue warps finish tile j from one of them
// while tile j + 1 accumulates in the other -- the epilogue, 40-50% of a
// one-tile CTA's time at the serving batch, runs under the next mainloop.  The
// epilogue scratch has its own shared memory (the ring is never idle here).
__global__ void __launch_bounds__(320, 1) gemm_tc_persist_kernel(const __grid_constant__ TcGemmParams p) {
  constexpr int EW = 8;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  const int S = p.stages, BN = p.BN;
  const uint32_t w_box = kTileRows * kTileK * 2;
  const int W = p.wpair ? 2 : 1;
  const uint32_t a_bytes = w_box * (uint32_t)W;
  const uint32_t b_bytes = (uint32_t)BN * kTileK * 2;   // one fp16 token box
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)S * a_bytes;
  float* epi_sm = reinterpret_cast<float*>(sB + (size_t)S * b_bytes);   // [2 halves][kEpiChunk][kEpiLd]
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_sm + 2 * kEpiChunk * kEpiLd);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;    // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wait_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
  float* row_sc = reinterpret_cast<float*>(tmem_slot + 4);
  long long* tdst = reinterpret_cast<long long*>(row_sc + 256);
  int* tpos = reinterpret_cast<int*>(tdst + kStageTok);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!p.late_trigger) pdl_trigger();   // (else after the dependency wait)
  const int T = p.p_tiles, TX = p.p_ttiles;   // tiles, token tiles per weight tile
  const uint32_t ncols = tmem_cols_for(BN * W);   // one accumulator
  auto decode = [&](int tau, int& tile, int& seg, int& row0, int& n0) {
    tile = tau / TX;
    n0 = (tau % TX) * BN;
    seg = 0;
    if (W == 2) {
      row0 = tile * kTileRows;
    } else {
      while (seg + 1 < p.nseg && tile >= p.seg_tile0[seg + 1]) ++seg;
      row0 = (tile - p.seg_tile0[seg]) * kTileRows;
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == EW + 1) {
    tmem_alloc(tmem_slot, 2 * ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  int issued = 0;   // producer: k-blocks whose loads were issued (over all tiles)
  if (warp == EW) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int pre = 0;
      if ((int)blockIdx.x < T) {   // the first tile's first weight boxes before the dependency
        int tile, seg, row0, n0;
        decode(blockIdx.x, tile, seg, row0, n0);
        pre = min(S, p.nkb);
        tma_prefetch_desc(&p.tm_w[seg]);
        if (W == 2) tma_prefetch_desc(&p.tm_w[1]);
        for (int kb = 0; kb < pre; ++kb) {
          mbar_expect_tx(&full[kb], a_bytes);
          for (int w = 0; w < W; ++w)
            tma_load_2d_hint(sA + (size_t)kb * a_bytes + w * w_box, &p.tm_w[seg + w], kb * kTileK, row0, &full[kb],
                             pol);
        }
      }
      pdl_wait_release(p.late_trigger);
      tma_prefetch_desc(&p.tm_x);
      int g = 0;
      for (int tau = blockIdx.x; tau < T && ok; tau += gridDim.x) {
        int tile, seg, row0, n0;
        decode(tau, tile, seg, row0, n0);
        for (int kb = 0; kb < p.nkb; ++kb, ++g) {
          const int st = g % S;
          const int kc = kb * kTileK;
          if (g >= pre) {
            if (!mbar_wait(&empty[st], (uint32_t)((g / S) & 1) ^ 1u, abort_flag, p.flags)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[st], a_bytes + b_bytes);
            for (int w = 0; w < W; ++w)
              tma_load_2d_hint(sA + (size_t)st * a_bytes + w * w_box, &p.tm_w[seg + w], kc, row0, &full[st], pol);
          } else {
            mbar_arrive_expect_tx(&full[st], b_bytes);
          }
          tma_load_3d(sB + (size_t)st * b_bytes, &p.tm_x, kc, n0, 0, &full[st]);
          issued = g + 1;
        }
      }
    } else {
      pdl_wait_release(p.late_trigger);
    }
  } else if (warp == EW + 1) {
    pdl_wait_release(p.late_trigger);
    if (lane == 0) {
      const uint32_t idesc = p.op16 ? umma_idesc_f16(kTileRows, BN) : umma_idesc_bf16(kTileRows, BN);
      int g = 0, j = 0;
      for (int tau = blockIdx.x; tau < T && ok; tau += gridDim.x, ++j) {
        const int a = j & 1;
        // the epilogue of tile j - 2 has read this accumulator
        if (!mbar_wait(&acc_empty[a], (uint32_t)((j >> 1) & 1) ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.nkb; ++kb, ++g) {
          const int st = g % S;
          if (!mbar_wait(&full[st], (uint32_t)((g / S) & 1), abort_flag, p.flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + (size_t)st * b_bytes));
          for (int w = 0; w < W; ++w) {
            const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + (size_t)st * a_bytes + w * w_box));
#pragma unroll
            for (int k = 0; k < kTileK / 16; ++k)
              umma_bf16(tmem + (uint32_t)a * ncols + (uint32_t)(w * BN), ad + 2u * k, bd + 2u * k, idesc,
                        (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[st]);
        }
        if (!ok) break;
        umma_commit(&acc_full[a]);
      }
      umma_commit(mma_done);
    }
  } else {
    // eight epilogue warps, two per tensor-memory lane quadrant, as in the
    // one-tile direct instance; between tiles both halves meet, then the
    // accumulator is handed back to the MMA issuer
    pdl_wait_release(p.late_trigger);
    const int half = warp >> 2;
    const int r = threadIdx.x & 127;
    int j = 0;
    for (int tau = blockIdx.x; tau < T && ok; tau += gridDim.x, ++j) {
      int tile, seg, row0, n0;
      decode(tau, tile, seg, row0, n0);
      const int a = j & 1;
      const uint32_t par = (uint32_t)((j >> 1) & 1);
      const int t_end = min(n0 + BN, p.M);
      if (half == 0) {
        if (n0 < t_end) {
          if (p.epi == EPI_QKV || p.epi == EPI_CTXKV)
            for (int c = n0; c < t_end; c += 128)
              rope_kv_stage(p, r, seg, row0, c, min(128, t_end - c), p.epi == EPI_CTXKV, tpos + (c - n0),
                            tdst + (c - n0));
          if (p.epi == EPI_QKV || p.epi == EPI_CTXKV || p.epi == EPI_SILU) row_scales(p, r, n0, t_end - n0, row_sc);
          epi_bar();
        }
        if (!group_wait(r, &acc_full[a], par, abort_flag, p.flags, wait_flag)) ok = false;
      }
      epi_pair_bar();   // staging done, accumulator verdict in *wait_flag
      if (half == 1) {
        ok = *wait_flag != 0;
        if (ok) (void)mbar_wait(&acc_full[a], par, nullptr);
      }
      if (ok) {
        tc_fence_after();
        const int nch = (t_end - n0 + kEpiChunk - 1) / kEpiChunk;
        const int mid = min(t_end, n0 + kEpiChunk * ((nch + 1) / 2));
        const int lo = half ? mid : n0, hi = half ? t_end : mid;
        float* sm = epi_sm + half * kEpiChunk * kEpiLd;
        const TmemRed red{tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)a * ncols, n0, BN, 0, BN};
        const int bar = 1 + half;
        const int off = lo - n0;
        if (lo < hi) {
          switch (p.epi) {
            case EPI_QKV:
              epi_rope_kv(p, red, r, seg, row0, lo, hi, sm, row_sc + off, false, tpos + off, tdst + off, 2, bar);
              break;
            case EPI_CTXKV:
              epi_rope_kv(p, red, r, seg, row0, lo, hi, sm, row_sc + off, true, tpos + off, tdst + off, 2, bar);
              break;
            case EPI_RESID: epi_resid(p, red, r, tile, seg, row0, lo, hi, sm, true, bar); break;
            case EPI_Y_SS: epi_resid(p, red, r, tile, seg, row0, lo, hi, sm, false, bar); break;
            case EPI_SILU: epi_silu(p, red, r, tile, lo, hi, row_sc + off); break;
            default: break;
          }
        }
      }
      // both halves are done with this accumulator and the staged tables
      tc_fence_before();
      epi_pair_bar();
      ok = ok && *wait_flag != 0;
      if (threadIdx.x == 0) mbar_arrive(&acc_empty[a]);
    }
  }

  if (!ok) {
    *abort_flag = 1;
    set_flag(p.flags, DFLASH_FLAG_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == EW && lane == 0) {
    for (int g = max(0, issued - S); g < issued; ++g) (void)mbar_wait(&full[g % S], (uint32_t)((g / S) & 1), nullptr);
  }
  if (warp == EW + 1) {
    if (lane == 0) (void)mbar_wait(mma_done, 0u, nullptr);   // every MMA done before TMEM is freed
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * ncols);
  }
}

}  // namespace

size_t gemm_tc_smem_bytes(int BN, int stages, int x_planes, int tt, int w_boxes) {
  const size_t per_stage = (size_t)w_boxes * kTileRows * kTileK * 2 + (size_t)tt * x_planes * BN * kTileK * 2;
  return 1024 + (size_t)stages * per_stage + (size_t)(2 * stages + 1) * 8 + 16 + 256 * sizeof(float) +
         kStageTok * (sizeof(long long) + sizeof(int));
}

// CTAs of gemm_tc_kernel resident per SM with `smem` bytes of dynamic shared
// memory (raises the kernel's shared-memory limit first); 0 on error.
using GemmKernelFn = void (*)(TcGemmParams);
constexpr int kEpiKinds = 7;   // GemmEpi values
// instance index: 0 tt 1 split-K with its epilogue compiled in (epi 0..6),
// 7 tt 1 split-K any epilogue, 8 tt 2 split-K, 9 tt 1 direct, 10 tt 2 direct
constexpr int kGemmInstances = kEpiKinds + 4;
static int gemm_tc_index(int tt, bool direct, int epi) {
  if (direct) return tt == 2 ? kEpiKinds + 3 : kEpiKinds + 2;
  if (tt == 2) return kEpiKinds + 1;
  return epi >= 0 && epi < kEpiKinds ? epi : kEpiKinds;
}
static GemmKernelFn gemm_tc_instance(int idx) {
  switch (idx) {
    case EPI_PARTIAL: return gemm_tc_kernel<1, false, EPI_PARTIAL>;
    case EPI_ARGMAX: return gemm_tc_kernel<1, false, EPI_ARGMAX>;
    case EPI_QKV: return gemm_tc_kernel<1, false, EPI_QKV>;
    case EPI_RESID: return gemm_tc_kernel<1, false, EPI_RESID>;
    case EPI_SILU: return gemm_tc_kernel<1, false, EPI_SILU>;
    case EPI_Y_SS: return gemm_tc_kernel<1, false, EPI_Y_SS>;
    case EPI_CTXKV: return gemm_tc_kernel<1, false, EPI_CTXKV>;
    case kEpiKinds: return gemm_tc_kernel<1, false, -1>;
    case kEpiKinds + 1: return gemm_tc_kernel<2, false, -1>;
    case kEpiKinds + 2: return gemm_tc_kernel<1, true, -1>;
    default: return gemm_tc_kernel<2, true, -1>;
  }
}
static cudaError_t gemm_tc_allow_smem(int idx, size_t smem) {
  static size_t allowed[kGemmInstances] = {};
  if (smem <= allowed[idx]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(gemm_tc_instance(idx), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) allowed[idx] = smem;
  return e;
}

// CTAs of gemm_tc_kernel<tt> resident per SM with `smem` bytes of dynamic
// shared memory, from the kernel's registers and the SM's register file,
// shared memory and thread limits (the occupancy API assumes a default
// shared-memory carveout and reports fewer) and from tensor memory: a CTA
// holds tmem_cols_for(n_cols) of the SM's 512 columns for its whole life, and
// one that cannot allocate them waits for another to exit, which a split-K
// partner never does before it; 0 when one CTA does not fit.
int gemm_tc_resident_ctas(int tt, bool direct, size_t smem, int n_cols, int epi) {
  static cudaFuncAttributes fa_all[kGemmInstances];
  static cudaDeviceProp prop;
  static bool have[kGemmInstances] = {}, have_prop = false;
  const int idx = gemm_tc_index(tt, direct, epi);
  if (gemm_tc_allow_smem(idx, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const cudaFuncAttributes* fa = &fa_all[idx];
  if (!have[idx]) {
    if (cudaFuncGetAttributes(&fa_all[idx], gemm_tc_instance(idx)) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    have[idx] = true;
  }
  if (!have_prop) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    have_prop = true;
  }
  const int threads = direct ? 320 : 192;
  const int warps = threads / 32;
  const int regs_warp = (fa->numRegs * 32 + 255) / 256 * 256;   // allocated per warp in units of 256
  const int by_regs = prop.regsPerMultiprocessor / (regs_warp * warps);
  const size_t per_cta = smem + fa->sharedSizeBytes + prop.reservedSharedMemPerBlock;
  const int by_smem = (int)(prop.sharedMemPerMultiprocessor / per_cta);
  const int by_threads = prop.maxThreadsPerMultiProcessor / threads;
  const int by_tmem = 512 / (int)tmem_cols_for(n_cols);
  return std::max(0, std::min({by_regs, by_smem, by_threads, by_tmem, prop.maxBlocksPerMultiProcessor}));
}

size_t gemm_tc_persist_smem_bytes(int BN, int stages, int w_boxes) {
  const size_t per_stage = (size_t)w_boxes * kTileRows * kTileK * 2 + (size_t)BN * kTileK * 2;
  return 1024 + (size_t)stages * per_stage + 2 * kEpiChunk * kEpiLd * sizeof(float) + (size_t)(2 * stages + 5) * 8 +
         16 + 256 * sizeof(float) + kStageTok * (sizeof(long long) + sizeof(int));
}

cudaError_t launch_gemm_tc_persist(const TcGemmParams& p, int grid, cudaStream_t s) {
  static size_t allowed = 0;
  const size_t smem = gemm_tc_persist_smem_bytes(p.BN, p.stages, p.wpair ? 2 : 1);
  if (smem > allowed) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_tc_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    allowed = smem;
  }
  const cudaError_t e = launch_k(gemm_tc_persist_kernel, dim3(grid), dim3(320), smem, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gemm_tc(const TcGemmParams& p, int n_tiles, int splits, int t_tiles, int stages,
                           cudaStream_t s, bool by_epi) {
  const size_t smem = gemm_tc_smem_bytes(p.BN, stages, p.x_planes, p.tt, p.wpair ? 2 : 1);
  const int tt = p.tt == 2 ? 2 : 1;
  const bool direct = p.direct != 0;
  const int idx = gemm_tc_index(tt, direct, by_epi ? p.epi : -1);
  cudaError_t e = gemm_tc_allow_smem(idx, smem);
  if (e != cudaSuccess) return e;
  e = launch_k(gemm_tc_instance(idx), dim3(t_tiles, n_tiles, splits), dim3(direct ? 320 : 192), smem, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dfl
