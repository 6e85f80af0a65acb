// Block-bidirectional GQA attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), bf16, head_dim 128.
//
// [GDB §用于注意力机制的“双缓存”方案]: block attention is non-causal, so no mask
// applies -- every query row of a KV head (G query heads x R block rows)
// attends to all kv_len_b context slots and all R block slots of its sequence.
//
// One CTA = (KV split, KV head x query tile, sequence).  A query tile is 128
// rows: JT = 128 / G consecutive block rows j times the G query heads of the KV
// head, row r = jj * G + g, loaded by one 3-D TMA box per half of head_dim.
//   warp 8   producer: the query tile once, then 64-position K and V tiles of
//            the KV arena into a 3-stage ring (two 64 x 64 boxes per operand,
//            128-byte swizzle)
//   warp 9   TMEM owner and MMA issuer: S = Q K^T (M = 128 rows, N = 64
//            positions, K = 128) into one of two TMEM score buffers, then
//            O += P V (N = 128 dims, K = 64 positions; V is read as an MN-major
//            operand straight from the TMA layout) into the TMEM output
//   warps 0-7 softmax, two threads per query row (TMEM lane = row; warps w and
//            w + 4 share the lane quarter w, each takes one half of a tile's 64
//            positions and of the 128 output dimensions): scores to registers,
//            the row maximum of the tile from both halves (exchanged in shared
//            memory), log2-domain softmax against a reference maximum that is
//            only raised when a row's maximum grows by more than kRescale (then
//            the row of O is rescaled in TMEM), P as split bf16 (hi + lo planes,
//            two MMAs, ~16 significant bits) into shared memory, and at the end
//            O / l out -- the final output (one split) or the split's normalised
//            partial and log2-sum-exp for the merge kernel.
// Softmax, the score buffers and the P buffers are double-buffered, so the
// scores of tile t+1 are computed while the softmax of tile t runs.
#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {

constexpr int kUTile = 64;                            // KV positions per tile
constexpr int kUStages = 3;
constexpr uint32_t kUBox = 64 * 128;                  // 64 rows x 64 bf16 (one swizzle span)
constexpr uint32_t kUStage = 4 * kUBox;               // K[0:64], K[64:128], V[0:64], V[64:128]
constexpr uint32_t kUQHalf = 128 * 128;               // [128 rows][64 dims] bf16
constexpr uint32_t kUPPlane = 128 * 128;              // [128 rows][64 positions] bf16
constexpr float kRescale = 8.0f;                      // log2 headroom of P before O is rescaled
constexpr uint32_t kUTmemCols = 256;                  // S[2] (2 x 64) + O (128)

// 32 lanes x 32 bits, 16 consecutive columns written from the thread's row.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits, 32 consecutive columns into the thread's registers; the
// caller waits (tmem_wait_ld) once for a batch of these before using them.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Shared-memory descriptor of an MN-major operand written by TMA with the
// 128-byte swizzle: rows of 64 MN elements (128 B) along K, 8-row K groups
// `sbo` bytes apart, 64-element MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// kind::f16 instruction descriptor with a K-major A and an MN-major B.
__host__ __device__ constexpr uint32_t umma_idesc_bf16_bmn(int M, int N) {
  return umma_idesc_bf16(M, N) | (1u << 16);
}

// One row (64 bf16 = 8 chunks of 16 B) of a K-major, 128-byte-swizzled tile
// whose base is 1024-B aligned: chunk c of row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ void st_swizzled_row(uint8_t* tile, int r, const uint32_t (&w)[32]) {
  uint8_t* row = tile + (size_t)r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Half a row: chunks c0 .. c0 + 3 (32 bf16) of row r of such a tile.
__device__ __forceinline__ void st_swizzled_half(uint8_t* tile, int r, int c0, const uint32_t (&w)[16]) {
  uint8_t* row = tile + (size_t)r * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(row + (((c0 + c) ^ (r & 7)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// The two softmax warps of TMEM lane quarter q (w and w + 4) meet on named
// barrier 1 + q; the _and form also returns whether v held in all 64 threads,
// so that both warps leave the tile loop on the same tile and meet the same
// number of times on every path.
__device__ __forceinline__ void quarter_bar(int q) { asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory"); }
__device__ __forceinline__ bool quarter_bar_and(int q, bool v) {
  uint32_t all;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, 64, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(all)
      : "r"((uint32_t)v), "r"(1 + q)
      : "memory");
  return all != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace

namespace {

// Bounded wait of one warp on a barrier phase: lane 0 waits, the answer is
// shared, and on success every lane observes the completed phase itself.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const uint32_t* flags) {
  int okv = 1;
  if ((threadIdx.x & 31) == 0) okv = mbar_wait(bar, parity, abort, flags) ? 1 : 0;
  okv = __shfl_sync(0xffffffffu, okv, 0);
  if (okv) (void)mbar_wait(bar, parity, nullptr);
  return okv != 0;
}

constexpr int kUThreads = 320;   // 8 softmax warps, the producer, the MMA issuer

__global__ void __launch_bounds__(kUThreads, 1) attn_umma_kernel(const __grid_constant__ AttnUParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem;                                   // 2 x [128 rows][64 dims]
  uint8_t* ring = sQ + 2 * kUQHalf;                     // kUStages x (K lo, K hi, V lo, V hi)
  uint8_t* sP = ring + kUStages * kUStage;              // [2 buffers][hi, lo][128 rows][64 positions]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 4 * kUPPlane);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + kUStages;
  uint64_t* s_full = bars + 1 + 2 * kUStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_free = p_full + 2;
  uint64_t* o_done = p_free + 2;     // one phase per PV (the softmax rescales after PV t-1)
  uint64_t* o_final = o_done + 1;    // the last PV
  uint64_t* mma_done = o_final + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the two halves' tile maxima [tile parity][half][row] and row sums [half][row]
  float* xmax = reinterpret_cast<float*>(tmem_slot + 4);
  float* xsum = xmax + 2 * 2 * 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kUStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 8);
      mbar_init(&p_full[i], 8);
      mbar_init(&p_free[i], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kUTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the successor may launch only once every CTA holds its tensor memory: a
  // successor CTA that took this SM's columns first would wait for this grid
  // while this CTA waited in its allocation
  pdl_trigger();
  pdl_wait();   // the queries and the KV arena come from the predecessors

  const int split = blockIdx.x;
  const int hk = blockIdx.y % p.n_kv, qt = blockIdx.y / p.n_kv;
  const int b = p.seq_order != nullptr ? p.seq_order[blockIdx.z] : blockIdx.z;
  const int cap = p.st.cap[b];
  int L = block_base(p.st, b) + p.st.rblk[b];   // context + this sequence's K_b + 1 block rows
  if (L > cap) {
    if (threadIdx.x == 0 && split == 0 && hk == 0 && qt == 0) set_flag(p.flags, DFLASH_FLAG_CAPACITY);
    L = cap;
  }
  // balanced split of [0, L) into n_splits ranges of whole tiles (live length)
  const int chunk = ((L + p.n_splits - 1) / p.n_splits + kUTile - 1) / kUTile * kUTile;
  const int p_begin = split * chunk;
  const int p_end = min(L, p_begin + chunk);
  const int ntiles = p_end > p_begin ? (p_end - p_begin + kUTile - 1) / kUTile : 0;
  const int64_t base = p.st.kv_base[b];
  const int rowK = (int)kv_row(p.kv, base, cap, p.layer, 0, hk, 0);
  const int rowV = (int)kv_row(p.kv, base, cap, p.layer, 1, hk, 0);

  bool ok = true;
  int issued = 0;
  bool q_issued = false;
  if (warp == 8) {
    // ------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_kv);
      mbar_arrive_expect_tx(q_full, 2 * kUQHalf);
      const int tok = b * p.R + qt * p.JT;
      tma_load_3d(sQ, &p.tm_q, 0, hk * p.G, tok, q_full);
      tma_load_3d(sQ + kUQHalf, &p.tm_q, 64, hk * p.G, tok, q_full);
      q_issued = true;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kUStages;
        if (!mbar_wait(&kv_empty[st], (uint32_t)((t / kUStages) & 1) ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], kUStage);
        const int pos = p_begin + t * kUTile;
        uint8_t* dst = ring + (size_t)st * kUStage;
        tma_load_2d(dst, &p.tm_kv, 0, rowK + pos, &kv_full[st]);
        tma_load_2d(dst + kUBox, &p.tm_kv, 64, rowK + pos, &kv_full[st]);
        tma_load_2d(dst + 2 * kUBox, &p.tm_kv, 0, rowV + pos, &kv_full[st]);
        tma_load_2d(dst + 3 * kUBox, &p.tm_kv, 64, rowV + pos, &kv_full[st]);
        issued = t + 1;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      const uint32_t idesc_s = umma_idesc_bf16(128, kUTile);
      const uint32_t idesc_o = umma_idesc_bf16_bmn(128, 128);
      const uint64_t qa[2] = {sw128_kmajor_desc(smem_u32(sQ)), sw128_kmajor_desc(smem_u32(sQ + kUQHalf))};
      // O += P(u) V(u): P hi and lo planes (K-major, 64 positions), V MN-major
      // (rows = positions, 128 B of dims; the two 64-dim halves 8 KB apart)
      auto pv = [&](int u) -> bool {
        const int pb = u & 1, st = u % kUStages;
        if (!mbar_wait(&p_full[pb], (uint32_t)((u >> 1) & 1), abort_flag, p.flags)) return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(ring + (size_t)st * kUStage + 2 * kUBox);
#pragma unroll
        for (int pl = 0; pl < 2; ++pl) {
          const uint64_t pa = sw128_kmajor_desc(smem_u32(sP + (size_t)(pb * 2 + pl) * kUPPlane));
#pragma unroll
          for (int k = 0; k < kUTile / 16; ++k)   // 16 positions = two 8-row groups = 2048 B of V
            umma_bf16(tmem + 128u, pa + 2u * k, sw128_mnmajor_desc(vb + 2048u * k, kUBox, 1024u), idesc_o,
                      (u | pl | k) != 0 ? 1u : 0u);
        }
        umma_commit(&kv_empty[st]);
        umma_commit(&p_free[pb]);
        umma_commit(o_done);
        return true;
      };
      if (!mbar_wait(q_full, 0u, abort_flag, p.flags)) ok = false;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int st = t % kUStages, sb = t & 1;
        if (!mbar_wait(&kv_full[st], (uint32_t)((t / kUStages) & 1), abort_flag, p.flags) ||
            !mbar_wait(&s_free[sb], (uint32_t)((t >> 1) & 1) ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* kt = ring + (size_t)st * kUStage;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t kd = sw128_kmajor_desc(smem_u32(kt + h * kUBox));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem + (uint32_t)(sb * kUTile), qa[h] + 2u * k, kd + 2u * k, idesc_s, (h | k) != 0 ? 1u : 0u);
        }
        umma_commit(&s_full[sb]);
        if (t > 0 && !pv(t - 1)) ok = false;
      }
      if (ok && !pv(ntiles - 1)) ok = false;
      if (ok) umma_commit(o_final);
    }
    if (lane == 0) umma_commit(mma_done);   // tracks every MMA issued above
  } else {
    // ------------------------------------------------ softmax, two threads per query row
    const int r = threadIdx.x & 127;                    // TMEM lane = tile row
    const int hf = threadIdx.x >> 7;                    // half: positions 32 hf .. of a tile, dims 64 hf ..
    const int qq = warp & 3;                            // TMEM lane quarter
    const int gq = r % p.G, j = qt * p.JT + r / p.G;    // query head hk * G + gq, block row j
    const bool rvalid = j < p.R;
    const int row_lim = block_base(p.st, b) + j;   // causal: the row's own position
    const uint32_t lane_base = (uint32_t)(qq * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;   // l: this half's share of the row sum
    // a failed wait skips the rest of its tile; the pair leaves the loop
    // together at the next meeting
    for (int t = 0; t < ntiles; ++t) {
      const int sb = t & 1;
      float s[kUTile / 2];
      float hmax = -INFINITY;
      if (ok && warp_wait(&s_full[sb], (uint32_t)((t >> 1) & 1), abort_flag, p.flags)) {
        tc_fence_after();
        tmem_ld32_issue(tmem + lane_base + (uint32_t)(sb * kUTile + 32 * hf), s);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);
        // scale into the log2 domain; positions past the split (and, causal,
        // past the row's own position) are masked
        const int pos0 = p_begin + t * kUTile + 32 * hf;
        const int p_row = p.causal ? min(p_end, row_lim + 1) : p_end;
#pragma unroll
        for (int i = 0; i < kUTile / 2; ++i) {
          const float v = pos0 + i < p_row ? s[i] * p.scale_log2 : -INFINITY;
          s[i] = v;
          hmax = fmaxf(hmax, v);
        }
      } else {
        ok = false;
      }
      // the row's maximum over the whole tile: this half's and the partner's
      // (double-buffered by tile parity, so one meeting per tile suffices)
      xmax[(sb * 2 + hf) * 128 + r] = hmax;
      if (!quarter_bar_and(qq, ok)) {
        ok = false;
        break;
      }
      const float tmax = fmaxf(hmax, xmax[(sb * 2 + (hf ^ 1)) * 128 + r]);
      // reference maximum: set by the first tile (which always holds the
      // split's first position), raised only when a row outgrows it by more
      // than kRescale -- then O and l of that row are rescaled (both halves
      // take the same decision from the same maximum)
      float factor = 1.f;
      bool resc = false;
      if (t == 0) {
        m_ref = tmax;
      } else if (tmax > m_ref + kRescale) {
        factor = exp2f(m_ref - tmax);
        m_ref = tmax;
        resc = true;
      }
      if (__any_sync(0xffffffffu, resc)) {   // the warp rescales its half of its 32 rows of O (PV of tile t-1 done)
        // S(t) was committed after PV(t-2) and PV(t) waits for this tile's P, so
        // o_done is in phase t-1 or t: the parity wait is unambiguous
        if (!warp_wait(o_done, (uint32_t)((t - 1) & 1), abort_flag, p.flags)) {
          ok = false;
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 64 * hf; c < 64 * hf + 64; c += 16) {
          float o16[16];
          tmem_ld16(tmem + lane_base + 128u + (uint32_t)c, o16);
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] *= factor;
          tmem_st16(tmem + lane_base + 128u + (uint32_t)c, o16);
        }
        tmem_wait_st();
        l *= factor;
      }
      // P = 2^(s - m_ref) <= 2^kRescale as split bf16
      // (a causal row may see no position of this split: its scores are all
      // -inf, and so is m_ref; 0 as the reference makes P = 0, l = 0)
      const float mr = m_ref == -INFINITY ? 0.f : m_ref;
      uint32_t hi[kUTile / 4], lo[kUTile / 4];
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < kUTile / 4; ++i) {
        const float p0 = exp2f(s[2 * i] - mr), p1 = exp2f(s[2 * i + 1] - mr);
        ps += p0 + p1;
        const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
        hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lo[i] = pack_bf16x2(p0 - __bfloat162float(h0), p1 - __bfloat162float(h1));
      }
      l += ps;
      const int pb = t & 1;
      if (!warp_wait(&p_free[pb], (uint32_t)((t >> 1) & 1) ^ 1u, abort_flag, p.flags)) {
        ok = false;
        continue;
      }
      st_swizzled_half(sP + (size_t)(pb * 2) * kUPPlane, r, 4 * hf, hi);
      st_swizzled_half(sP + (size_t)(pb * 2 + 1) * kUPPlane, r, 4 * hf, lo);
      fence_proxy_async_smem();   // generic-proxy P writes -> the tensor core's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    // ------------------------------------------------ output: O / l
    // the row sum from both halves, in half order (both threads get the same
    // value); every softmax thread meets its partner here on every path
    xsum[hf * 128 + r] = l;
    quarter_bar(qq);
    const float lrow = xsum[r] + xsum[128 + r];
    if (ok) {
      const int qd = p.n_q * 128;
      const float inv = lrow > 0.f ? 1.0f / lrow : 0.f;
      const float lse = lrow > 0.f ? m_ref + log2f(lrow) : -INFINITY;
      // the last PV has its own barrier: by now o_done may be anywhere between
      // the last two phases, so a parity wait on it would be ambiguous
      const bool have = ntiles > 0 && warp_wait(o_final, 0u, abort_flag, p.flags);
      if (ntiles > 0 && !have) ok = false;
      if (ok) {
        tc_fence_after();
        const int rq = gq * p.R + j;   // row of the merge kernel's layout
        const size_t prow = (((size_t)(b * p.n_kv + hk) * p.n_splits + split) * p.rows_pad + rq);
        __nv_bfloat16* orow = p.o + (size_t)(b * p.R + j) * qd + (size_t)(hk * p.G + gq) * 128;
        {
          const int h = 64 * hf;   // this half's 64 output columns in one batch of TMEM loads
          float o64[64];
          if (have) {
            tmem_ld32_issue(tmem + lane_base + 128u + (uint32_t)h, o64);
            tmem_ld32_issue(tmem + lane_base + 128u + (uint32_t)(h + 32), o64 + 32);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) o64[i] = 0.f;
          }
          if (rvalid) {
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
              const float* o16 = o64 + cc;
              const int c = h + cc;
              if (p.n_splits == 1 && p.o_plane == kF16Plane) {   // one fp16 plane
                uint32_t wh[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  check_f16(o16[2 * i] * inv, p.flags);
                  check_f16(o16[2 * i + 1] * inv, p.flags);
                  const __half2 v = __floats2half2_rn(o16[2 * i] * inv, o16[2 * i + 1] * inv);
                  wh[i] = *reinterpret_cast<const uint32_t*>(&v);
                }
                uint4* dh = reinterpret_cast<uint4*>(orow + c);
                dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
              } else if (p.n_splits == 1) {   // split bf16: hi plane, lo plane o_plane further
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  __nv_bfloat16 h0, l0, h1, l1;
                  split_bf16(o16[2 * i] * inv, &h0, &l0);
                  split_bf16(o16[2 * i + 1] * inv, &h1, &l1);
                  wh[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                  wl[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                uint4* dh = reinterpret_cast<uint4*>(orow + c);
                uint4* dl = reinterpret_cast<uint4*>(orow + p.o_plane + c);
                dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
                dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
              } else {
                float4* po = reinterpret_cast<float4*>(p.part_o + prow * 128 + c);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  po[i] = make_float4(o16[4 * i] * inv, o16[4 * i + 1] * inv, o16[4 * i + 2] * inv,
                                      o16[4 * i + 3] * inv);
              }
            }
          }
        }
        if (rvalid && p.n_splits > 1 && hf == 0) p.part_lse[prow] = lse;
      }
    }
  }

  if (!ok) {
    *abort_flag = 1;
    set_flag(p.flags, DFLASH_FLAG_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 8 && lane == 0) {
    // let every load still in flight land before the shared memory goes away
    if (q_issued) (void)mbar_wait(q_full, 0u, nullptr);
    for (int t = max(0, issued - kUStages); t < issued; ++t)
      (void)mbar_wait(&kv_full[t % kUStages], (uint32_t)((t / kUStages) & 1), nullptr);
  }
  if (warp == 9) {
    if (lane == 0) (void)mbar_wait(mma_done, 0u, nullptr);   // MMAs done before TMEM is freed
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUTmemCols);
  }
}

}  // namespace

size_t attn_umma_smem_bytes() {
  return 1024 + 2 * kUQHalf + kUStages * kUStage + 4 * kUPPlane + (1 + 2 * kUStages + 8 + 3) * 8 + 16 +
         (2 * 2 * 128 + 2 * 128) * sizeof(float);
}

cudaError_t launch_attention_umma(const AttnUParams& p, int B, cudaStream_t s) {
  static bool configured = false;
  const size_t smem = attn_umma_smem_bytes();
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(attn_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  launch_k(attn_umma_kernel, dim3(p.n_splits, p.n_kv * p.n_qtiles, B), dim3(kUThreads), smem, s, p);
  return cudaGetLastError();
}

}  // namespace dfl
