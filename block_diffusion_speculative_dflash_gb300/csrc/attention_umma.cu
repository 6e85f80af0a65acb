// Block-bidirectional GQA attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), bf16, head_dim 128.
//
// [GDB §用于注意力机制的“双缓存”方案]: block attention is non-causal, so no mask
// applies -- every query row of a KV head (G query heads x R block rows)
// attends to all kv_len_b context slots and all R block slots of its sequence.
//
// A work item = (sequence, KV head x query tile, KV split).  A query tile is
// 128 rows: JT = 128 / G consecutive block rows j times the G query heads of
// the KV head, row r = jj * G + g, loaded by one 3-D TMA box per half of
// head_dim.  A batch's items come from a schedule planned on the device once
// per draft (splits per sequence from its live length, longest items first)
// and are taken by one persistent CTA per SM; a single sequence runs one item
// per CTA from the grid.  Roles:
//   warp 8   item fetch (persistent: from the launch's counter, published to
//            the other roles through a shared-memory slot ring), the query
//            tile of each item, and the K tiles (64 positions, two 64 x 64
//            boxes, 128-byte swizzle) into a 3-stage ring
//   warp 10  the V tiles into the same stages; K and V of a stage have
//            barriers of their own, so the next K may land as soon as S has
//            read the last one while PV still reads V
//   warp 9   TMEM owner and MMA issuer: S = Q K^T (M = 128 rows, N = 64
//            positions, K = 128) into one of two TMEM score buffers, then
//            O += P V (N = 128 dims, K = 64 positions; V is read as an MN-major
//            operand straight from the TMA layout) into one of two TMEM output
//            buffers (alternating by item, so that one item's output phase
//            overlaps the next item's MMAs)
//   warps 0-7 softmax, two threads per query row (TMEM lane = row; warps w and
//            w + 4 share the lane quarter w, each takes one half of a tile's 64
//            positions and of the 128 output dimensions): scores to registers,
//            the row maximum of the tile from both halves (exchanged in shared
//            memory), log2-domain softmax against a reference maximum that is
//            only raised when a row's maximum grows by more than kRescale (then
//            the row of O is rescaled in TMEM), P rounded to bf16 (the type of
//            the V operand it meets) into shared memory, and at the end O / l
//            out -- the final output (one split) or the split's normalised
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
constexpr uint32_t kUTmemCols = 512;                  // S[2] (2 x 64) + one O (128) per softmax part

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

// NW / 4 chunks of 16 bytes (c0 ..) of row r of a K-major, 128-byte-swizzled
// tile whose base is 1024-B aligned: chunk c of row r sits at chunk c ^ (r & 7).
template <int NW>
__device__ __forceinline__ void st_swizzled_part(uint8_t* tile, int r, int c0, const uint32_t (&w)[NW]) {
  uint8_t* row = tile + (size_t)r * 128;
#pragma unroll
  for (int c = 0; c < NW / 4; ++c)
    *reinterpret_cast<uint4*>(row + (((c0 + c) ^ (r & 7)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Threads per query row of the softmax: a row's tile of 64 positions and its
// 128 output dimensions are split between kParts warps of one TMEM lane quarter
// (warps w, w + 4, ..), which meet on named barrier 1 + q; the _and form also
// returns whether v held in all of them, so that they leave the tile loop on
// the same tile and meet the same number of times on every path.
constexpr int kParts = 2;
constexpr int kPCols = kUTile / kParts;    // score positions per thread
constexpr int kODims = 128 / kParts;       // output dimensions per thread
__device__ __forceinline__ void quarter_bar(int q) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + q), "n"(32 * kParts) : "memory");
}
__device__ __forceinline__ bool quarter_bar_and(int q, bool v) {
  uint32_t all;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(all)
      : "r"((uint32_t)v), "r"(1 + q), "n"(32 * kParts)
      : "memory");
  return all != 0;
}

// 2^x by the MUFU approximation (one instruction; results below 2^-126 flush to
// zero, far under the bf16 planes of P whose largest entry is ~1)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

constexpr int kSoftWarps = 4 * kParts;
// bf16 planes of P: 1 (round to nearest: 8 significant bits, like the bf16 V
// it multiplies) or 2 (hi + lo, ~16 bits, two PV MMAs)
constexpr int kPPlanes = 1;
constexpr int kWarpQK = kSoftWarps, kWarpMma = kSoftWarps + 1, kWarpV = kSoftWarps + 2;
constexpr int kUThreads = 32 * (kSoftWarps + 3);   // softmax warps, the query/K producer, the MMA issuer, the V producer
constexpr int kUSlots = 4;       // work items published ahead of the consumers
constexpr int kUItem = 10;       // ints per published item

// One work item: query tile qt of KV head hk of sequence b against the
// sequence's KV split `split` of S, positions [p_begin, p_end); partials of a
// sequence with S > 1 go to partial group pg + split (b < 0: no more items);
// rowK / rowV: the arena rows of the head's K and V at position 0.
struct UItem {
  int b, split, hk, qt, p_begin, p_end, S, pg, rowK, rowV;
  int base;   // first block row (every position below it holds context K/V written before this draft)
};

// Item w of the launch: from the grid (one item per CTA), or the w-th of the
// persistent schedule (units in the planned order, every head-tile of a unit
// consecutive); the split's range is the balanced share of the live length.
template <bool grid_mode>
__device__ __forceinline__ UItem decode_item(const AttnUParams& p, int w) {
  UItem x;
  const int n_hq = p.n_kv * p.n_qtiles;
  int hq;
  // (the sequence state through L2 only: grid mode may read it before the
  // dependency wait, when only its release, not a cache flush, orders it
  // after the kernels that wrote it)
  if constexpr (grid_mode) {
    x.b = p.seq_order != nullptr ? __ldcg(p.seq_order + blockIdx.z) : blockIdx.z;
    x.split = blockIdx.x;
    hq = blockIdx.y;
    x.S = p.n_splits;
    x.pg = x.b * x.S;
  } else {
    const int unit = p.work[w / n_hq];
    hq = w % n_hq;
    x.b = unit >> 8;
    x.split = unit & 255;
    x.S = p.seq_split[2 * x.b];
    x.pg = p.seq_split[2 * x.b + 1];
  }
  x.hk = hq % p.n_kv;
  x.qt = hq / p.n_kv;
  // every load of the sequence's state at once (one round trip)
  const int cap = __ldcg(p.st.cap + x.b);
  const long long kv_base = __ldcg(reinterpret_cast<const long long*>(p.st.kv_base) + x.b);
  x.base = p.st.ctx_kv ? __ldcg(p.st.kv_len + x.b) : 0;   // block_base
  int L = x.base + __ldcg(p.st.rblk + x.b);   // context + this sequence's K_b + 1 block rows
  x.rowK = (int)kv_row(p.kv, kv_base, cap, p.layer, 0, x.hk, 0);
  x.rowV = (int)kv_row(p.kv, kv_base, cap, p.layer, 1, x.hk, 0);
  if (L > cap) {
    if (x.split == 0 && hq == 0) set_flag(p.flags, DFLASH_FLAG_CAPACITY);
    L = cap;
  }
  // balanced split of [0, L) into S ranges of whole tiles (live length)
  const int chunk = ((L + x.S - 1) / x.S + kUTile - 1) / kUTile * kUTile;
  x.p_begin = x.split * chunk;
  x.p_end = min(L, x.p_begin + chunk);
  return x;
}
__device__ __forceinline__ int item_tiles(const UItem& x) {
  return x.p_end > x.p_begin ? (x.p_end - x.p_begin + kUTile - 1) / kUTile : 0;
}
// Leading K/V tiles of an item whose whole box lies below the block rows (at
// most one ring's worth): nothing the predecessor writes is in them.
__device__ __forceinline__ int early_tiles(const UItem& x) {
  const int below = (x.base - x.p_begin) / kUTile;
  return max(0, min(min(below, item_tiles(x)), kUStages));
}

// Persistent (p.work set): one CTA per SM takes items from the launch's
// counter until they run out, the producer running ahead into the next item's
// queries and K/V while the last tiles and the output of the current one are
// processed; two output accumulators in tensor memory let one item's output
// phase overlap the next item's MMAs.  Grid mode (p.work null): the grid
// (split, head x query tile, sequence) with one item per CTA.
// (Two instances, so that the one-item-per-CTA grid carries none of the
// persistent schedule's code: its CTAs start cold, and every instruction
// fetched on the way to the first loads is on the critical path.)
template <bool PERSIST>
__global__ void __launch_bounds__(kUThreads, 1) attn_umma_kernel(const __grid_constant__ AttnUParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sQ = smem;                                   // 2 x [128 rows][64 dims]
  uint8_t* ring = sQ + 2 * kUQHalf;                     // kUStages x (K lo, K hi, V lo, V hi)
  uint8_t* sP = ring + kUStages * kUStage;              // [2 buffers][kPPlanes][128 rows][64 positions]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * kPPlanes * kUPPlane);
  uint64_t* q_full = bars;
  uint64_t* q_free = bars + 1;       // the item's last S MMA is done: the next queries may land
  // K and V of a stage have barriers of their own: a K slot is free once S has
  // read it, a V slot once PV has
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + kUStages;
  uint64_t* v_full = k_empty + kUStages;
  uint64_t* v_empty = v_full + kUStages;
  uint64_t* s_full = v_empty + kUStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_free = p_full + 2;
  uint64_t* o_done = p_free + 2;     // one phase per PV (the softmax rescales after PV t-1)
  uint64_t* o_final = o_done + 1;    // [2] the last PV of an item, by output buffer
  uint64_t* o_free = o_final + 2;    // [2] the softmax has read an output buffer
  uint64_t* it_full = o_free + 2;    // [kUSlots] an item is published
  uint64_t* it_free = it_full + kUSlots;   // [kUSlots] every consumer has read it
  uint64_t* mma_done = it_free + kUSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* items = reinterpret_cast<int*>(tmem_slot + 4);           // [kUSlots][kUItem]
  // the two halves' tile maxima [tile parity][half][row] and row sums [item parity][half][row]
  float* xmax = reinterpret_cast<float*>(items + kUSlots * kUItem);
  float* xsum = xmax + 2 * kParts * 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int i = 0; i < kUStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kSoftWarps);
      mbar_init(&p_full[i], kSoftWarps);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_final[i], 1);
      mbar_init(&o_free[i], kSoftWarps);
    }
    for (int i = 0; i < kUSlots; ++i) {
      mbar_init(&it_full[i], 1);
      mbar_init(&it_free[i], kSoftWarps + 2);   // the softmax warps, the MMA issuer and the V producer
    }
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  constexpr bool grid_mode = !PERSIST;
  const uint32_t tmem_cols = kUTmemCols;
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, tmem_cols);
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
  // grid mode: the CTA's one item, decoded by every thread at once.  With
  // early_kv the predecessor released this launch only after its own wait, so
  // every kernel before it is complete: the item and its leading K/V tiles
  // below the block rows are read before the wait (the queries and the block
  // rows' K/V, which the predecessor writes, only after it).
  UItem gx;
  int issued = 0, q_loads = 0;   // producers: K (or V) tiles and query tiles whose loads were issued
  int n_early = 0;
  if constexpr (grid_mode) {
    if (p.early_kv) {
      gx = decode_item<true>(p, 0);
      n_early = early_tiles(gx);
      if (lane == 0 && (warp == kWarpQK || warp == kWarpV)) {
        const bool is_k = warp == kWarpQK;
        uint64_t* full = is_k ? k_full : v_full;
        const int row0 = is_k ? gx.rowK : gx.rowV;
        for (int t = 0; t < n_early; ++t) {   // stage t's first use: no wait for a free slot
          mbar_arrive_expect_tx(&full[t], 2 * kUBox);
          uint8_t* dst = ring + (size_t)t * kUStage + (is_k ? 0 : 2 * kUBox);
          const int pos = gx.p_begin + t * kUTile;
          tma_load_2d(dst, &p.tm_kv, 0, row0 + pos, &full[t]);
          tma_load_2d(dst + kUBox, &p.tm_kv, 64, row0 + pos, &full[t]);
        }
        issued = n_early;
      }
    }
  }
  pdl_wait();   // the queries, the KV arena and the schedule come from the predecessors
  if constexpr (grid_mode) {
    if (!p.early_kv) gx = decode_item<true>(p, 0);
  }
  bool ok = true;
  if (warp == kWarpQK) {
    // ------------------------------------------------ queries and K
    if (lane == 0) {
      const int n_items = grid_mode ? 1 : *p.n_units * p.n_kv * p.n_qtiles;
      (void)n_items;
      for (int i = 0;; ++i) {
        UItem x;
        if constexpr (grid_mode) {   // the CTA's one item, known to every role
          if (i > 0) break;
          x = gx;
        } else {
          const int slot = i % kUSlots;
          if (!mbar_wait(&it_free[slot], (uint32_t)((i / kUSlots) & 1) ^ 1u, abort_flag, p.flags)) {
            ok = false;
            break;
          }
          const int w = (int)atomicAdd(p.item_ctr, 1u);
          if (w < n_items) {
            x = decode_item<false>(p, w);
          } else {
            x.b = -1;
            x.split = x.hk = x.qt = x.p_begin = x.p_end = x.S = x.pg = x.rowK = x.rowV = x.base = 0;
          }
          int* it = items + slot * kUItem;
          it[0] = x.b;
          it[1] = x.split;
          it[2] = x.hk;
          it[3] = x.qt;
          it[4] = x.p_begin;
          it[5] = x.p_end;
          it[6] = x.S;
          it[7] = x.pg;
          it[8] = x.rowK;
          it[9] = x.rowV;
          mbar_arrive(&it_full[slot]);   // (release: the fields above before the arrival)
          if (x.b < 0) break;
        }
        const int nt = item_tiles(x);
        if (nt == 0) continue;
        const int rowK = x.rowK;
        if (q_loads == 0) {   // (after the item's loads: a descriptor prefetch ahead of them delays them)
          tma_prefetch_desc(&p.tm_q);
          tma_prefetch_desc(&p.tm_kv);
        }
        // the queries: once the previous item's last S has read its own
        if (!mbar_wait(q_free, (uint32_t)(q_loads & 1) ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * kUQHalf);
        const int tok = x.b * p.R + x.qt * p.JT;
        tma_load_3d(sQ, &p.tm_q, 0, x.hk * p.G, tok, q_full);
        tma_load_3d(sQ + kUQHalf, &p.tm_q, 64, x.hk * p.G, tok, q_full);
        ++q_loads;
        for (int t = grid_mode ? n_early : 0; t < nt; ++t) {
          const int g = issued, st = g % kUStages;
          if (!mbar_wait(&k_empty[st], (uint32_t)((g / kUStages) & 1) ^ 1u, abort_flag, p.flags)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[st], 2 * kUBox);
          const int pos = x.p_begin + t * kUTile;
          uint8_t* dst = ring + (size_t)st * kUStage;
          tma_load_2d(dst, &p.tm_kv, 0, rowK + pos, &k_full[st]);
          tma_load_2d(dst + kUBox, &p.tm_kv, 64, rowK + pos, &k_full[st]);
          issued = g + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == kWarpV) {
    // ------------------------------------------------ V
    if (lane == 0) {
      for (int i = 0;; ++i) {
        int b, p_begin, p_end, rowV;
        if constexpr (grid_mode) {
          if (i > 0) break;
          b = gx.b, p_begin = gx.p_begin, p_end = gx.p_end, rowV = gx.rowV;
        } else {
          const int slot = i % kUSlots;
          if (!mbar_wait(&it_full[slot], (uint32_t)((i / kUSlots) & 1), abort_flag, p.flags)) {
            ok = false;
            break;
          }
          const int* it = items + slot * kUItem;
          b = it[0], p_begin = it[4], p_end = it[5], rowV = it[9];
          mbar_arrive(&it_free[slot]);
          if (b < 0) break;
        }
        const int nt = p_end > p_begin ? (p_end - p_begin + kUTile - 1) / kUTile : 0;
        if (nt == 0) continue;
        for (int t = grid_mode ? n_early : 0; t < nt; ++t) {
          const int g = issued, st = g % kUStages;
          if (!mbar_wait(&v_empty[st], (uint32_t)((g / kUStages) & 1) ^ 1u, abort_flag, p.flags)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[st], 2 * kUBox);
          const int pos = p_begin + t * kUTile;
          uint8_t* dst = ring + (size_t)st * kUStage + 2 * kUBox;
          tma_load_2d(dst, &p.tm_kv, 0, rowV + pos, &v_full[st]);
          tma_load_2d(dst + kUBox, &p.tm_kv, 64, rowV + pos, &v_full[st]);
          issued = g + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_bf16(128, kUTile);
      const uint32_t idesc_o = umma_idesc_bf16_bmn(128, 128);
      const uint64_t qa[2] = {sw128_kmajor_desc(smem_u32(sQ)), sw128_kmajor_desc(smem_u32(sQ + kUQHalf))};
      struct Pv {
        int g, st, ob, mi;
        bool first, last;
      };
      // O_h += P(g)[:, part h's positions] V(g)[those positions, :] for each
      // softmax part h (its own reference maximum, so its own accumulator):
      // P K-major (64 positions, 128-byte rows), V MN-major (rows = positions,
      // 128 B of dims; the two 64-dim halves 8 KB apart); the first PV of an
      // item overwrites the accumulators, once the softmax has read the last
      // item's
      auto pv = [&](const Pv& x) -> bool {
        const int pb = x.g & 1;
        if (!mbar_wait(&p_full[pb], (uint32_t)((x.g >> 1) & 1), abort_flag, p.flags) ||
            !mbar_wait(&v_full[x.st], (uint32_t)((x.g / kUStages) & 1), abort_flag, p.flags))
          return false;
        if (x.first && !mbar_wait(o_free, (uint32_t)(x.mi & 1) ^ 1u, abort_flag, p.flags)) return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(ring + (size_t)x.st * kUStage + 2 * kUBox);
        constexpr int kPerPart = kUTile / 16 / kParts;   // K = 16 steps of a part's positions
#pragma unroll
        for (int pl = 0; pl < kPPlanes; ++pl) {
          const uint64_t pa = sw128_kmajor_desc(smem_u32(sP + (size_t)(pb * kPPlanes + pl) * kUPPlane));
#pragma unroll
          for (int k = 0; k < kUTile / 16; ++k)   // 16 positions = two 8-row groups = 2048 B of V
            umma_bf16(tmem + 128u + 128u * (uint32_t)(k / kPerPart), pa + 2u * k,
                      sw128_mnmajor_desc(vb + 2048u * k, kUBox, 1024u), idesc_o,
                      (!x.first || pl != 0 || k % kPerPart != 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[x.st]);
        umma_commit(&p_free[pb]);
        umma_commit(o_done);
        if (x.last) umma_commit(o_final);
        return true;
      };
      int g = 0, mi = 0;   // K/V tiles and items with tiles so far
      for (int i = 0; ok; ++i) {
        int p_begin, p_end;
        if constexpr (grid_mode) {
          if (i > 0) break;
          p_begin = gx.p_begin, p_end = gx.p_end;
        } else {
          const int slot = i % kUSlots;
          if (!mbar_wait(&it_full[slot], (uint32_t)((i / kUSlots) & 1), abort_flag, p.flags)) {
            ok = false;
            break;
          }
          const int* it = items + slot * kUItem;
          const int b = it[0];
          p_begin = it[4], p_end = it[5];
          mbar_arrive(&it_free[slot]);
          if (b < 0) break;
        }
        const int nt = p_end > p_begin ? (p_end - p_begin + kUTile - 1) / kUTile : 0;
        if (nt == 0) continue;
        if (!mbar_wait(q_full, (uint32_t)(mi & 1), abort_flag, p.flags)) {
          ok = false;
          break;
        }
        Pv prev{};
        for (int t = 0; t < nt; ++t, ++g) {
          const int st = g % kUStages, sb = g & 1;
          if (!mbar_wait(&k_full[st], (uint32_t)((g / kUStages) & 1), abort_flag, p.flags) ||
              !mbar_wait(&s_free[sb], (uint32_t)((g >> 1) & 1) ^ 1u, abort_flag, p.flags)) {
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
          umma_commit(&k_empty[st]);              // K is read: the slot may take a later tile's K
          if (t == nt - 1) umma_commit(q_free);   // the queries are read: the next item's may land
          if (t > 0 && !pv(prev)) {
            ok = false;
            break;
          }
          prev = Pv{g, st, 0, mi, t == 0, t == nt - 1};
        }
        // the item's last PV at once, so that its output does not wait for
        // the next item's first tile
        if (ok && !pv(prev)) ok = false;
        ++mi;
      }
    }
    if (lane == 0) umma_commit(mma_done);   // tracks every MMA issued above
  } else {
    // ------------------------------------------------ softmax, two threads per query row
    const int r = threadIdx.x & 127;                    // TMEM lane = tile row
    const int hf = threadIdx.x >> 7;                    // part: positions kPCols hf .. of a tile, dims kODims hf ..
    const int qq = warp & 3;                            // TMEM lane quarter
    const uint32_t lane_base = (uint32_t)(qq * 32) << 16;
    int g = 0, mi = 0;   // K/V tiles and items with tiles so far
    for (int i = 0;; ++i) {
      UItem x;
      if constexpr (grid_mode) {
        if (i > 0) break;
        x = gx;
      } else {
        const int slot = i % kUSlots;
        // the pair takes every item together (and leaves together on a failure)
        const bool got = ok && warp_wait(&it_full[slot], (uint32_t)((i / kUSlots) & 1), abort_flag, p.flags);
        if (!quarter_bar_and(qq, got)) {
          ok = false;
          break;
        }
        const int* it = items + slot * kUItem;
        x.b = it[0], x.split = it[1], x.hk = it[2], x.qt = it[3], x.p_begin = it[4], x.p_end = it[5], x.S = it[6],
        x.pg = it[7], x.rowK = x.rowV = 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&it_free[slot]);
        if (x.b < 0) break;
      }
      const int b = x.b, split = x.split, hk = x.hk, qt = x.qt, p_begin = x.p_begin, p_end = x.p_end, S = x.S,
                pg = x.pg;
      const int nt = p_end > p_begin ? (p_end - p_begin + kUTile - 1) / kUTile : 0;
      const int gq = r % p.G, j = qt * p.JT + r / p.G;   // query head hk * G + gq, block row j
      const bool rvalid = j < p.R;
      const int row_lim = block_base(p.st, b) + j;       // causal: the row's own position
      const uint32_t o_tm = tmem + lane_base + 128u + 128u * (uint32_t)hf;   // this part's accumulator
      // this part's reference maximum and row sum over its positions of every
      // tile; the parts combine once, at the output
      float m_ref = -INFINITY, l = 0.f;
      for (int t = 0; t < nt; ++t, ++g) {
        const int sb = g & 1;
        float s[kPCols];
        float hmax = -INFINITY;
        if (ok && warp_wait(&s_full[sb], (uint32_t)((g >> 1) & 1), abort_flag, p.flags)) {
          tc_fence_after();
          if constexpr (kPCols == 32)
            tmem_ld32_issue(tmem + lane_base + (uint32_t)(sb * kUTile + kPCols * hf), s);
          else
            tmem_ld16(tmem + lane_base + (uint32_t)(sb * kUTile + kPCols * hf), s);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[sb]);
          // positions past the split (and, causal, past the row's own
          // position) are masked; the scores stay unscaled (the log2-domain
          // scale goes into the exponent's FMA below and into the maximum)
          const int pos0 = p_begin + t * kUTile + kPCols * hf;
          const int p_row = p.causal ? min(p_end, row_lim + 1) : p_end;
          if (pos0 + kPCols <= p_row) {   // the whole half in range (every tile but a split's last)
#pragma unroll
            for (int i2 = 0; i2 < kPCols; ++i2) hmax = fmaxf(hmax, s[i2]);
          } else {
#pragma unroll
            for (int i2 = 0; i2 < kPCols; ++i2) {
              const float v = pos0 + i2 < p_row ? s[i2] : -INFINITY;
              s[i2] = v;
              hmax = fmaxf(hmax, v);
            }
          }
        } else {
          ok = false;
          break;
        }
        const float tmax = hmax * p.scale_log2;   // this part's tile maximum in the log2 domain
        // reference maximum: set by the part's first tile with a position in
        // range (O and l are still 0 until then), raised only when the part's
        // maximum grows by more than kRescale -- then the part's O and l are
        // rescaled
        float factor = 1.f;
        bool resc = false;
        if (m_ref == -INFINITY) {
          m_ref = tmax;
        } else if (tmax > m_ref + kRescale) {
          factor = exp2f(m_ref - tmax);
          m_ref = tmax;
          resc = true;
        }
        if (__any_sync(0xffffffffu, resc)) {   // the warp rescales its half of its 32 rows of O (PV of tile t-1 done)
          // S(g) was committed after PV(g-2) and PV(g) waits for this tile's P, so
          // o_done is in phase g-1 or g: the parity wait is unambiguous
          if (!warp_wait(o_done, (uint32_t)((g - 1) & 1), abort_flag, p.flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 16) {
            float o16[16];
            tmem_ld16(o_tm + (uint32_t)c, o16);
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) o16[i2] *= factor;
            tmem_st16(o_tm + (uint32_t)c, o16);
          }
          tmem_wait_st();
          l *= factor;
        }
        // P = 2^(s * scale - m_ref) <= 2^kRescale in bf16
        // (a causal row may see no position of this split: its scores are all
        // -inf, and so is m_ref; 0 as the reference makes P = 0, l = 0); the
        // exponent's FMA and the row sum on pairs (packed fp32 instructions)
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        uint32_t hi[kPCols / 2], lo[kPCols / 2];
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-mr, -mr);
        float2 ps2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i2 = 0; i2 < kPCols / 2; ++i2) {
          const float2 x2 = __ffma2_rn(make_float2(s[2 * i2], s[2 * i2 + 1]), sc2, nm2);
          const float p0 = ex2_ftz(x2.x), p1 = ex2_ftz(x2.y);
          ps2 = __fadd2_rn(ps2, make_float2(p0, p1));
          // hi = p with its low 16 bits cleared (p >= 0: truncation, exact as
          // bf16), lo = the exact remainder rounded to bf16
          if constexpr (kPPlanes == 2) {
            const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
            hi[i2] = __byte_perm(u0, u1, 0x7632);
            lo[i2] = pack_bf16x2(p0 - __uint_as_float(u0 & 0xffff0000u), p1 - __uint_as_float(u1 & 0xffff0000u));
          } else {
            hi[i2] = pack_bf16x2(p0, p1);
          }
        }
        l += ps2.x + ps2.y;
        const int pb = g & 1;
        if (!warp_wait(&p_free[pb], (uint32_t)((g >> 1) & 1) ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        st_swizzled_part(sP + (size_t)(pb * kPPlanes) * kUPPlane, r, (kPCols / 8) * hf, hi);
        if constexpr (kPPlanes == 2) st_swizzled_part(sP + (size_t)(pb * 2 + 1) * kUPPlane, r, (kPCols / 8) * hf, lo);
        fence_proxy_async_smem();   // generic-proxy P writes -> the tensor core's reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[pb]);
      }
      // ------------------------------------------------ output: O / l
      // the parts combine: their reference maxima and row sums meet in shared
      // memory (every softmax thread meets its partners here on every path),
      // each part's O is weighted by 2^(m_part - M), M the largest, and the
      // sums are taken in part order (every thread of the row gets the same)
      float* xm = xmax + (i & 1) * kParts * 128;
      float* xs = xsum + (i & 1) * kParts * 128;
      xm[hf * 128 + r] = m_ref;
      xs[hf * 128 + r] = l;
      quarter_bar(qq);
      float w[kParts];
      float mrow = xm[r];
#pragma unroll
      for (int q2 = 1; q2 < kParts; ++q2) mrow = fmaxf(mrow, xm[q2 * 128 + r]);
      float lrow = 0.f;
#pragma unroll
      for (int q2 = 0; q2 < kParts; ++q2) {
        const float mq = xm[q2 * 128 + r];
        w[q2] = mq == -INFINITY ? 0.f : exp2f(mq - mrow);
        lrow += xs[q2 * 128 + r] * w[q2];
      }
      if (ok) {
        const int qd = p.n_q * 128;
        const float inv = lrow > 0.f ? 1.0f / lrow : 0.f;
        const float lse = lrow > 0.f ? mrow + log2f(lrow) : -INFINITY;
        // the item's last PV has its own barrier: by now o_done may be anywhere
        // between the last two phases, so a parity wait on it would be ambiguous
        const bool have = nt > 0 && warp_wait(o_final, (uint32_t)(mi & 1), abort_flag, p.flags);
        if (nt > 0 && !have) ok = false;
        if (ok) {
          tc_fence_after();
          const int rq = gq * p.R + j;   // row of the merge kernel's layout
          const size_t prow = ((size_t)pg * p.n_kv + (size_t)hk * S + split) * p.rows_pad + rq;
          __nv_bfloat16* orow = p.o + (size_t)(b * p.R + j) * qd + (size_t)(hk * p.G + gq) * 128;
          const int h = kODims * hf;   // this thread's output columns, from every part's accumulator
          float o64[kODims];
#pragma unroll
          for (int i2 = 0; i2 < kODims; ++i2) o64[i2] = 0.f;
          if (have) {
#pragma unroll
            for (int q2 = 0; q2 < kParts; ++q2) {
              const uint32_t oq = tmem + lane_base + 128u + 128u * (uint32_t)q2;
#pragma unroll
              for (int c32 = 0; c32 < kODims; c32 += 32) {
                float v32[32];
                tmem_ld32_issue(oq + (uint32_t)(h + c32), v32);
                tmem_wait_ld();
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) o64[c32 + i2] = fmaf(v32[i2], w[q2], o64[c32 + i2]);
              }
            }
            // the accumulators are read: the next item may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
          }
          bool bad = false;   // an fp16 output out of range, latched once below
          if (rvalid) {
#pragma unroll
            for (int cc = 0; cc < kODims; cc += 16) {
              const float* o16 = o64 + cc;
              const int c = h + cc;
              if (S == 1 && p.o_plane == kF16Plane) {   // one fp16 plane
                uint32_t wh[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {
                  bad |= f16_out_of_range(o16[2 * i2] * inv) || f16_out_of_range(o16[2 * i2 + 1] * inv);
                  const __half2 v = __floats2half2_rn(o16[2 * i2] * inv, o16[2 * i2 + 1] * inv);
                  wh[i2] = *reinterpret_cast<const uint32_t*>(&v);
                }
                uint4* dh = reinterpret_cast<uint4*>(orow + c);
                dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
              } else if (S == 1) {   // split bf16: hi plane, lo plane o_plane further
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {
                  __nv_bfloat16 h0, l0, h1, l1;
                  split_bf16(o16[2 * i2] * inv, &h0, &l0);
                  split_bf16(o16[2 * i2 + 1] * inv, &h1, &l1);
                  wh[i2] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                  wl[i2] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
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
                for (int i2 = 0; i2 < 4; ++i2)
                  po[i2] = make_float4(o16[4 * i2] * inv, o16[4 * i2 + 1] * inv, o16[4 * i2 + 2] * inv,
                                       o16[4 * i2 + 3] * inv);
              }
            }
          }
          if (bad) set_flag(p.flags, DFLASH_FLAG_F16_RANGE);
          if (rvalid && S > 1 && hf == 0) p.part_lse[prow] = lse;
        }
      }
      if (nt > 0) ++mi;
    }
  }

  if (!ok) {
    *abort_flag = 1;
    set_flag(p.flags, DFLASH_FLAG_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && (warp == kWarpQK || warp == kWarpV) && lane == 0) {
    // let every load still in flight land before the shared memory goes away
    if (q_loads > 0) (void)mbar_wait(q_full, (uint32_t)((q_loads - 1) & 1), nullptr);
    uint64_t* full = warp == kWarpQK ? k_full : v_full;
    for (int t = max(0, issued - kUStages); t < issued; ++t)
      (void)mbar_wait(&full[t % kUStages], (uint32_t)((t / kUStages) & 1), nullptr);
  }
  if (warp == kWarpMma) {
    if (lane == 0) (void)mbar_wait(mma_done, 0u, nullptr);   // MMAs done before TMEM is freed
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

size_t attn_umma_smem_bytes() {
  return 1024 + 2 * kUQHalf + kUStages * kUStage + 2 * kPPlanes * kUPPlane +
         (2 + 4 * kUStages + 8 + 1 + 4 + 2 * kUSlots + 1) * 8 + 16 + kUSlots * kUItem * sizeof(int) +
         (2 * kParts * 128 + 2 * kParts * 128) * sizeof(float);
}

cudaError_t launch_attention_umma(const AttnUParams& p, int B, int grid, cudaStream_t s) {
  static bool configured = false;
  const size_t smem = attn_umma_smem_bytes();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_umma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_umma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 g = p.work != nullptr ? dim3(grid) : dim3(p.n_splits, p.n_kv * p.n_qtiles, B);
  if (p.work != nullptr)
    launch_k(attn_umma_kernel<true>, g, dim3(kUThreads), smem, s, p);
  else
    launch_k(attn_umma_kernel<false>, g, dim3(kUThreads), smem, s, p);
  return cudaGetLastError();
}

}  // namespace dfl
