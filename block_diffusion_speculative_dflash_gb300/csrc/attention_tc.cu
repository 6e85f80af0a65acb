// Block-bidirectional GQA attention on tensor cores (bf16, head_dim 128).
//
// [GDB §用于注意力机制的“双缓存”方案]: block attention is non-causal, so no mask
// applies -- each of the G*R query rows of a KV head (G = n_q / n_kv query
// heads x R block rows) attends to all kv_len_b context slots and all R block
// slots of its sequence.
//
// One CTA = (KV split, KV head x query tile, sequence).  A producer warp
// streams 64-position K and V tiles of the KV arena into a 3-stage shared
// memory ring with TMA (two 64 x 64 boxes per operand, 128-byte swizzle);
// each consumer warp owns 16 query rows, computes S = Q K^T (bf16 in) and
// O += P V (P and V as fp16) with mma.sync m16n8k16 and fp32 accumulators
// (ldmatrix reads the swizzled tiles conflict-free), keeps the online softmax in fp32 with
// quad shuffles for the row max and sum.  With more than one KV split, each
// split writes its normalised partial output and log2-sum-exp, and a merge
// kernel combines them; splits are balanced on the device from the live
// kv_len, so a captured graph stays correct as the context grows.
#include <algorithm>
#include <cstdlib>

#include "attn_mma.cuh"
#include "common.cuh"
#include "internal.h"

namespace dfl {

namespace {

constexpr int kTile = 64;                            // KV positions per tile
constexpr int kStages = 3;
constexpr uint32_t kBoxBytes = 64 * 128;             // 64 rows x 64 bf16 (one swizzle span)
constexpr uint32_t kStageBytes = 4 * kBoxBytes;      // K[0:64], K[64:128], V[0:64], V[64:128]

__global__ void __launch_bounds__(288, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  const int NW = (int)(blockDim.x >> 5) - 1;  // consumer warps; the last warp produces
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int hk = blockIdx.y % p.n_kv, qt = blockIdx.y / p.n_kv;
  const int b = blockIdx.z;

  const int cap = p.st.cap[b];
  int L = block_base(p.st, b) + p.st.rblk[b];   // context + this sequence's K_b + 1 block rows
  if (L > cap) {
    if (threadIdx.x == 0 && split == 0 && hk == 0 && qt == 0) set_flag(p.flags, DFLASH_FLAG_CAPACITY);
    L = cap;
  }
  // balanced split of [0, L) into n_splits ranges of whole tiles
  const int chunk = ((L + p.n_splits - 1) / p.n_splits + kTile - 1) / kTile * kTile;
  const int p_begin = split * chunk;
  const int p_end = min(L, p_begin + chunk);
  const int ntiles = p_end > p_begin ? (p_end - p_begin + kTile - 1) / kTile : 0;
  const int64_t base = p.st.kv_base[b];
  const int rowK = (int)kv_row(p.kv, base, cap, p.layer, 0, hk, 0);
  const int rowV = (int)kv_row(p.kv, base, cap, p.layer, 1, hk, 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], (uint32_t)NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  bool ok = true;
  int issued = 0;
  if (warp == NW) {
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&p.tm_kv);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kStages;
        const uint32_t ph = (uint32_t)(t / kStages) & 1u;
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.flags)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        const int pos = p_begin + t * kTile;
        uint8_t* dst = tiles + (size_t)st * kStageBytes;
        tma_load_2d(dst, &p.tm_kv, 0, rowK + pos, &full[st]);
        tma_load_2d(dst + kBoxBytes, &p.tm_kv, 64, rowK + pos, &full[st]);
        tma_load_2d(dst + 2 * kBoxBytes, &p.tm_kv, 0, rowV + pos, &full[st]);
        tma_load_2d(dst + 3 * kBoxBytes, &p.tm_kv, 64, rowV + pos, &full[st]);
        issued = t + 1;
      }
    }
  } else {
    const int g = lane >> 2, q4 = lane & 3;
    const int r0 = (qt * NW + warp) * 16;
    const int qd = p.n_q * 128;
    // Q fragments (A operand, row-major 16 x 128) straight from global memory
    uint32_t qa[8][4];
    const __nv_bfloat16* qrow[2];
    bool rv[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = r0 + g + 8 * hf;
      rv[hf] = r < p.rows;
      const int rr = rv[hf] ? r : 0;
      const int gq = rr / p.R, j = rr % p.R;
      qrow[hf] = p.q + (size_t)(b * p.R + j) * qd + (size_t)(hk * p.G + gq) * 128;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        qa[ks][hf] = rv[hf] ? *reinterpret_cast<const uint32_t*>(qrow[hf] + ks * 16 + 2 * q4) : 0u;
        qa[ks][2 + hf] = rv[hf] ? *reinterpret_cast<const uint32_t*>(qrow[hf] + ks * 16 + 8 + 2 * q4) : 0u;
      }

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int mi = lane >> 3, rr8 = lane & 7;

    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kStages;
      const uint32_t ph = (uint32_t)(t / kStages) & 1u;
      if (!mbar_wait(&full[st], ph, abort_flag, p.flags)) {
        ok = false;
        break;
      }
      const uint32_t kb = smem_u32(tiles + (size_t)st * kStageBytes);
      const uint32_t vb = kb + 2 * kBoxBytes;

      // S = Q K^T over 64 positions (8 n-tiles of 8)
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        const int row = nt * 8 + rr8;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          const int d0 = kp * 32 + mi * 8;
          uint32_t bk[4];
          ldsm_x4(kb + (uint32_t)(d0 >> 6) * kBoxBytes + swz(row, (d0 & 63) >> 3), bk);
          mma_bf16(s[nt], qa[2 * kp], bk[0], bk[1]);
          mma_bf16(s[nt], qa[2 * kp + 1], bk[2], bk[3]);
        }
      }
      // mask, running max (quad shuffles), rescale
      const int pos0 = p_begin + t * kTile;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = pos0 + nt * 8 + 2 * q4 + (e & 1);
          const float v = pos < p_end ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      float corr[2];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        mx[hf] = fmaxf(mx[hf], __shfl_xor_sync(0xffffffffu, mx[hf], 1));
        mx[hf] = fmaxf(mx[hf], __shfl_xor_sync(0xffffffffu, mx[hf], 2));
        const float mn = fmaxf(m_run[hf], mx[hf]);
        corr[hf] = exp2f(m_run[hf] - mn);
        m_run[hf] = mn;
        l_run[hf] *= corr[hf];
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= corr[0];
        o[i][1] *= corr[0];
        o[i][2] *= corr[1];
        o[i][3] *= corr[1];
      }
      // P = exp2(S - m) as bf16 A fragments; O += P V
      uint32_t pa[4][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float p0 = exp2f(s[nt][0] - m_run[0]), p1 = exp2f(s[nt][1] - m_run[0]);
        const float p2 = exp2f(s[nt][2] - m_run[1]), p3 = exp2f(s[nt][3] - m_run[1]);
        l_run[0] += p0 + p1;
        l_run[1] += p2 + p3;
        pa[nt >> 1][(nt & 1) * 2 + 0] = pack_f16(p0, p1);
        pa[nt >> 1][(nt & 1) * 2 + 1] = pack_f16(p2, p3);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = kk * 16 + (mi & 1) * 8 + rr8;
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const int d0 = dp * 16 + (mi >> 1) * 8;
          uint32_t bv[4];
          ldsm_x4_t(vb + (uint32_t)(d0 >> 6) * kBoxBytes + swz(row, (d0 & 63) >> 3), bv);
#pragma unroll
          for (int e = 0; e < 4; ++e) bv[e] = bf16x2_to_f16x2(bv[e]);
          mma_f16(o[2 * dp], pa[kk], bv[0], bv[1]);
          mma_f16(o[2 * dp + 1], pa[kk], bv[2], bv[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // finish the row sums across the quad
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 1);
      l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 2);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (!rv[hf]) continue;
      const int r = r0 + g + 8 * hf;
      const float inv = l_run[hf] > 0.f ? 1.0f / l_run[hf] : 0.f;
      if (p.n_splits == 1) {
        const int gq = r / p.R, j = r % p.R;
        __nv_bfloat16* orow = p.o + (size_t)(b * p.R + j) * qd + (size_t)(hk * p.G + gq) * 128;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {   // split bf16: hi plane, lo plane o_plane further
          if (p.o_plane == kF16Plane) {     // or one fp16 plane
            check_f16(o[dt][2 * hf] * inv, p.flags);
            check_f16(o[dt][2 * hf + 1] * inv, p.flags);
            *reinterpret_cast<__half2*>(orow + dt * 8 + 2 * q4) =
                __floats2half2_rn(o[dt][2 * hf] * inv, o[dt][2 * hf + 1] * inv);
            continue;
          }
          __nv_bfloat16 h0, l0, h1, l1;
          split_bf16(o[dt][2 * hf] * inv, &h0, &l0);
          split_bf16(o[dt][2 * hf + 1] * inv, &h1, &l1);
          *reinterpret_cast<__nv_bfloat162*>(orow + dt * 8 + 2 * q4) = __halves2bfloat162(h0, h1);
          *reinterpret_cast<__nv_bfloat162*>(orow + p.o_plane + dt * 8 + 2 * q4) = __halves2bfloat162(l0, l1);
        }
      } else {
        const size_t prow = (((size_t)(b * p.n_kv + hk) * p.n_splits + split) * p.rows_pad + r);
        float* po = p.part_o + prow * 128;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
          *reinterpret_cast<float2*>(po + dt * 8 + 2 * q4) = make_float2(o[dt][2 * hf] * inv, o[dt][2 * hf + 1] * inv);
        if (q4 == 0) p.part_lse[prow] = l_run[hf] > 0.f ? m_run[hf] + log2f(l_run[hf]) : -INFINITY;
      }
    }
  }

  if (!ok) {
    *abort_flag = 1;
    set_flag(p.flags, DFLASH_FLAG_WAIT_TIMEOUT);
  }
  __syncthreads();
  if (*abort_flag && warp == NW && lane == 0) {
    for (int t = max(0, issued - kStages); t < issued; ++t)
      (void)mbar_wait(&full[t % kStages], (uint32_t)(t / kStages) & 1u, nullptr);
  }
}

// The same merge with one CTA per row and thread d = output dimension d (four
// warps per row): for grids of few rows, where one warp per row leaves the
// SMs short of warps to hide the partials' latency.  Up to kMergeBatch
// partials per thread are requested together.
constexpr int kMergeBatch = 32;   // = warp size: lane d holds split d's lse
__global__ void __launch_bounds__(128) attn_merge_dim_kernel(const float* __restrict__ part_o,
                                                             const float* __restrict__ part_lse, int n_kv, int S,
                                                             int rows, int rows_pad, int R, int G, int n_q,
                                                             __nv_bfloat16* __restrict__ o, size_t o_plane,
                                                             uint32_t* flags, const int32_t* __restrict__ seq_split) {
  pdl_trigger();
  pdl_wait();
  __shared__ float w_s[kMergeBatch];
  __shared__ float mx_s;
  const int r = blockIdx.x, hk = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  if (r >= rows) return;
  size_t base;
  if (seq_split != nullptr) {   // per-sequence splits; one split was written directly
    S = seq_split[2 * b];
    if (S <= 1) return;
    base = ((size_t)seq_split[2 * b + 1] * n_kv + (size_t)hk * S) * rows_pad + r;
  } else {
    base = (size_t)(b * n_kv + hk) * S * rows_pad + r;
  }
  float v[kMergeBatch];
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k) v[k] = k < S ? __ldcg(part_o + (base + (size_t)k * rows_pad) * 128 + d) : 0.f;
  float mx = -INFINITY, l_first = -INFINITY;
  if (d < 32) {   // max over every split's lse, one warp
    for (int s0 = 0; s0 < S; s0 += 32) {
      const float l = s0 + d < S ? __ldcg(part_lse + base + (size_t)(s0 + d) * rows_pad) : -INFINITY;
      if (s0 == 0) l_first = l;
      mx = fmaxf(mx, l);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
    if (d == 0) mx_s = mx;
  }
  __syncthreads();
  mx = mx_s;
  float acc = 0.f, wsum = 0.f;
  for (int s0 = 0; s0 < S; s0 += kMergeBatch) {
    if (s0 > 0) {
      __syncthreads();   // every thread is done with the previous weights
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k)
        v[k] = s0 + k < S ? __ldcg(part_o + (base + (size_t)(s0 + k) * rows_pad) * 128 + d) : 0.f;
    }
    if (d < kMergeBatch) {   // weight of split s0 + d (0 where skipped or past S)
      const float l = s0 == 0 ? l_first
                              : s0 + d < S ? __ldcg(part_lse + base + (size_t)(s0 + d) * rows_pad) : -INFINITY;
      w_s[d] = l == -INFINITY ? 0.f : exp2f(l - mx);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      if (s0 + k >= S) break;
      const float w = w_s[k];
      if (w == 0.f) continue;
      acc += w * v[k];
      wsum += w;
    }
  }
  const int gq = r / R, j = r % R;
  __nv_bfloat16* od = o + (size_t)(b * R + j) * n_q * 128 + (size_t)(hk * G + gq) * 128 + d;
  put_op(wsum > 0.f ? acc / wsum : 0.f, od, o_plane, flags);
}

// o = sum_s w_s o_s / sum_s w_s with w_s = 2^(lse_s - max lse), sums in split
// order; splits with no position (lse = -inf) are skipped.  One warp per row,
// up to kMergeRows rows per CTA (fewer when the rows would not fill the GPU); lane l owns output dimensions 4l .. 4l+3 (16-byte
// loads), and lane k computes split k's weight, which the warp broadcasts.  The
// partials of up to VEC splits are requested together (one round trip for a
// row with that many splits; VEC follows S); loads past S are not issued.
constexpr int kMergeRows = 8;
template <int VEC>
__global__ void __launch_bounds__(32 * kMergeRows) attn_merge_kernel(const float* __restrict__ part_o,
                                                                    const float* __restrict__ part_lse, int n_kv,
                                                                    int S, int rows, int rows_pad, int R, int G,
                                                                    int n_q, __nv_bfloat16* __restrict__ o,
                                                                    size_t o_plane, uint32_t* flags,
                                                                    const int32_t* __restrict__ seq_split) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), hk = blockIdx.y, b = blockIdx.z;
  if (r >= rows) return;   // (whole warps)
  size_t base;
  if (seq_split != nullptr) {   // per-sequence splits; one split was written directly
    S = seq_split[2 * b];
    if (S <= 1) return;
    base = ((size_t)seq_split[2 * b + 1] * n_kv + (size_t)hk * S) * rows_pad + r;
  } else {
    base = (size_t)(b * n_kv + hk) * S * rows_pad + r;
  }
  float mx = -INFINITY;
  for (int s0 = 0; s0 < S; s0 += 32)
    mx = fmaxf(mx, s0 + lane < S ? __ldcg(part_lse + base + (size_t)(s0 + lane) * rows_pad) : -INFINITY);
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, wsum = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const float l = s0 + lane < S ? __ldcg(part_lse + base + (size_t)(s0 + lane) * rows_pad) : -INFINITY;
    const float wl = l == -INFINITY ? 0.f : exp2f(l - mx);
    const int n = min(32, S - s0);   // warp-uniform
    for (int k0 = 0; k0 < n; k0 += VEC) {
      float4 v[VEC];
#pragma unroll
      for (int k = 0; k < VEC; ++k)
        v[k] = k0 + k < n
                   ? __ldcg(reinterpret_cast<const float4*>(part_o + (base + (size_t)(s0 + k0 + k) * rows_pad) * 128) +
                            lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        if (k0 + k >= n) break;                                  // uniform
        const float w = __shfl_sync(0xffffffffu, wl, k0 + k);   // k0 + k < 32
        if (w == 0.f) continue;                                  // uniform
        a0 += w * v[k].x;
        a1 += w * v[k].y;
        a2 += w * v[k].z;
        a3 += w * v[k].w;
        wsum += w;
      }
    }
  }
  const float y[4] = {wsum > 0.f ? a0 / wsum : 0.f, wsum > 0.f ? a1 / wsum : 0.f, wsum > 0.f ? a2 / wsum : 0.f,
                      wsum > 0.f ? a3 / wsum : 0.f};
  const int gq = r / R, j = r % R;
  __nv_bfloat16* od = o + (size_t)(b * R + j) * n_q * 128 + (size_t)(hk * G + gq) * 128 + 4 * lane;
  if (o_plane == kF16Plane) {   // one fp16 plane
#pragma unroll
    for (int i = 0; i < 4; ++i) check_f16(y[i], flags);
    const __half2 h01 = __floats2half2_rn(y[0], y[1]), h23 = __floats2half2_rn(y[2], y[3]);
    *reinterpret_cast<uint2*>(od) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
    return;
  }
  __nv_bfloat16 hi[4], lo[4];   // split bf16: hi plane, lo plane o_plane further
#pragma unroll
  for (int q = 0; q < 4; ++q) split_bf16(y[q], &hi[q], &lo[q]);
  const auto pk = [](__nv_bfloat16 x0, __nv_bfloat16 x1) {
    return (uint32_t)__bfloat16_as_ushort(x0) | ((uint32_t)__bfloat16_as_ushort(x1) << 16);
  };
  *reinterpret_cast<uint2*>(od) = make_uint2(pk(hi[0], hi[1]), pk(hi[2], hi[3]));
  *reinterpret_cast<uint2*>(od + o_plane) = make_uint2(pk(lo[0], lo[1]), pk(lo[2], lo[3]));
}

}  // namespace

size_t attn_tc_smem_bytes() { return 1024 + kStages * kStageBytes + 2 * kStages * 8 + 16; }

cudaError_t launch_attn_merge(const float* part_o, const float* part_lse, int n_kv, int S, int rows, int rows_pad,
                              int R, int G, int n_q, __nv_bfloat16* o, size_t o_plane, int B, cudaStream_t s,
                              uint32_t* flags, const int32_t* seq_split) {
  // rows per CTA: up to kMergeRows while the grid still gives every SM about two CTAs
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n_sm = 1;
  }
  const int64_t total = (int64_t)rows * n_kv * B;
  static int mode = -1;   // DFLASH_MERGE=dim / warp: one shape at every size
  if (mode < 0) {
    const char* m = getenv("DFLASH_MERGE");
    mode = m && m[0] == 'd' ? 1 : m && m[0] == 'w' ? 2 : 0;
  }
  if (mode == 1 || (mode == 0 && total < 8 * 2 * (int64_t)n_sm)) {
    launch_k(attn_merge_dim_kernel, dim3(rows, n_kv, B), dim3(128), 0, s, part_o, part_lse, n_kv, S, rows, rows_pad, R,
             G, n_q, o, o_plane, flags, seq_split);
    return cudaGetLastError();
  }
  const int rpc = (int)std::max<int64_t>(1, std::min<int64_t>(kMergeRows, total / (2 * (int64_t)n_sm)));
  const dim3 grid((rows + rpc - 1) / rpc, n_kv, B), block(32 * rpc);
  if (S <= 4)
    launch_k(attn_merge_kernel<4>, grid, block, 0, s, part_o, part_lse, n_kv, S, rows, rows_pad, R, G, n_q, o, o_plane,
             flags, seq_split);
  else if (S <= 16)
    launch_k(attn_merge_kernel<16>, grid, block, 0, s, part_o, part_lse, n_kv, S, rows, rows_pad, R, G, n_q, o, o_plane,
             flags, seq_split);
  else
    launch_k(attn_merge_kernel<32>, grid, block, 0, s, part_o, part_lse, n_kv, S, rows, rows_pad, R, G, n_q, o, o_plane,
             flags, seq_split);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const AttnTcParams& p, int n_consumer_warps, int B, cudaStream_t s) {
  static bool configured = false;
  const size_t smem = attn_tc_smem_bytes();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.n_splits, p.n_kv * p.n_qtiles, B);
  launch_k(attn_tc_kernel, dim3(grid), dim3((n_consumer_warps + 1) * 32), smem, s, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_splits == 1) return e;
  return launch_attn_merge(p.part_o, p.part_lse, p.n_kv, p.n_splits, p.rows, p.rows_pad, p.R, p.G, p.n_q, p.o, p.o_plane,
                           B, s, p.flags);
}

}  // namespace dfl
