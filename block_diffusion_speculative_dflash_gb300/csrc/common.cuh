// Device helpers shared by the drafter kernels: bf16 access, bounded mbarrier
// waits, TMA (cp.async.bulk.tensor) and tcgen05 (5th-generation tensor core,
// accumulators in tensor memory) wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash.h"
#include "internal.h"

namespace dfl {

// ---------------------------------------------------------------- types

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <typename T> __device__ __forceinline__ float ldf(const T* p) { return Elem<T>::load(p); }
template <typename T> __device__ __forceinline__ T stf(float v) { return Elem<T>::from_f(v); }

__device__ __forceinline__ void set_flag(uint32_t* flags, uint32_t bit) {
  if (flags) atomicOr(flags, bit);
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Eight warp sums at once: lane l returns the sum over all lanes of
// v[4*b4 + 2*b3 + b2] (b_k = bit k of l).  Each slot is summed by the same xor
// tree as warp_sum (partners 16, 8, 4, 2, 1, every node an own + partner add), so
// each result equals warp_sum of that slot bit for bit, in 9 shuffles, not 40.
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
  const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
  float w[4], x[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float keep = b4 ? v[4 + k] : v[k], send = b4 ? v[k] : v[4 + k];
    w[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float keep = b3 ? w[2 + k] : w[k], send = b3 ? w[k] : w[2 + k];
    x[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
  y += __shfl_xor_sync(0xffffffffu, y, 2);
  y += __shfl_xor_sync(0xffffffffu, y, 1);
  return y;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum; `red` holds >= 32 floats of shared memory.  All threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
  if (warp == 0) {
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Packed (value, index) key: max over keys = max value, lowest index on ties.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  return ((unsigned long long)ordered_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}

// ---------------------------------------------------------------- RoPE

// cos / sin of the rotate-half RoPE angle pos * theta^(-2i/d) of pair i.  The
// frequency comes as F = theta^(-2i/d) / (2 pi) in turns, as a 0.64 fixed-point
// fraction; pos * F in 64-bit integers wraps exactly modulo one turn, so the
// reduction is exact for any position, and the turn fraction goes to sincospif
// (sin / cos of pi * x, x = 2 * turns in [0, 2)).
__device__ __forceinline__ void rope_cs(int pos, uint64_t turns, float* c, float* s) {
  const uint64_t ph = (uint64_t)(uint32_t)pos * turns;
  const float x = (float)(uint32_t)(ph >> 32) * 4.656612873077392578125e-10f;   // 2^-31
  sincospif(x, s, c);
}
// The same reduction, with the hardware sin / cos on pi * x for x taken into
// [-1, 1) (absolute error ~1e-6, three orders below the bf16 rounding of the
// rotated q and K rows it serves): the tensor-core epilogues rotate hundreds
// of tokens per thread, where the library routine's code and latency dominate.
__device__ __forceinline__ void rope_cs_fast(int pos, uint64_t turns, float* c, float* s) {
  const uint64_t ph = (uint64_t)(uint32_t)pos * turns;
  const int32_t q = (int32_t)(uint32_t)(ph >> 32);   // turns as a signed 0.32 fraction: [-1/2, 1/2)
  __sincosf((float)q * 1.46291808e-9f, s, c);           // 2 pi / 2^32 rad per unit
}

// ---------------------------------------------------------------- timing / waits

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Every spin-wait in these kernels gives up after a time limit, latches
// DFLASH_FLAG_WAIT_TIMEOUT and lets the kernel unwind.  The limit is the
// context's (dflash_set_wait_limit): a 64-bit count of nanoseconds kept next to
// its device flag word, at flags + 2 (zero: this default).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// The flag word and the wait limit in one 16-byte load (the flags are 16-byte
// aligned): a waiting thread checks both without an extra round trip.
__device__ __forceinline__ void ld_flags_limit(const uint32_t* gflags, uint32_t* fl, uint64_t* limit) {
  uint64_t a, b;
  asm volatile("ld.volatile.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(gflags) : "memory");
  *fl = (uint32_t)a;
  *limit = b != 0 ? b : kWaitLimitNs;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Raise the barrier's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`.  Returns false when the time limit
// ran out, another role of the CTA raised `*abort`, or any CTA already latched
// DFLASH_FLAG_WAIT_TIMEOUT in the context's device flags (so that one stuck
// CTA does not make every later CTA wait out its own limit).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          const uint32_t* gflags = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint64_t limit = kWaitLimitNs;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (gflags != nullptr) {
        uint32_t fl;
        ld_flags_limit(gflags, &fl, &limit);
        if (fl & DFLASH_FLAG_WAIT_TIMEOUT) return false;
      }
      if (globaltimer_ns() - t0 > limit) return false;
    }
  }
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation: a kernel may
// start while its predecessor drains.  Every kernel first allows its own
// successor to launch (pdl_trigger) and waits for its predecessor (pdl_wait)
// before touching anything the predecessor writes or reads; work that depends
// on neither (weight prefetch, barrier set-up) goes before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// The dependency wait of a kernel that releases its dependents either at its
// start (late == 0: the caller triggered already) or only here, after the wait
// (late != 0).  Released late, a dependent launches only once this kernel's
// predecessor has completed, and with it (each kernel completes only after its
// own wait) every kernel before: it may then read, before its own wait,
// anything those kernels wrote.
__device__ __forceinline__ void pdl_wait_release(int late) {
  pdl_wait();
  if (late) pdl_trigger();
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
// 2D tiled bulk tensor load global -> shared, completion on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* tm, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// L2 cache policy for data read once (the weight stream): its lines are the
// first to be evicted, so streaming the weights does not push the small working
// set (activations, partial sums, K/V tiles) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_2d with an L2 cache policy
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Hint: bring one tensor box from HBM into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_hint(const CUtensorMap* tm, int c0, int c1, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(c0), "r"(c1), "l"(policy)
               : "memory");
}

// Hint: bring one 2-D tensor box from HBM into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_box(const CUtensorMap* tm, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tm)),
               "r"(c0), "r"(c1)
               : "memory");
}

// 3D tiled bulk tensor load global -> shared, completion on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Split bf16 storage of an activation x: hi = bf16(x), lo = bf16(x - hi); the
// tensor cores multiply both planes and the epilogue adds the two products, so
// a GEMM's token operand carries about 16 significant bits instead of 8.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16* hi, __nv_bfloat16* lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *hi = h;
  *lo = __float2bfloat16_rn(x - __bfloat162float(h));
}

// fp16 operands hold |x| <= 65504: a value outside (or NaN) latches
// DFLASH_FLAG_F16_RANGE, so the silent inf of the conversion is reported.
__device__ __forceinline__ void check_f16(float x, uint32_t* flags) {
  if (!(fabsf(x) <= 65504.0f)) set_flag(flags, DFLASH_FLAG_F16_RANGE);
}

// Whether x lies outside fp16's range (|x| > 65504, or NaN).
__device__ __forceinline__ bool f16_out_of_range(float x) { return !(fabsf(x) <= 65504.0f); }

// A token operand written as one fp16 plane instead (11 significant bits, one
// MMA against fp16 copies of the weights): the lo-plane offset kF16Plane says so.
__device__ __forceinline__ void put_op(float x, __nv_bfloat16* hi, size_t plane, uint32_t* flags) {
  if (plane == kF16Plane) {
    check_f16(x, flags);
    *reinterpret_cast<__half*>(hi) = __float2half_rn(x);
  } else {
    split_bf16(x, hi, hi + plane);
  }
}
// The same inside a loop: an fp16 value out of range only raises `bad`, which
// the caller latches once after the loop (a flag write per value, even
// predicated off, weighs on the unrolled epilogues' instruction stream).
__device__ __forceinline__ void put_op_acc(float x, __nv_bfloat16* hi, size_t plane, bool& bad) {
  if (plane == kF16Plane) {
    bad |= f16_out_of_range(x);
    *reinterpret_cast<__half*>(hi) = __float2half_rn(x);
  } else {
    split_bf16(x, hi, hi + plane);
  }
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, single thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all tcgen05.mma previously issued by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor: K-major operand tile whose rows are 128 B
// (64 bf16) and were written by TMA with the 128-byte swizzle; 8-row core
// groups are 1024 B apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1u << 16;                              // leading byte offset (unused when swizzled)
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;        // stride byte offset: 8 rows * 128 B
  d |= (uint64_t)1u << 46;                              // descriptor version
  d |= (uint64_t)2u << 61;                              // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}
// the same with A and B both fp16 (format code 0)
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp receives
// row (lane base + t), columns [col, col + 16) of the accumulator.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive columns into r without waiting: a batch of these is followed
// by one tmem_wait_hold8 per 8 registers (the first waits for the batch).
__device__ __forceinline__ void tmem_ld8_issue(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
// Wait for every tensor-memory load this thread issued; the empty statement
// after it takes the loaded registers as operands, so no use of them can be
// scheduled above the wait.
__device__ __forceinline__ void tmem_wait_ld_all() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_hold8(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
}

// The same for 8 consecutive columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace dfl
