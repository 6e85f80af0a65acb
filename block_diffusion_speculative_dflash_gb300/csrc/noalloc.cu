// dflash_draft_block_noalloc: a draft that allocates no device memory.
//
// Who needs it: code that must not call cudaMalloc (or any allocating routine)
// while it drafts -- a decode loop recorded by stream capture in global mode,
// where an allocation call is an error and breaks the capture, or a serving
// process that partitions device memory once at start-up and forbids any later
// allocation.  dflash_draft_block itself may grow a workspace the first time a
// larger draft needs it; this variant never does.
//
// What changes: the one draft kernel whose scratch depends on the live context
// length -- the tensor-core attention's split-KV partial outputs and
// log-sum-exps -- takes that scratch from the file-scope static device array
// below instead of a context workspace, and every context workspace stays at
// its current size (a draft that would need a larger one fails with
// DFLASH_ERR_CAPACITY instead of allocating).  When the split count the draft
// would pick does not fit the array, the attention runs with as many splits as
// fit (down to one split, which needs no scratch), so the ids and logits agree
// with dflash_draft_block's up to the summation order of the split-KV merge
// (fp32 rounding), not bit for bit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dflash.h"

// Capacity of the static split-KV scratch: 2M floats = 8 MiB.  A draft needs
// batch x kv_heads x splits x rows_pad x 129 floats, rows_pad being the query
// rows of a KV head rounded up to 128 (G query heads x (K + 1) block rows); for
// one sequence of 8 KV heads with K + 1 <= 32 block rows of 4 query heads that
// is 8 x 128 x 129 floats per split, so up to 15 splits fit.  Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kScratchFloats = (size_t)2 << 20;
static __device__ __align__(256) float g_split_kv_scratch[kScratchFloats];

int dfl_draft_block_with_scratch(dflash_ctx* c, const int32_t* anchor_ids, int32_t K, int32_t* draft_ids,
                                 float* logits, float* scratch, size_t scratch_floats, void* stream);
int dfl_fail(int code, const char* msg);

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// the array's device address per device, valid for the CUDA context current
// when it was looked up (a reset device gets a new context and a new module
// load, so the address is looked up again)
float* g_addr[kMaxDevices] = {};
CUcontext g_addr_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    cudaGetLastError();
    looked = true;
  }
  return fn;
}

// Device address of the static scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress (with the device current) the first time a device
// -- or a new context on it -- calls, and reused while that context lives.
int scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return dfl_fail(DFLASH_ERR_CUDA, "cannot determine the current device");
  }
  std::lock_guard<std::mutex> lock(g_mu);
  CUcontext cur = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr || get(&cur) != CUDA_SUCCESS) cur = nullptr;
  if (g_addr[dev] == nullptr || cur == nullptr || cur != g_addr_ctx[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_split_kv_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return dfl_fail(DFLASH_ERR_CUDA, "cudaGetSymbolAddress of the static split-KV scratch failed");
    }
    g_addr[dev] = static_cast<float*>(p);
    if (cur == nullptr && get != nullptr && get(&cur) != CUDA_SUCCESS) cur = nullptr;
    g_addr_ctx[dev] = cur;   // null: unknown context, looked up again next call
  }
  *out = g_addr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_draft_block_noalloc(dflash_ctx* ctx, const int32_t* anchor_ids, int32_t K,
                                          int32_t* draft_ids, float* logits, void* stream) {
  float* scratch = nullptr;
  const int r = scratch_address(&scratch);
  if (r != DFLASH_OK) return r;
  return dfl_draft_block_with_scratch(ctx, anchor_ids, K, draft_ids, logits, scratch, kScratchFloats, stream);
}
