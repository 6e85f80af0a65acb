// C-ABI of the drafter: per-context state, KV arena (buddy allocator over
// power-of-two capacities), workspaces, tensor maps and the launch sequences
// of ctx_append / draft_block / verify_accept.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <set>
#include <atomic>
#include <string>
#include <tuple>
#include <vector>

#include "dflash.h"
#include "internal.h"

using namespace dfl;

namespace dfl {
bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("DFLASH_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}
}  // namespace dfl

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                                          \
  do {                                                                                                    \
    cudaError_t e_ = (call);                                                                              \
    if (e_ != cudaSuccess)                                                                                \
      return fail(DFLASH_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
  } while (0)

#define RET(x)                 \
  do {                         \
    int r_ = (x);              \
    if (r_ != DFLASH_OK) return r_; \
  } while (0)

// Allocation-failure injection (dflash_inject_alloc_failure): while >= 0, the
// count of device allocations still to succeed before one fails.
std::atomic<int64_t> g_alloc_fail_after{-1};
bool injected_alloc_failure() {
  int64_t v = g_alloc_fail_after.load();
  while (v >= 0) {
    if (g_alloc_fail_after.compare_exchange_weak(v, v - 1)) return v == 0;
  }
  return false;
}

int64_t next_pow2(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Buddy allocator over token slots of the KV arena.  Blocks are 64 << order
// slots, aligned to their size, so every sequence capacity is a power of two
// and freed neighbours merge back.
struct Buddy {
  static constexpr int64_t kUnit = 64;
  int max_order = 0;
  std::vector<std::set<int64_t>> free_lists;

  void init(int64_t pool_tokens) {
    max_order = 0;
    while ((kUnit << max_order) < pool_tokens) ++max_order;
    free_lists.assign(max_order + 1, {});
    free_lists[max_order].insert(0);
  }
  int64_t pool() const { return kUnit << max_order; }
  static int order_of(int64_t tokens) {
    int o = 0;
    while ((kUnit << o) < tokens) ++o;
    return o;
  }
  int64_t alloc(int64_t tokens) {
    const int o = order_of(tokens);
    if (o > max_order) return -1;
    int k = o;
    while (k <= max_order && free_lists[k].empty()) ++k;
    if (k > max_order) return -1;
    int64_t off = *free_lists[k].begin();
    free_lists[k].erase(free_lists[k].begin());
    while (k > o) {  // split, keep the low half
      --k;
      free_lists[k].insert(off + (kUnit << k));
    }
    return off;
  }
  void release(int64_t off, int64_t tokens) {
    int o = order_of(tokens);
    while (o < max_order) {
      const int64_t buddy = off ^ (kUnit << o);
      auto it = free_lists[o].find(buddy);
      if (it == free_lists[o].end()) break;
      free_lists[o].erase(it);
      off = std::min(off, buddy);
      ++o;
    }
    free_lists[o].insert(off);
  }
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    return false;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix; boxes of
// box_outer rows x 64 columns land in shared memory with the 128-byte swizzle.
int tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_outer) {
  if (!load_encoder()) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)kTileK, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): base %p inner %llu outer %llu", (int)r, base,
                (unsigned long long)inner, (unsigned long long)outer);
  return DFLASH_OK;
}

// Token operand map: bf16 [planes][rows][inner] (planes of rows*inner elements),
// boxes of box_rows x 64 from one plane, 128-byte swizzle.
int tmap_tokens(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, int planes, uint32_t box_rows) {
  if (!load_encoder()) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {inner, rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {(cuuint32_t)kTileK, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled (tokens) failed (%d): base %p inner %llu rows %llu", (int)r,
                base, (unsigned long long)inner, (unsigned long long)rows);
  return DFLASH_OK;
}

// Rotated queries [M][n_q * 128] as a 3-D tensor (dims, heads, tokens) with
// 64 x G x JT boxes: one box is half of head_dim for G heads of JT block rows.
int tmap_queries(CUtensorMap* tm, const void* base, int n_q, uint64_t M, int G, int JT) {
  if (!load_encoder()) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {128, (cuuint64_t)n_q, M};
  cuuint64_t strides[2] = {256, (cuuint64_t)n_q * 256};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)JT};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", (int)r);
  return DFLASH_OK;
}

bool is_device_ptr(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Page-locked host memory (a stream capture can record copies to it).
bool is_pinned_host(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// Bumped whenever a workspace is (re)allocated: a recorded draft graph holds
// the addresses it was captured with and is re-recorded after any change.
std::atomic<uint64_t> g_grow_epoch{0};

bool is_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

struct SegRef {
  const void* w;
  int rows;
  const CUtensorMap* tm;
};

constexpr size_t kCounters = 1u << 16;   // arrival counters of the fused GEMM epilogues

}  // namespace

// Guard bands around the KV arena: bytes of kGuardByte on either side.
constexpr size_t kGuardBytes = 4096;
constexpr int kGuardByte = 0xA5;

struct dflash_ctx {
  dflash_config cfg{};
  dflash_weights w{};
  int B = 0;
  bool bf16 = false;
  size_t esz = 4;
  int num_sms = 148;
  int H = 0, F = 0, I = 0, V = 0, d = 0, nl = 0, q_dim = 0, kv_dim = 0;
  int64_t rows_per_token = 0;  // n_layers * 2 * n_kv arena rows per token slot

  // device state and small buffers
  int32_t* d_i32 = nullptr;
  int32_t* d_pend_base = nullptr;        // [B] kv_len before the last append
  int32_t* d_rblk = nullptr;             // [B] block rows of the last draft (K_b + 1)
  int cond = DFLASH_COND_KV;             // dflash_conditioning of the drafts
  // target model (dflash_target_*): forwards of given tokens with causal
  // attention, an id for every row, features of the selected layers
  bool target = false;
  bool target_plain = false;             // the target's layer inputs plain bf16 at every M (DFLASH_TARGET_PLAIN=1)
  int n_feat = 0;
  int feat_layers[8] = {};
  struct TargetRun {                      // the forward in flight (set by dflash_target_forward)
    const int32_t* tokens;                // device [B][R]
    int32_t* ids;                         // device [B][R]
    float* logits;                        // device [B][R][V] or null
    __nv_bfloat16* feats;                 // device [B][R][n_feat][H] or null
  };
  const TargetRun* trun = nullptr;
  float* d_ulast = nullptr;              // [B][H] input fusion: each sequence's last context feature
  // persistent attention schedule, planned on the device at every draft of a
  // batch: units [B * 64], per-sequence (S_b, pg_b) [B][2], unit count, one
  // item counter per layer
  int32_t* d_plan = nullptr;
  int32_t *d_work = nullptr, *d_seq_split = nullptr, *d_n_units = nullptr, *d_seq_order = nullptr;
  uint32_t* d_attn_ctr = nullptr;
  // the current draft's plan: 0 none, 1 the grid in longest-first order, 2 persistent
  int plan_mode = 0;
  int plan_chunk = 0, plan_groups = 0, plan_grid = 0, plan_smax = 0;
  int32_t* d_kseq_in = nullptr;          // [B] staging of a host per-sequence K
  const int32_t* kseq_dev = nullptr;     // the current draft's per-sequence K (device) or null
  int64_t* d_kv_base = nullptr;
  uint32_t* d_flags = nullptr;
  int32_t *d_ctx_len = nullptr, *d_kv_len = nullptr, *d_anchor = nullptr, *d_cap = nullptr, *d_rows = nullptr,
          *d_rows_in = nullptr, *d_accept = nullptr, *d_next = nullptr, *d_anchor_in = nullptr;
  int32_t* d_draft = nullptr;    // [B, k_max]
  int32_t* d_targets = nullptr;  // [B, k_max + 1]
  uint64_t* d_rope = nullptr;          // RoPE frequencies in turns, 0.64 fixed point
  SeqState st{};

  // KV arena (inside arena_raw, between two guard bands of kGuardBytes)
  void* arena = nullptr;
  void* arena_raw = nullptr;
  size_t arena_bytes = 0;
  Buddy buddy;
  std::vector<int64_t> seg_tok, cap, ub_ctx, ub_kv;
  KvArena kv{};

  // activations and workspaces
  int M_max = 0;
  float* h = nullptr;
  void *xn = nullptr, *qb = nullptr, *ob = nullptr, *ab = nullptr, *xf = nullptr;
  float* ws = nullptr;
  size_t ws_cap = 0;
  void* stage = nullptr;
  size_t stage_cap = 0;
  void* ub = nullptr;
  size_t ub_cap = 0;
  void* attn_ws = nullptr;       // split-KV partial outputs and log-sum-exps
  size_t attn_ws_cap = 0;
  unsigned long long* d_keys = nullptr;  // [B * k_max][kKeySlots][kKeyStride] packed argmax keys
  unsigned int* d_counters = nullptr;    // per-tile arrival counters of the fused GEMM epilogues
  float* d_ss = nullptr;                 // per-tile row sums of squares [H/128][rows]
  size_t ss_rows = 0;
  void* ybuf = nullptr;                  // append: fc output rows (fp32)
  size_t ybuf_cap = 0;
  CUtensorMap tm_kv{};           // the KV arena as [rows, head_dim] bf16

  // tensor maps of the weights (bf16)
  struct LayerMaps {
    CUtensorMap wq, wk, wv, wo, wg, wu, wd;
  };
  std::vector<LayerMaps> lmaps;
  CUtensorMap tm_fc{}, tm_lm{};
  // fp16 copies of every layer's projections and of the LM head (one
  // allocation, made at the first draft of more than 128 rows): the tensor
  // cores take fp16 token operands only against fp16 weights
  bool f16_ops = true;                       // DFLASH_F16_OPS=0: split bf16 operands at every M
  // fp16 operands from this many GEMM rows up (DFLASH_F16_MIN_ROWS): from 33 the
  // split operand's second MMA and wider token boxes cost more than fp16's
  // coarser rounding is worth (Llama-3.1-8B shape, batch 8: 1264 -> 1077 us)
  int f16_min_rows = 33;
  bool op16_now = false;                     // the running draft's token operands are fp16
  bool w16_failed = false;
  char* w16 = nullptr;
  std::vector<dflash_layer_weights> wl16;    // the layers with their matrices in w16
  const void* lm16 = nullptr;
  std::vector<LayerMaps> lmaps16;
  CUtensorMap tm_lm16{};
  std::map<std::tuple<const void*, int, int, int>, CUtensorMap> xmaps;

  int last_K = 0;

  bool attn_umma = true;                 // bf16 attention on tcgen05 (else the mma.sync kernel)
  int gemm_ctas = 0;                     // stand-alone GEMM CTAs per SM the grid is sized for (0: by width)
  int gemm_smem_kb = 0;                  // stand-alone GEMM stage-ring budget per CTA (0: by CTAs per SM)
  bool gemm_pairs = true;                // two token tiles of a split operand per CTA
  bool gemm_direct = true;               // single-split tiles: epilogue straight from tensor memory
  int gemm_bn_max = 192;                 // widest plain-operand token tile (MMA N)
  bool gemm_persist = true;              // multi-wave one-split GEMMs on the persistent instance
  bool gemm_by_epi = true;               // split-K one-tile GEMMs on their epilogue's own instance
  bool attn_early = true;                // grid-mode attention loads its first context K/V before its wait
  bool attn_early_now = false;           // (set around one layer's attention launch)
  bool lm_fused = false;                 // LM head as one GEMM with the argmax in its epilogue (every M)
  // With fuse_append, an append of <= 128 rows leaves its per-layer K/V
  // projection pending: the next draft's QKV GEMMs take the rows u along (each
  // W_k / W_v read once per iteration); anything else that needs the K/V first
  // flushes it.  Off by default: at 17 block rows the wider QKV GEMMs cost the
  // draft 11 us and the iteration gains only 4 us.
  bool fuse_append = false;
  bool pending = false;                  // ub / d_ss_ctx / d_rows / pend_base hold an unprojected append
  int pend_m = 0, pend_rows_max = 0;     // its rows (B * rows_max) and rows_max
  float* d_ss_ctx = nullptr;             // [H / 128][128] folded-norm sums of the pending rows
  bool bn8 = true;                       // split-operand token tiles in steps of 8 rows (else 16)
  bool split_ops = true;                 // GEMM token operands as split bf16 (hi + lo) when M <= 128

  // tracing (event pairs, round-robin) and launch accounting
  std::vector<cudaEvent_t> ev;
  int n_pairs = 0, next_pair = 0;
  // Recorded draft: a dflash_draft_block_k call whose arguments (K and the
  // caller's pointers) and workspaces match the last recorded one replays that
  // graph on a private stream, forked from and joined to the caller's stream,
  // instead of launching its ~35 kernels one by one (the per-sequence state
  // lives in device memory, so a replay is the same draft).  DFLASH_GRAPH=0:
  // every draft launched eagerly.
  bool graph_drafts = true;
  struct DraftGraph {
    bool valid = false;
    int K = 0;
    const void *anchor = nullptr, *kseq = nullptr, *ids = nullptr, *logits = nullptr;
    uint64_t epoch = 0;
    int64_t launches = 0;
    cudaGraphExec_t exec = nullptr;
  } dg;
  cudaStream_t gstream = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  struct TraceEntry {
    int kind, pair;
    double bytes;
  };
  std::vector<TraceEntry> trace;
  int64_t launches = 0;
  int64_t replays = 0;   // drafts served by the recorded graph

  // set only for the duration of a dflash_draft_block_noalloc call
  float* attn_scratch_ext = nullptr;  // caller-provided split-KV scratch
  size_t attn_scratch_ext_floats = 0;
  bool no_grow = false;               // a workspace that would have to grow is an error
};

namespace {

int grow_buffer(void** p, size_t* cap, size_t bytes, cudaStream_t s, const char* what) {
  if (bytes <= *cap) return DFLASH_OK;
  if (is_capturing(s)) return fail(DFLASH_ERR_CAPACITY, "%s must grow to %zu bytes during stream capture", what, bytes);
  if (*p) CK(cudaFreeAsync(*p, s));
  *p = nullptr;
  *cap = 0;
  g_grow_epoch.fetch_add(1);
  if (injected_alloc_failure() || cudaMallocAsync(p, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(DFLASH_ERR_OOM, "allocation of %zu bytes for %s failed", bytes, what);
  }
  *cap = bytes;
  return DFLASH_OK;
}

int ensure_ws(dflash_ctx* c, size_t elems, cudaStream_t s) {
  if (c->no_grow && elems * sizeof(float) > c->ws_cap)
    return fail(DFLASH_ERR_CAPACITY, "GEMM workspace of %zu bytes not yet allocated (have %zu); run one "
                "dflash_draft_block with this K first", elems * sizeof(float), c->ws_cap);
  void* p = c->ws;
  int r = grow_buffer(&p, &c->ws_cap, elems * sizeof(float), s, "GEMM workspace");
  c->ws = reinterpret_cast<float*>(p);
  return r;
}

int trace_begin(dflash_ctx* c, int kind, double bytes, cudaStream_t s) {
  if (c->n_pairs <= 0) return -1;
  const int i = c->next_pair;
  c->next_pair = (c->next_pair + 1) % c->n_pairs;
  // cudaEventRecordExternal: under stream capture the record becomes a graph
  // node that fires on every replay (a plain record only orders the capture).
  if (cudaEventRecordWithFlags(c->ev[2 * i], s, cudaEventRecordExternal) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if ((int)c->trace.size() >= c->n_pairs) c->trace.erase(c->trace.begin());
  c->trace.push_back({kind, i, bytes});
  return i;
}
void trace_end(dflash_ctx* c, int i, cudaStream_t s) {
  if (i >= 0 && cudaEventRecordWithFlags(c->ev[2 * i + 1], s, cudaEventRecordExternal) != cudaSuccess)
    cudaGetLastError();
}

// tensor-memory columns of an accumulator of n columns (allocation granularity)
uint32_t tmem_cols_for_host(int n) { return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u; }

// cached token tensor map: bf16 [planes][M][K], box BN x 64, 128-byte swizzle
int get_xmap(dflash_ctx* c, const void* x, int K, int M, int BN, int planes, const CUtensorMap** out) {
  auto key = std::make_tuple(x, K, M, BN * 4 + planes);
  auto it = c->xmaps.find(key);
  if (it == c->xmaps.end()) {
    CUtensorMap tm;
    RET(tmap_tokens(&tm, x, (uint64_t)K, (uint64_t)M, planes, (uint32_t)BN));
    if (c->xmaps.size() > 4096) c->xmaps.clear();
    it = c->xmaps.emplace(key, tm).first;
  }
  *out = &it->second;
  return DFLASH_OK;
}

// Fused-GEMM options: which epilogue the CTAs of each tile apply and the
// folded RMSNorm on either side (see TcGemmParams).
struct GemmOp {
  int epi = EPI_PARTIAL;
  int x_planes = 2;               // token operand: split bf16 (2 planes) or plain bf16 (1)
  bool op16 = false;              // one fp16 plane against the fp16 weight copies (segs point there)
  bool force_split = false;       // split even when M > 128 (several narrower token tiles)
  const float* ss_in = nullptr;   // folded RMSNorm of the token operand (null: none)
  int n_ss = 0, ss_ld = 0;
  void* xn_out = nullptr;         // residual epilogues: bf16 rows * xn_gain for the next norm
  const void* xn_gain = nullptr;
  float* logits = nullptr;
  int32_t* ids = nullptr;
  float* h = nullptr;
  float* ss_out = nullptr;
  void* q_out = nullptr;
  void* a_out = nullptr;
  int layer = 0, R = 0;
  const int32_t* rows = nullptr;
  int rows_max = 0, t0 = 0;
  int* splits_out = nullptr;      // EPI_PARTIAL: receives the number of K splits in ws
  bool trace = true;              // false: the caller traces this launch with what follows it
  bool late_trigger = false;      // release the dependent launch only after the dependency wait
  // EPI_QKV: the pending context rows u of an append ride along as token tile 1
  // (split bf16 [2][ctx_m][K], folded-norm sums ctx_ss [n_ss][ctx_m]; rows /
  // rows_max as for EPI_CTXKV): their K/V are written with the block's
  const void* ctx_x = nullptr;
  int ctx_m = 0;
  const float* ctx_ss = nullptr;
};
// Launch shape of one tensor-core GEMM: token planes and tiles, weight tiles,
// stage ring, K splits.
struct GemmPlan {
  int N, nkb, XP, BN, t_tiles, tt, t_groups, n_tiles, stages, splits, kps;
  int resident;   // CTAs per SM at this shared-memory size (0: the kernel cannot run)
  bool direct;    // one split: the epilogue reads the CTA's accumulator (no ws partials, no counters)
  bool wpair;     // EPI_SILU, direct: a CTA computes a gate tile and its up tile (n_tiles = pairs)
};
GemmPlan plan_gemm(const dflash_ctx* c, int M, int K, const SegRef* segs, int nseg, const GemmOp& op) {
  GemmPlan g;
  g.N = 0;
  for (int i = 0; i < nseg; ++i) g.N += segs[i].rows;
  g.nkb = K / kTileK;
  // split token operands only while both planes fit one MMA (2 * BN <= 256); the
  // hi plane alone is the plain bf16 operand
  g.XP = (!op.op16 && op.x_planes == 2 && c->split_ops && (M <= 128 || op.force_split)) ? 2 : 1;
  const int bn_max = (g.XP == 1 ? c->gemm_bn_max : 256) / g.XP;   // MMA N = XP * BN <= 256
  g.t_tiles = (M + bn_max - 1) / bn_max;
  // token rows per tile: the MMA's N = XP * BN must be a multiple of 16, so a
  // split operand (two planes) rounds BN to 8 rows and a plain one to 16
  const int align = (g.XP == 2 && c->bn8) ? 8 : 16;
  g.BN = std::max(align, ((M + g.t_tiles - 1) / g.t_tiles + align - 1) / align * align);
  g.n_tiles = 0;
  for (int i = 0; i < nseg; ++i) g.n_tiles += (segs[i].rows + kTileRows - 1) / kTileRows;
  // two token tiles of a split operand per CTA: each weight box is staged once
  // for both (one MMA per tile), instead of once per token tile
  // (a plain operand only for the partial store, whose epilogue has no per-token
  // scratch: TT * BN may reach 512 there)
  g.tt = ((g.XP == 2 || op.epi == EPI_PARTIAL) && g.t_tiles >= 2 && op.epi != EPI_ARGMAX &&
          c->gemm_pairs)
             ? 2
             : 1;
  if (op.ctx_x != nullptr) {   // block rows as tile 0, the append's context rows as tile 1
    g.XP = 2;
    g.t_tiles = 2;
    g.tt = 2;
    g.BN = std::max(8, (std::max(M, op.ctx_m) + 7) / 8 * 8);
  }
  g.t_groups = (g.t_tiles + g.tt - 1) / g.tt;
  const int stage_bytes = kTileRows * kTileK * 2 + g.tt * g.XP * g.BN * kTileK * 2;
  // two CTAs per SM (one's epilogue overlaps the other's weight stream) with 4+
  // stages of narrow token tiles in 100 KB each, or 3 stages of tiles up to 160
  // columns in 110 KB each (measured faster than one CTA with 6 stages); one
  // CTA with a deep ring otherwise
  // The LM head's narrow partial-store tiles (1187 weight tiles at the
  // Qwen3-4B shape) stream best four CTAs to an SM with two stages each: a
  // CTA's turnover then stalls a quarter of the SM's loads in flight instead
  // of half (17 rows: 125.2 -> 121.1 us; the projections measured slower so).
  const int n_cols = g.tt * g.XP * g.BN;
  int ctas_per_sm = c->gemm_ctas > 0                             ? c->gemm_ctas
                    : op.epi == EPI_PARTIAL && n_cols <= 64       ? 4
                    : n_cols <= 64                                ? 2
                    : (op.ctx_x != nullptr && 4 * g.BN <= 128)      ? 2
                    : 3 * stage_bytes <= (110 << 10) - 4096       ? 2
                                                                  : 1;
  const int budget_kb = ctas_per_sm == 4   ? 54
                        : ctas_per_sm == 2 ? (n_cols <= 64 || op.ctx_x != nullptr ? 100 : 110)
                                           : 212;
  const int budget = (c->gemm_smem_kb > 0 ? c->gemm_smem_kb : budget_kb) * 1024;
  g.stages = std::max(2, std::min(8, budget / stage_bytes));
  // the split CTAs of a tile wait for each other in the epilogue, so a split
  // grid must be resident at once: size it by the occupancy actually reached
  const int resident = gemm_tc_resident_ctas(g.tt, false, gemm_tc_smem_bytes(g.BN, g.stages, g.XP, g.tt), n_cols,
                                             c->gemm_by_epi ? op.epi : -1);
  g.resident = resident;
  ctas_per_sm = std::max(1, std::min(ctas_per_sm, resident));
  const int base = g.n_tiles * g.t_groups;
  const int want = ctas_per_sm * c->num_sms;
  g.splits = 1;
  // split K so the grid fills the GPU in one wave (at least 2 k-blocks per split);
  // the tile's CTAs meet in the epilogue, so a split grid must fit one wave
  if (base < want && op.epi != EPI_ARGMAX) g.splits = std::max(1, std::min(want / base, std::max(1, g.nkb / 2)));
  g.kps = (g.nkb + g.splits - 1) / g.splits;
  g.splits = (g.nkb + g.kps - 1) / g.kps;
  // a tile of one split owns its whole sum: the epilogue reads it from tensor
  // memory instead of a round trip of fp32 partials through L2 and a counter
  g.direct = false;
  g.wpair = false;
  if (c->gemm_direct && g.splits == 1 && op.epi != EPI_PARTIAL && op.ctx_x == nullptr) {
    if (op.epi != EPI_SILU) {
      g.direct = true;
      g.resident = gemm_tc_resident_ctas(g.tt, true, gemm_tc_smem_bytes(g.BN, g.stages, g.XP, g.tt), n_cols);
    } else if (g.n_tiles % 2 == 0 && 2 * g.XP * g.BN <= 512) {
      // SwiGLU needs the gate and up sums of a token together: one CTA takes
      // both tiles of a pair (two weight boxes per stage, one token tile), when
      // the pairs alone still fill the GPU without splitting K
      const int pcols = 2 * g.XP * g.BN;
      const int pstage = 2 * kTileRows * kTileK * 2 + g.XP * g.BN * kTileK * 2;
      const int pc = c->gemm_ctas > 0 ? c->gemm_ctas : 3 * pstage <= (110 << 10) - 4096 ? 2 : 1;
      const int pbudget = (c->gemm_smem_kb > 0 ? c->gemm_smem_kb : (pc == 2 ? 110 : 212)) * 1024;
      const int pst = std::max(2, std::min(8, pbudget / pstage));
      const int pres = gemm_tc_resident_ctas(1, true, gemm_tc_smem_bytes(g.BN, pst, g.XP, 1, 2), pcols);
      if (pres >= 1 && (g.n_tiles / 2) * g.t_tiles >= c->num_sms * std::min(pc, pres)) {
        g.wpair = true;
        g.direct = true;
        g.tt = 1;
        g.t_groups = g.t_tiles;
        g.stages = pst;
        g.resident = pres;
        g.n_tiles /= 2;
        // (on the persistent instance the pairs would need 128-row token tiles,
        // two accumulators of gate + up columns in 512 TMEM columns: measured
        // slower than one 192-row tile per CTA, 116.6 vs 112.5 us at the
        // serving batch)
      }
    }
  }
  return g;
}

// Tensor-core GEMM Y = X W^T over concatenated weight segments, M tokens, with
// the epilogue of `op`.  x: bf16 [M, K] tokens for x_mode 0 (ignored otherwise).
int run_gemm_tc(dflash_ctx* c, const void* x, int M, int K, const SegRef* segs, int nseg, const GemmOp& op,
                cudaStream_t s) {
  const GemmPlan pl = plan_gemm(c, M, K, segs, nseg, op);
  const int N = pl.N, nkb = pl.nkb, XP = pl.XP, BN = pl.BN, t_tiles = pl.t_groups, n_tiles = pl.n_tiles;
  const int stages = pl.stages, kps = pl.kps, splits = pl.splits;
  if (pl.resident < 1) return fail(DFLASH_ERR_CUDA, "GEMM of %d shared-memory stages does not fit an SM", stages);
  const bool fuse = op.ctx_x != nullptr;
  if (fuse && (op.epi != EPI_QKV || M > 128 || op.ctx_m > 128 || op.ctx_m < 1))
    return fail(DFLASH_ERR_UNSUPPORTED, "context rows ride only along a QKV GEMM of <= 128 rows");
  const int M_blk = M;
  if (fuse) M = 2 * BN;   // virtual tokens: block tile, then context tile
  if (op.epi != EPI_ARGMAX && !pl.direct) RET(ensure_ws(c, (size_t)splits * M * N, s));
  if (op.splits_out) *op.splits_out = splits;
  if (2 * (size_t)n_tiles * t_tiles >= kCounters) return fail(DFLASH_ERR_UNSUPPORTED, "too many GEMM tiles");
  TcGemmParams p;
  memset(&p, 0, sizeof(p));
  int tiles = 0, cols = 0;
  for (int i = 0; i < nseg; ++i) {
    p.tm_w[i] = *segs[i].tm;
    p.seg_rows[i] = segs[i].rows;
    p.seg_tile0[i] = tiles;
    p.seg_col0[i] = cols;
    tiles += (segs[i].rows + kTileRows - 1) / kTileRows;
    cols += segs[i].rows;
  }
  p.seg_tile0[nseg] = tiles;
  p.seg_col0[nseg] = cols;
  {
    const CUtensorMap* xm = nullptr;
    RET(get_xmap(c, x, K, M_blk, BN, XP, &xm));
    p.tm_x = *xm;
    if (fuse) {
      RET(get_xmap(c, op.ctx_x, K, op.ctx_m, BN, XP, &xm));
      p.tm_x2 = *xm;
      p.fuse_ctx = 1;
      p.m_blk = M_blk;
      p.m_ctx = op.ctx_m;
      p.ss_ctx = op.ctx_ss;
      p.ss_ctx_ld = op.ctx_m;
    }
  }
  p.x_planes = XP;
  p.op16 = op.op16 ? 1 : 0;
  p.tt = pl.tt;
  p.direct = pl.direct ? 1 : 0;
  p.wpair = pl.wpair ? 1 : 0;
  p.nseg = nseg;
  p.N = N;
  p.M = M;
  p.BN = BN;
  p.stages = stages;
  p.kb_per_split = kps;
  p.nkb = nkb;
  p.splits = splits;
  p.ws = c->ws;
  p.flags = c->d_flags;
  p.ss_in = op.ss_in;
  p.n_ss = op.n_ss;
  p.ss_ld = op.ss_ld;
  p.xn_out = reinterpret_cast<__nv_bfloat16*>(op.xn_out);
  p.xn_gain = reinterpret_cast<const __nv_bfloat16*>(op.xn_gain);
  p.eps = c->cfg.rms_eps;
  p.epi = op.epi;
  p.late_trigger = op.late_trigger ? 1 : 0;
  p.counters = c->d_counters;
  p.argmax_keys = c->d_keys;
  p.logits = op.logits;
  p.ids = op.ids;
  p.h = op.h;
  p.ss_out = op.ss_out;
  p.q_out = reinterpret_cast<__nv_bfloat16*>(op.q_out);
  p.a_out = reinterpret_cast<__nv_bfloat16*>(op.a_out);
  p.st = c->st;
  p.kv = c->kv;
  p.rope_turns = c->d_rope;
  p.layer = op.layer;
  p.R = op.R;
  p.rows = op.rows;
  p.rows_max = op.rows_max;
  p.t0 = op.t0;
  p.half_tiles = nseg > 0 ? (segs[0].rows + kTileRows - 1) / kTileRows : 1;
  p.interleave2 = op.epi == EPI_SILU ? 1 : 0;
  if (op.epi == EPI_SILU && (nseg != 2 || segs[0].rows != segs[1].rows || segs[0].rows % kTileRows))
    return fail(DFLASH_ERR_UNSUPPORTED, "SwiGLU epilogue needs two equal segments of whole tiles");
  const double out_bytes = op.epi == EPI_ARGMAX ? (op.logits ? 4.0 * M * N : 8.0 * M) : 4.0 * M * N;
  const int tr = op.trace ? trace_begin(c, DFLASH_TRACE_GEMM, 2.0 * ((double)N * K + (double)M * K) + out_bytes, s)
                         : -1;
  // more one-split tiles than SMs: the persistent instance, one CTA per SM
  // with two accumulators, so that each tile's epilogue runs under the next
  // tile's mainloop (plain operands, one token tile per CTA)
  const int wb = pl.wpair ? 2 : 1;
  const bool persist = c->gemm_persist && pl.direct && XP == 1 && pl.tt == 1 && !fuse &&
                       (op.epi == EPI_QKV || op.epi == EPI_CTXKV || op.epi == EPI_RESID || op.epi == EPI_Y_SS ||
                        (op.epi == EPI_SILU && pl.wpair)) &&
                       (int64_t)n_tiles * t_tiles > c->num_sms && 2 * tmem_cols_for_host(BN * wb) <= 512;
  if (persist) {
    const size_t fixed = gemm_tc_persist_smem_bytes(BN, 0, wb);
    const size_t stage = (size_t)wb * kTileRows * kTileK * 2 + (size_t)BN * kTileK * 2;
    p.stages = (int)std::min<size_t>(8, ((size_t)227 * 1024 - fixed) / (stage + 16));
    p.p_tiles = n_tiles * t_tiles;
    p.p_ttiles = t_tiles;
  }
  if (persist && p.stages >= 2) {
    CK(launch_gemm_tc_persist(p, std::min(c->num_sms, p.p_tiles), s));
  } else {
    p.stages = stages;
    CK(launch_gemm_tc(p, n_tiles, splits, t_tiles, stages, s, c->gemm_by_epi));
  }
  trace_end(c, tr, s);
  c->launches += 1;
  return DFLASH_OK;
}

// fp32 (CUDA-core) GEMM: Y[t][n] for t < M over the concatenated segments;
// partials land in c->ws as [splits][M][N].  Returns the split count.
int run_gemm(dflash_ctx* c, const void* x, int M, int K, const SegRef* segs, int nseg, int* splits_out,
             cudaStream_t s) {
  int N = 0;
  for (int i = 0; i < nseg; ++i) N += segs[i].rows;
  if (c->bf16) {
    return fail(DFLASH_ERR_UNSUPPORTED, "bf16 projections run through run_gemm_tc");
  } else {
    const int n_tiles = (N + 63) / 64, t_tiles = (M + 31) / 32;
    const int base = n_tiles * t_tiles;
    const int ksteps = (K + 31) / 32;
    int splits = 1;
    if (base < 2 * c->num_sms) splits = std::min((2 * c->num_sms + base - 1) / base, std::max(1, ksteps / 2));
    const int kps_steps = (ksteps + splits - 1) / splits;
    splits = (ksteps + kps_steps - 1) / kps_steps;
    RET(ensure_ws(c, (size_t)splits * M * N, s));
    GemmSegs g;
    g.n = nseg;
    for (int i = 0; i < nseg; ++i) {
      g.w[i] = segs[i].w;
      g.rows[i] = segs[i].rows;
    }
    const int tr = trace_begin(c, DFLASH_TRACE_GEMM, 4.0 * ((double)N * K + (double)M * K + (double)M * N), s);
    CK(launch_gemm_simt<float>(reinterpret_cast<const float*>(x), K, M, K, g, N, c->ws, splits, kps_steps * 32, s));
    trace_end(c, tr, s);
    c->launches += 1;
    *splits_out = splits;
  }
  return DFLASH_OK;
}

// Upper bound of the context keys sequence b's block attends to (0 without
// K/V injection: the block sees itself only).
int64_t ctx_keys_ub(const dflash_ctx* c, int b) {
  return c->cond == DFLASH_COND_KV ? std::min<int64_t>(c->ub_kv[b], c->cap[b]) : 0;
}

// Capacity of sequence b must cover `need` slots (power of two, >= 64).
int ensure_capacity(dflash_ctx* c, int b, int64_t need, cudaStream_t s) {
  if (need <= c->cap[b]) return DFLASH_OK;
  if (is_capturing(s))
    return fail(DFLASH_ERR_CAPACITY,
                "sequence %d needs %lld KV slots (capacity %lld) while the stream is captured; call dflash_reserve first",
                b, (long long)need, (long long)c->cap[b]);
  const int64_t new_cap = std::max<int64_t>(64, next_pow2(need));
  if (new_cap > (int64_t)1 << 30) return fail(DFLASH_ERR_INVALID, "capacity %lld too large", (long long)new_cap);
  const int64_t off = c->buddy.alloc(new_cap);
  if (off < 0)
    return fail(DFLASH_ERR_OOM, "KV arena full: %lld slots for sequence %d (pool %lld slots)", (long long)new_cap, b,
                (long long)c->buddy.pool());
  if (c->cap[b] > 0) {
    launch_arena_copy(c->arena, c->esz, c->d, c->seg_tok[b] * c->rows_per_token, off * c->rows_per_token,
                      (int)c->cap[b], (int)new_cap, (int)c->rows_per_token, (int)c->cap[b], s);
    CK(cudaGetLastError());
    c->launches += 1;
    c->buddy.release(c->seg_tok[b], c->cap[b]);
  }
  c->seg_tok[b] = off;
  c->cap[b] = new_cap;
  launch_set_seq(c->st, b, off * c->rows_per_token, (int)new_cap, s);
  CK(cudaGetLastError());
  c->launches += 1;
  return DFLASH_OK;
}

// Host or device int32 input of n values -> a device pointer (staged in dst).
int stage_i32(const int32_t* src, int32_t* dst, size_t n, cudaStream_t s, const int32_t** out) {
  if (is_device_ptr(src)) {
    *out = src;
    return DFLASH_OK;
  }
  if (is_capturing(s)) return fail(DFLASH_ERR_INVALID, "host input while the stream is captured");
  CK(cudaMemcpyAsync(dst, src, n * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  *out = dst;
  return DFLASH_OK;
}

int copy_out(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (dst == nullptr || bytes == 0) return DFLASH_OK;
  const bool dev = is_device_ptr(dst);
  if (!dev && is_capturing(s) && !is_pinned_host(dst))
    return fail(DFLASH_ERR_INVALID, "pageable host output while the stream is captured");
  CK(cudaMemcpyAsync(dst, src, bytes, dev ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, s));
  return DFLASH_OK;
}

// Split-KV workspace of n rows of 128 outputs + 1 log-sum-exp, with room for
// twice the splits: the split count follows the host's upper bound of the
// context, which grows between an eager call and a capture.
// With a caller-provided split-KV scratch (the no-allocation draft), the most
// KV splits whose partials fit it: `per_split` rows of 128 outputs + 1
// log-sum-exp each.  One split needs no scratch at all (the attention writes
// its output directly), so a draft never fails for want of scratch; it only
// runs with fewer, longer splits.
int clamp_splits_to_scratch(const dflash_ctx* c, int n_splits, size_t per_split) {
  if (c->attn_scratch_ext == nullptr || n_splits <= 1) return n_splits;
  const size_t fit = c->attn_scratch_ext_floats / (per_split * 129);
  return (int)std::max<size_t>(1, std::min<size_t>((size_t)n_splits, fit));
}

int attn_workspace(dflash_ctx* c, size_t n, float** part_o, float** part_lse, cudaStream_t s) {
  if (c->attn_scratch_ext != nullptr) {
    if (n * 129 > c->attn_scratch_ext_floats)
      return fail(DFLASH_ERR_CAPACITY, "split-KV scratch of %zu bytes exceeds the %zu-byte static array",
                  n * 129 * sizeof(float), c->attn_scratch_ext_floats * sizeof(float));
    *part_o = c->attn_scratch_ext;
  } else {
    size_t want = n * 129 * sizeof(float);
    if (want > c->attn_ws_cap) want = std::max(2 * want, 2 * c->attn_ws_cap);
    RET(grow_buffer(&c->attn_ws, &c->attn_ws_cap, want, s, "attention workspace"));
    *part_o = reinterpret_cast<float*>(c->attn_ws);
  }
  *part_lse = *part_o + n * 128;
  return DFLASH_OK;
}

// Does run_attention take the tcgen05 kernel?
bool attention_on_umma(const dflash_ctx* c) {
  const dflash_config& g = c->cfg;
  return c->bf16 && c->d == 128 && (c->attn_umma || c->target) && 128 % (g.n_q_heads / g.n_kv_heads) == 0;
}

// Work items of the persistent attention per SM: enough for the longest-first
// order to even out the SMs' loads, few enough that each item streams several
// tiles.
constexpr int kAttnItemsPerSm = 1;
// Batches from this size take the persistent attention; smaller ones one CTA
// per (split, head, sequence) in longest-first order.
constexpr int kAttnPersistentMinBatch = 16;

// The attention schedule of a batch's draft with R block rows per sequence:
// the host's upper bounds of the contexts give the tiles per split (chunk),
// the partial groups to provide and the grid; the device plans with the live
// lengths (launch_attn_plan) once, for every layer.
int plan_attention(dflash_ctx* c, int R, cudaStream_t s) {
  const dflash_config& g = c->cfg;
  const int G = g.n_q_heads / g.n_kv_heads;
  const int n_qtiles = (R + 128 / G - 1) / (128 / G);
  const int rows_pad = n_qtiles * 128;
  const int64_t n_hq = (int64_t)g.n_kv_heads * n_qtiles;
  int64_t tiles_total = 0;
  for (int b = 0; b < c->B; ++b) tiles_total += (ctx_keys_ub(c, b) + R + 63) / 64;
  const int64_t items = (int64_t)kAttnItemsPerSm * c->num_sms;
  const int chunk = (int)std::max<int64_t>(2, (tiles_total * n_hq + items - 1) / items);
  const int s_max = 64;
  int64_t groups_ub = 0, units_ub = 0;
  int s_ub = 1;
  for (int b = 0; b < c->B; ++b) {
    const int64_t tb = (ctx_keys_ub(c, b) + R + 63) / 64;
    const int sb = (int)std::min<int64_t>(s_max, std::max<int64_t>(1, (tb + chunk - 1) / chunk));
    units_ub += sb;
    if (sb > 1) groups_ub += sb;
    s_ub = std::max(s_ub, sb);
  }
  const size_t group_floats = (size_t)g.n_kv_heads * rows_pad * 129;
  int64_t max_groups = 0;   // 0: every sequence in one split, no partials and no merge
  if (groups_ub > 0) {
    if (c->attn_scratch_ext != nullptr) {
      max_groups = (int64_t)(c->attn_scratch_ext_floats / group_floats);
      if (max_groups < 2) max_groups = 0;
    } else {
      max_groups = 2 * groups_ub;   // room for the contexts to grow under a recorded draft
    }
  }
  c->plan_groups = (int)std::min<int64_t>(max_groups, 1 << 30);
  c->plan_smax = max_groups > 0 ? s_ub : 1;
  c->plan_grid = (int)std::max<int64_t>(1, std::min<int64_t>(c->num_sms, units_ub * n_hq));
  c->plan_chunk = chunk;
  launch_attn_plan(c->st, c->B, chunk, s_max, c->plan_groups, c->d_work, c->d_seq_split, c->d_n_units,
                   c->d_seq_order, c->d_attn_ctr, c->nl, s);
  CK(cudaGetLastError());
  c->launches += 1;
  c->plan_mode = c->B >= kAttnPersistentMinBatch ? 2 : 1;
  return DFLASH_OK;
}

// tcgen05 attention (bf16, head_dim 128): query tiles of 128 rows.  With a
// draft's plan (a batch), the persistent kernel works through the planned
// items; otherwise (one sequence, or the target's forward) one CTA per
// (split, head x query tile, sequence) with about one CTA per SM of at least
// two 64-position tiles.  Then the split merge.
int run_attention_umma(dflash_ctx* c, const void* qb, void* ob, int l, int R, cudaStream_t s) {
  const dflash_config& g = c->cfg;
  AttnUParams p;
  memset(&p, 0, sizeof(p));
  p.tm_kv = c->tm_kv;
  p.G = g.n_q_heads / g.n_kv_heads;
  p.JT = 128 / p.G;
  const int M = c->B * R;
  {
    auto key = std::make_tuple(qb, R, M, -1 - p.G);
    auto it = c->xmaps.find(key);
    if (it == c->xmaps.end()) {
      CUtensorMap tm;
      RET(tmap_queries(&tm, qb, g.n_q_heads, (uint64_t)M, p.G, p.JT));
      if (c->xmaps.size() > 4096) c->xmaps.clear();
      it = c->xmaps.emplace(key, tm).first;
    }
    p.tm_q = it->second;
  }
  p.o = reinterpret_cast<__nv_bfloat16*>(ob);
  p.st = c->st;
  p.kv = c->kv;
  p.layer = l;
  p.R = R;
  p.n_q = g.n_q_heads;
  p.n_kv = g.n_kv_heads;
  p.n_qtiles = (R + p.JT - 1) / p.JT;
  p.rows_pad = p.n_qtiles * 128;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->d));
  p.flags = c->d_flags;
  p.o_plane = c->op16_now ? kF16Plane : (size_t)M * c->q_dim;
  p.causal = c->target ? 1 : 0;
  if (c->plan_mode == 2) {
    p.work = c->d_work;
    p.seq_split = c->d_seq_split;
    p.n_units = c->d_n_units;
    p.item_ctr = c->d_attn_ctr + l;
    if (c->plan_groups > 0)
      RET(attn_workspace(c, (size_t)c->plan_groups * p.n_kv * p.rows_pad, &p.part_o, &p.part_lse, s));
    CK(launch_attention_umma(p, c->B, c->plan_grid, s));
    c->launches += 1;
    if (c->plan_groups > 0) {
      CK(launch_attn_merge(p.part_o, p.part_lse, p.n_kv, c->plan_smax, p.G * R, p.rows_pad, R, p.G, p.n_q, p.o,
                           p.o_plane, c->B, s, c->d_flags, c->d_seq_split));
      c->launches += 1;
    }
    return DFLASH_OK;
  }
  int64_t tiles_total = 0;
  int max_tiles = 1;
  for (int b = 0; b < c->B; ++b) {
    const int tb = (int)((ctx_keys_ub(c, b) + R + 63) / 64);
    tiles_total += tb;
    max_tiles = std::max(max_tiles, tb);
  }
  tiles_total *= (int64_t)p.n_kv * p.n_qtiles;
  const int64_t per_cta = std::max<int64_t>(2, (tiles_total + c->num_sms - 1) / c->num_sms);
  p.n_splits = (int)std::max<int64_t>(1, std::min<int64_t>(64, (max_tiles + per_cta - 1) / per_cta));
  p.n_splits = clamp_splits_to_scratch(c, p.n_splits, (size_t)c->B * p.n_kv * p.rows_pad);
  if (c->plan_mode == 1) p.seq_order = c->d_seq_order;   // longest contexts first
  p.early_kv = c->attn_early_now ? 1 : 0;
  if (p.n_splits > 1)
    RET(attn_workspace(c, (size_t)c->B * p.n_kv * p.n_splits * p.rows_pad, &p.part_o, &p.part_lse, s));
  CK(launch_attention_umma(p, c->B, 0, s));
  c->launches += 1;
  if (p.n_splits > 1) {
    CK(launch_attn_merge(p.part_o, p.part_lse, p.n_kv, p.n_splits, p.G * R, p.rows_pad, R, p.G, p.n_q,
                         p.o, p.o_plane, c->B, s, c->d_flags));
    c->launches += 1;
  }
  return DFLASH_OK;
}

// Attention of layer l over [context ; block] for every sequence; q in qb, output in ob.
template <typename T>
int run_attention(dflash_ctx* c, const T* qb, T* ob, int l, int R, cudaStream_t s) {
  const dflash_config& g = c->cfg;
  if (!c->bf16 || c->d != 128) {
    launch_attention<T>(qb, c->st, c->kv, l, c->B, R, g.n_q_heads, g.n_kv_heads, c->d, ob, c->d_flags, s,
                        c->target ? 1 : 0);
    c->launches += 1;
    return DFLASH_OK;
  }
  // (the target's causal mask is in the tcgen05 kernel and the generic one)
  if (attention_on_umma(c)) return run_attention_umma(c, qb, ob, l, R, s);
  AttnTcParams p;
  memset(&p, 0, sizeof(p));
  p.tm_kv = c->tm_kv;
  p.q = reinterpret_cast<const __nv_bfloat16*>(qb);
  p.o = reinterpret_cast<__nv_bfloat16*>(ob);
  p.st = c->st;
  p.kv = c->kv;
  p.layer = l;
  p.R = R;
  p.n_q = g.n_q_heads;
  p.n_kv = g.n_kv_heads;
  p.G = g.n_q_heads / g.n_kv_heads;
  p.rows = p.G * R;
  const int nw = std::min(8, (p.rows + 15) / 16);
  p.n_qtiles = (p.rows + 16 * nw - 1) / (16 * nw);
  p.rows_pad = p.n_qtiles * nw * 16;
  // KV splits: about two CTAs of >= 2 tiles per SM over the whole batch (host
  // upper bounds of the context; the kernel balances on the live length)
  int64_t tiles_total = 0;
  int max_tiles = 1;
  for (int b = 0; b < c->B; ++b) {
    const int tb = (int)((ctx_keys_ub(c, b) + R + 63) / 64);
    tiles_total += tb;
    max_tiles = std::max(max_tiles, tb);
  }
  tiles_total *= (int64_t)p.n_kv * p.n_qtiles;
  const int64_t per_cta = std::max<int64_t>(2, (tiles_total + 2 * c->num_sms - 1) / (2 * c->num_sms));
  p.n_splits = (int)std::max<int64_t>(1, std::min<int64_t>(64, (max_tiles + per_cta - 1) / per_cta));
  p.n_splits = clamp_splits_to_scratch(c, p.n_splits, (size_t)c->B * p.n_kv * p.rows_pad);
  if (p.n_splits > 1) {
    const size_t n = (size_t)c->B * p.n_kv * p.n_splits * p.rows_pad;
    if (c->attn_scratch_ext != nullptr) {
      if (n * 129 > c->attn_scratch_ext_floats)
        return fail(DFLASH_ERR_CAPACITY, "split-KV scratch of %zu bytes exceeds the %zu-byte static array",
                    n * 129 * sizeof(float), c->attn_scratch_ext_floats * sizeof(float));
      p.part_o = c->attn_scratch_ext;
    } else {
      // room for twice the splits: the split count follows the host's upper
      // bound of the context, which grows between an eager call and a capture
      size_t want = n * 129 * sizeof(float);
      if (want > c->attn_ws_cap) want = std::max(2 * want, 2 * c->attn_ws_cap);
      RET(grow_buffer(&c->attn_ws, &c->attn_ws_cap, want, s, "attention workspace"));
      p.part_o = reinterpret_cast<float*>(c->attn_ws);
    }
    p.part_lse = p.part_o + n * 128;
  }
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->d));
  p.flags = c->d_flags;
  p.o_plane = c->op16_now ? kF16Plane : (size_t)c->B * R * c->q_dim;
  CK(launch_attention_tc(p, nw, c->B, s));
  c->launches += p.n_splits > 1 ? 2 : 1;
  return DFLASH_OK;
}

template <typename T>
int draft_impl(dflash_ctx* c, const int32_t* anchor_dev, int K, float* logits_dev, cudaStream_t s) {
  const int B = c->B, R = K + 1, M = B * R, H = c->H;
  const dflash_config& g = c->cfg;
  T* xn = reinterpret_cast<T*>(c->xn);
  T* qb = reinterpret_cast<T*>(c->qb);
  T* ob = reinterpret_cast<T*>(c->ob);
  T* ab = reinterpret_cast<T*>(c->ab);
  T* xf = reinterpret_cast<T*>(c->xf);
  launch_embed_norm<T>(reinterpret_cast<const T*>(c->w.embed), anchor_dev, c->st, B, R, H, c->V, g.mask_token_id,
                       reinterpret_cast<const T*>(c->w.layers[0].attn_norm), g.rms_eps, c->h, xn, 0, c->d_flags,
                       c->kseq_dev, s);
  int splits = 1;
  for (int l = 0; l < c->nl; ++l) {
    const dflash_layer_weights& lw = c->w.layers[l];
    const auto* lm = c->bf16 ? &c->lmaps[l] : nullptr;
    SegRef qkv[3] = {{lw.wq, c->q_dim, lm ? &lm->wq : nullptr},
                     {lw.wk, c->kv_dim, lm ? &lm->wk : nullptr},
                     {lw.wv, c->kv_dim, lm ? &lm->wv : nullptr}};
    RET(run_gemm(c, xn, M, H, qkv, 3, &splits, s));
    launch_epi_qkv<T>(c->ws, splits, M, R, l, g.n_q_heads, g.n_kv_heads, c->d, c->d_rope, c->st, c->kv, qb,
                      c->d_flags, s);
    RET(run_attention<T>(c, qb, ob, l, R, s));
    SegRef wo[1] = {{lw.wo, H, lm ? &lm->wo : nullptr}};
    RET(run_gemm(c, ob, M, c->q_dim, wo, 1, &splits, s));
    launch_epi_residual_norm<T>(c->ws, splits, M, H, c->h, reinterpret_cast<const T*>(lw.mlp_norm), g.rms_eps, xn, R,
                                0, s);
    SegRef gu[2] = {{lw.w_gate, c->I, lm ? &lm->wg : nullptr}, {lw.w_up, c->I, lm ? &lm->wu : nullptr}};
    RET(run_gemm(c, xn, M, H, gu, 2, &splits, s));
    launch_epi_silu<T>(c->ws, splits, M, c->I, ab, s);
    SegRef wd[1] = {{lw.w_down, H, lm ? &lm->wd : nullptr}};
    RET(run_gemm(c, ab, M, c->I, wd, 1, &splits, s));
    // residual, then the next layer's attention norm (or the final norm of the mask rows)
    if (l + 1 < c->nl)
      launch_epi_residual_norm<T>(c->ws, splits, M, H, c->h,
                                  reinterpret_cast<const T*>(c->w.layers[l + 1].attn_norm), g.rms_eps, xn, R, 0, s);
    else
      launch_epi_residual_norm<T>(c->ws, splits, M, H, c->h, reinterpret_cast<const T*>(c->w.final_norm), g.rms_eps,
                                  xf, R, K, s);
  }
  SegRef lmh[1] = {{c->w.lm_head, c->V, nullptr}};
  RET(run_gemm(c, xf, B * K, H, lmh, 1, &splits, s));
  launch_argmax(c->ws, splits, B * K, c->V, c->d_draft, s);
  CK(cudaGetLastError());
  c->launches += 1 + 4 * (int64_t)c->nl + 1;  // non-GEMM, non-attention kernels of the draft
  return DFLASH_OK;
}


int lm_head_bf16(dflash_ctx* c, int K, float* logits_dev, cudaStream_t s, bool op16 = false);

// The fp16 weight copies, made once (see dflash_ctx::w16); false, and the
// draft keeps split bf16 operands, inside a stream capture, without the memory
// or when a weight lies outside fp16's range.  The weights must not change
// after the copy.
bool ensure_w16(dflash_ctx* c, cudaStream_t s) {
  if (c->w16) return true;
  if (c->w16_failed || c->no_grow || is_capturing(s)) return false;   // (a no-allocation draft keeps split operands)
  const size_t H = c->H;
  const size_t sz[7] = {H * c->q_dim, H * c->kv_dim, H * c->kv_dim, (size_t)c->q_dim * H,
                        H * c->I,     H * c->I,      (size_t)c->I * H};
  size_t n = (size_t)c->V * H;
  for (int l = 0; l < c->nl; ++l)
    for (size_t e : sz) n += e;
  const size_t bad_off = (2 * n + 15) & ~(size_t)15;
  char* buf = nullptr;
  if (injected_alloc_failure() || cudaMalloc(&buf, bad_off + 16) != cudaSuccess) {
    cudaGetLastError();
    c->w16_failed = true;
    return false;
  }
  uint32_t* bad = reinterpret_cast<uint32_t*>(buf + bad_off);
  bool ok = cudaMemsetAsync(bad, 0, 4, s) == cudaSuccess;
  size_t off = 0;   // elements; every matrix is a multiple of 128 x 128 of them, so copies stay 16-byte aligned
  auto copy = [&](const void* w, size_t e) -> const void* {
    char* dst = buf + 2 * off;
    off += e;
    if (ok) ok = launch_bf16_to_f16(static_cast<const __nv_bfloat16*>(w), dst, e, bad, s) == cudaSuccess;
    c->launches += 1;
    return dst;
  };
  c->wl16.assign(c->w.layers, c->w.layers + c->nl);
  for (dflash_layer_weights& w : c->wl16) {
    w.wq = copy(w.wq, sz[0]);
    w.wk = copy(w.wk, sz[1]);
    w.wv = copy(w.wv, sz[2]);
    w.wo = copy(w.wo, sz[3]);
    w.w_gate = copy(w.w_gate, sz[4]);
    w.w_up = copy(w.w_up, sz[5]);
    w.w_down = copy(w.w_down, sz[6]);
  }
  c->lm16 = copy(c->w.lm_head, (size_t)c->V * H);
  uint32_t h_bad = 1;
  if (ok)
    ok = cudaMemcpyAsync(&h_bad, bad, 4, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess && h_bad == 0;
  const uint64_t Hb = H * 2;
  c->lmaps16.resize(c->nl);
  int r = ok ? tmap_bf16(&c->tm_lm16, c->lm16, H, c->V, Hb, kTileRows) : DFLASH_ERR_INVALID;
  for (int l = 0; l < c->nl && r == DFLASH_OK; ++l) {   // the same boxes as the bf16 maps (TMA moves 2-byte elements)
    const dflash_layer_weights& lw = c->wl16[l];
    auto& m = c->lmaps16[l];
    r = tmap_bf16(&m.wq, lw.wq, H, c->q_dim, Hb, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wk, lw.wk, H, c->kv_dim, Hb, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wv, lw.wv, H, c->kv_dim, Hb, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wo, lw.wo, c->q_dim, H, (uint64_t)c->q_dim * 2, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wg, lw.w_gate, H, c->I, Hb, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wu, lw.w_up, H, c->I, Hb, kTileRows);
    if (r == DFLASH_OK) r = tmap_bf16(&m.wd, lw.w_down, c->I, H, (uint64_t)c->I * 2, kTileRows);
  }
  if (r != DFLASH_OK) {
    cudaStreamSynchronize(s);
    cudaFree(buf);
    cudaGetLastError();
    g_err.clear();
    c->w16_failed = true;
    return false;
  }
  c->w16 = buf;
  return true;
}
int lm_head_rows(dflash_ctx* c, int M, cudaStream_t s);
int flush_pending(dflash_ctx* c, cudaStream_t s);

// bf16 draft on fused tensor-core GEMMs.  Per layer: QKV (epilogue: RMSNorm
// row scale, RoPE, q, block K/V slots) -> attention -> O (epilogue: residual,
// sums of squares, rows * mlp_norm gain) -> gate/up (epilogue: row scale,
// SwiGLU) -> down (epilogue: residual, sums of squares, rows * the next norm's
// gain); the LM head's epilogue applies the final norm's row scale and takes
// the greedy argmax of the mask rows.
int draft_bf16(dflash_ctx* c, const int32_t* anchor_dev, int K, float* logits_dev, cudaStream_t s) {
  const int B = c->B, R = K + 1, M = B * R, H = c->H;
  const dflash_config& g = c->cfg;
  using bf = __nv_bfloat16;
  bf* xn = reinterpret_cast<bf*>(c->xn);
  // from f16_min_rows GEMM rows the split operands' doubled tensor work and
  // token boxes cost more than they buy: there every token operand is one fp16
  // plane (11 significant bits) against the fp16 weight copies
  const bool op16 = c->f16_ops && !c->target && M >= c->f16_min_rows && c->d == 128 && ensure_w16(c, s);
  c->op16_now = op16;   // read by the attention launches
  struct Op16Scope {
    dflash_ctx* c;
    ~Op16Scope() { c->op16_now = false; }
  } op16_scope{c};
  launch_embed_norm<bf>(reinterpret_cast<const bf*>(c->w.embed), anchor_dev, c->st, B, R, H, c->V, g.mask_token_id,
                        reinterpret_cast<const bf*>(c->w.layers[0].attn_norm), g.rms_eps, c->h, xn,
                        op16 ? kF16Plane : (size_t)M * H, c->d_flags, c->kseq_dev, s,
                        c->trun ? c->trun->tokens : nullptr);
  c->launches += 1;
  struct PlanScope {
    dflash_ctx* c;
    ~PlanScope() { c->plan_mode = 0; }
  } plan_scope{c};
  // a batch's attention: one persistent schedule for every layer
  if (B > 1 && B <= attn_plan_max_batch() && attention_on_umma(c)) RET(plan_attention(c, R, s));
  const int n_ss = H / kTileRows;
  // a pending append's K/V are projected with the layers' QKV when both fit
  // one token tile each, else on their own first
  const bool fuse_ctx = c->pending && M <= 128 && c->pend_m <= 128 && !op16;   // (its rows are split bf16)
  if (c->pending && !fuse_ctx) RET(flush_pending(c, s));
  // per layer: QKV, attention, O, gate/up, down
  struct LayerOps {
    SegRef qkv[3], wo[1], gu[2], wd[1];
    GemmOp oq, oo, og, od;
  };
  auto build = [&](int l, LayerOps& L) {
    const dflash_layer_weights& lw = op16 ? c->wl16[l] : c->w.layers[l];
    const auto& lm = op16 ? c->lmaps16[l] : c->lmaps[l];
    L.qkv[0] = {lw.wq, c->q_dim, &lm.wq};
    L.qkv[1] = {lw.wk, c->kv_dim, &lm.wk};
    L.qkv[2] = {lw.wv, c->kv_dim, &lm.wv};
    L.wo[0] = {lw.wo, H, &lm.wo};
    L.gu[0] = {lw.w_gate, c->I, &lm.wg};
    L.gu[1] = {lw.w_up, c->I, &lm.wu};
    L.wd[0] = {lw.w_down, H, &lm.wd};
    L.oq = GemmOp();
    L.oq.epi = EPI_QKV;
    L.oq.op16 = op16;
    // the drafter's layer inputs keep ~16 bits at any M (its logit error budget
    // needs it); the target's are plain bf16 above one token tile (its logits
    // are the reference, and at large M the split doubles the tensor work)
    L.oq.force_split = !c->target;
    L.oq.x_planes = c->target && c->target_plain ? 1 : 2;
    L.oq.q_out = c->qb;
    L.oq.layer = l;
    L.oq.R = R;
    if (l > 0) {   // layer 0's rows come normalised from the embedding kernel
      L.oq.ss_in = c->d_ss;
      L.oq.n_ss = n_ss;
      L.oq.ss_ld = M;
    }
    if (fuse_ctx) {   // the pending append's rows u ride along: their K/V for layer l
      L.oq.ctx_x = c->ub;
      L.oq.ctx_m = c->pend_m;
      L.oq.ctx_ss = c->d_ss_ctx;
      L.oq.rows = c->d_rows;
      L.oq.rows_max = c->pend_rows_max;
      L.oq.n_ss = n_ss;
    }
    L.oo = GemmOp();
    L.oo.epi = EPI_RESID;
    L.oo.force_split = !c->target;
    L.oo.x_planes = L.oq.x_planes;
    L.oo.op16 = op16;
    L.oo.h = c->h;
    L.oo.ss_out = c->d_ss;
    L.oo.xn_out = xn;
    L.oo.xn_gain = lw.mlp_norm;
    L.og = GemmOp();
    L.og.epi = EPI_SILU;
    L.og.force_split = !c->target;
    L.og.x_planes = L.oq.x_planes;
    L.og.op16 = op16;
    L.og.a_out = c->ab;
    L.og.ss_in = c->d_ss;
    L.og.n_ss = n_ss;
    L.og.ss_ld = M;
    L.od = L.oo;
    L.od.xn_gain = l + 1 < c->nl ? c->w.layers[l + 1].attn_norm : c->w.final_norm;
  };
  // A grid-mode tcgen05 attention loads its first context K/V tiles before its
  // dependency wait: its QKV GEMM then releases it only after its own wait (so
  // every kernel before the GEMM is complete) and must write no K/V below the
  // block rows (no pending append rides along).
  const bool early_kv = c->attn_early && !fuse_ctx && c->plan_mode != 2 && attention_on_umma(c);
  LayerOps L[2];
  build(0, L[0]);
  for (int l = 0; l < c->nl; ++l) {
    LayerOps& cur = L[l & 1];
    LayerOps& nxt = L[(l + 1) & 1];
    if (l + 1 < c->nl) build(l + 1, nxt);
    cur.oq.late_trigger = early_kv;
    RET(run_gemm_tc(c, xn, M, H, cur.qkv, 3, cur.oq, s));
    c->attn_early_now = early_kv;
    const int ra = run_attention<bf>(c, reinterpret_cast<const bf*>(c->qb), reinterpret_cast<bf*>(c->ob), l, R, s);
    c->attn_early_now = false;
    RET(ra);
    RET(run_gemm_tc(c, c->ob, M, c->q_dim, cur.wo, 1, cur.oo, s));
    RET(run_gemm_tc(c, xn, M, H, cur.gu, 2, cur.og, s));
    RET(run_gemm_tc(c, c->ab, M, c->I, cur.wd, 1, cur.od, s));
    if (c->trun && c->trun->feats)   // the target's residual stream after a feature layer
      for (int fi = 0; fi < c->n_feat; ++fi)
        if (c->feat_layers[fi] == l) {
          launch_feat_copy(c->h, M, H, c->n_feat, fi, c->trun->feats, s);
          c->launches += 1;
        }
  }
  c->pending = false;
  return c->trun ? lm_head_rows(c, M, s) : lm_head_bf16(c, K, logits_dev, s, op16);
}

// LM head of a bf16 draft: c->xn holds the last layer's output rows times the
// final norm's gain (split bf16) and d_ss their per-tile sums of squares; the
// mask rows' greedy ids go to d_draft (and their logits to logits_dev).
// The target's LM head: the greedy id (and optionally the logits) of every one
// of the M rows -- partial-store GEMM, then the argmax kernel with R = 0.
int lm_head_rows(dflash_ctx* c, int M, cudaStream_t s) {
  const int H = c->H, n_ss = H / kTileRows;
  SegRef lmh[1] = {{c->w.lm_head, c->V, &c->tm_lm}};
  GemmOp oh;
  oh.epi = EPI_PARTIAL;
  int splits = 1;
  oh.splits_out = &splits;
  oh.trace = false;
  const double lm_bytes = 2.0 * ((double)c->V * H + (double)M * H) + 4.0 * M * (c->trun->logits ? c->V + 1.0 : 1.0);
  const int tr = trace_begin(c, DFLASH_TRACE_GEMM, lm_bytes, s);
  RET(run_gemm_tc(c, c->xn, M, H, lmh, 1, oh, s));
  launch_lm_argmax(c->ws, splits, M, c->V, 0, c->d_ss, n_ss, M, H, c->cfg.rms_eps, c->trun->logits, c->d_keys,
                   c->d_counters + kCounters - 1, c->trun->ids, M, s);
  CK(cudaGetLastError());
  trace_end(c, tr, s);
  c->launches += 1;
  return DFLASH_OK;
}

int lm_head_bf16(dflash_ctx* c, int K, float* logits_dev, cudaStream_t s, bool op16) {
  const int B = c->B, R = K + 1, M = B * R, H = c->H;
  const dflash_config& g = c->cfg;
  const int n_ss = H / kTileRows;
  const void* xn = c->xn;
  // (the fused-argmax GEMM, DFLASH_LM_FUSED=1, measured at 1088 / 1025 / 257
  // rows: 1265 / 1320 / 453 us against 1299 / 1116 / 320 us for this path)
  if (!c->lm_fused) {
    // the LM head streams its weights in a plain partial-store GEMM (raw dot
    // products, fp32; L2-resident at drafting sizes) and a separate kernel
    // applies the final norm's row scale and takes the argmax: faster than any
    // fused epilogue measured (125 + ~6 us vs 148 us for a persistent one-phase
    // program at 17 rows; 963 us for the fused-argmax GEMM at 257 rows, which
    // streams the weights once per token tile)
    SegRef lmh[1] = {{op16 ? c->lm16 : c->w.lm_head, c->V, op16 ? &c->tm_lm16 : &c->tm_lm}};
    GemmOp oh;
    oh.epi = EPI_PARTIAL;
    oh.op16 = op16;
    int splits = 1;
    oh.splits_out = &splits;
    // traced as a GEMM of its own (weights and tokens in, fp32 dot products out)
    RET(run_gemm_tc(c, xn, M, H, lmh, 1, oh, s));
    // its arrival counter is the last one, which no GEMM or attention tile uses
    launch_lm_argmax(c->ws, splits, M, c->V, R, c->d_ss, n_ss, M, H, g.rms_eps, logits_dev, c->d_keys,
                     c->d_counters + kCounters - 1, c->d_draft, B * K, s);
    CK(cudaGetLastError());
    c->launches += 1;
    return DFLASH_OK;
  }
  SegRef lmh[1] = {{op16 ? c->lm16 : c->w.lm_head, c->V, op16 ? &c->tm_lm16 : &c->tm_lm}};
  GemmOp oh;
  oh.epi = EPI_ARGMAX;
  oh.op16 = op16;
  oh.logits = logits_dev;
  oh.ids = c->d_draft;
  oh.R = R;
  oh.ss_in = c->d_ss;
  oh.n_ss = n_ss;
  oh.ss_ld = M;
  RET(run_gemm_tc(c, xn, M, H, lmh, 1, oh, s));
  return DFLASH_OK;
}

// bf16 append: fc (epilogue: sums of squares, rows * fc_norm gain in bf16) ->
// every layer's [W_k; W_v] (epilogue: RMSNorm row scale, RoPE, KV slots), per
// chunk of rows.
// The pending append's K/V projection on its own (every layer's [W_k; W_v]
// over the rows u in ub, their slots from pend_base).
int flush_pending(dflash_ctx* c, cudaStream_t s) {
  if (!c->pending) return DFLASH_OK;
  std::vector<SegRef> kvsegs;
  for (int l = 0; l < c->nl; ++l) {
    kvsegs.push_back({c->w.layers[l].wk, c->kv_dim, &c->lmaps[l].wk});
    kvsegs.push_back({c->w.layers[l].wv, c->kv_dim, &c->lmaps[l].wv});
  }
  GemmOp okv;
  okv.epi = EPI_CTXKV;
  okv.force_split = true;
  okv.rows = c->d_rows;
  okv.rows_max = c->pend_rows_max;
  okv.t0 = 0;
  okv.ss_in = c->d_ss_ctx;
  okv.n_ss = c->H / kTileRows;
  okv.ss_ld = c->pend_m;
  RET(run_gemm_tc(c, c->ub, c->pend_m, c->H, kvsegs.data(), (int)kvsegs.size(), okv, s));
  c->pending = false;
  return DFLASH_OK;
}

int append_bf16(dflash_ctx* c, const void* feats, bool feats_dev, int rows_max, cudaStream_t s) {
  const int B = c->B, F = c->F, H = c->H;
  const int total = B * rows_max;
  const int chunk = std::min(total, (int)c->ss_rows);
  RET(grow_buffer(&c->ub, &c->ub_cap, 2 * (size_t)chunk * H * c->esz, s, "append feature buffer"));   // split bf16
  if (!feats_dev) RET(grow_buffer(&c->stage, &c->stage_cap, (size_t)chunk * F * c->esz, s, "append staging"));
  std::vector<SegRef> kvsegs;
  for (int l = 0; l < c->nl; ++l) {
    kvsegs.push_back({c->w.layers[l].wk, c->kv_dim, &c->lmaps[l].wk});
    kvsegs.push_back({c->w.layers[l].wv, c->kv_dim, &c->lmaps[l].wv});
  }
  SegRef fc[1] = {{c->w.w_fc, H, &c->tm_fc}};
  // commit first (kv_len += rows, pend_base = the first new slot): the K/V
  // epilogue addresses the new rows from pend_base
  launch_append_commit(c->d_rows, c->st, B, s);
  c->launches += 1;
  for (int t0 = 0; t0 < total; t0 += chunk) {
    const int Mc = std::min(chunk, total - t0);
    const char* src = reinterpret_cast<const char*>(feats) + (size_t)t0 * F * c->esz;
    const void* x = src;
    if (!feats_dev) {
      CK(cudaMemcpyAsync(c->stage, src, (size_t)Mc * F * c->esz, cudaMemcpyHostToDevice, s));
      x = c->stage;
    }
    // rows that the next draft's QKV GEMMs can carry leave their K/V pending
    const bool defer = c->fuse_append && total <= 128 && Mc == total && c->cond == DFLASH_COND_KV;
    GemmOp of;
    of.epi = EPI_Y_SS;
    of.x_planes = 1;   // the caller's feature rows
    of.ss_out = defer ? c->d_ss_ctx : c->d_ss;
    of.xn_out = c->ub;
    of.xn_gain = c->w.fc_norm;
    RET(run_gemm_tc(c, x, Mc, F, fc, 1, of, s));
    if (defer) {
      c->pending = true;
      c->pend_m = total;
      c->pend_rows_max = rows_max;
      break;
    }
    GemmOp okv;
    okv.epi = EPI_CTXKV;
    okv.force_split = true;   // the context feature u feeds every layer's K/V: keep its 16 bits at any M
    okv.rows = c->d_rows;
    okv.rows_max = rows_max;
    okv.t0 = t0;
    okv.ss_in = c->d_ss;
    okv.n_ss = H / kTileRows;
    okv.ss_ld = Mc;
    RET(run_gemm_tc(c, c->ub, Mc, H, kvsegs.data(), (int)kvsegs.size(), okv, s));
  }
  CK(cudaGetLastError());
  return DFLASH_OK;
}

// Append without K/V injection (input fusion, or no context): the rows are
// consumed (kv_len += rows, ctx_len follows); with input fusion each
// sequence's last row also leaves its context feature u = RMSNorm(W_fc f) in
// d_ulast, for the next draft's embeddings.  No layer's K/V is computed.
int append_cond(dflash_ctx* c, const void* feats, bool feats_dev, int rows_max, cudaStream_t s) {
  const int B = c->B, F = c->F, H = c->H;
  const float eps = c->cfg.rms_eps;
  const int total = B * rows_max;
  if (c->cond == DFLASH_COND_INPUT) {
    const int chunk = std::min(total, c->bf16 ? (int)c->ss_rows : 4096);
    RET(grow_buffer(&c->ub, &c->ub_cap, (c->bf16 ? 2 : 1) * (size_t)chunk * H * c->esz, s, "append feature buffer"));
    if (!feats_dev) RET(grow_buffer(&c->stage, &c->stage_cap, (size_t)chunk * F * c->esz, s, "append staging"));
    for (int t0 = 0; t0 < total; t0 += chunk) {
      const int Mc = std::min(chunk, total - t0);
      const char* src = reinterpret_cast<const char*>(feats) + (size_t)t0 * F * c->esz;
      const void* x = src;
      if (!feats_dev) {
        CK(cudaMemcpyAsync(c->stage, src, (size_t)Mc * F * c->esz, cudaMemcpyHostToDevice, s));
        x = c->stage;
      }
      if (c->bf16) {   // fc epilogue: split bf16 of y * gain and per-tile sums of squares of y
        using bf = __nv_bfloat16;
        SegRef fc[1] = {{c->w.w_fc, H, &c->tm_fc}};
        GemmOp of;
        of.epi = EPI_Y_SS;
        of.x_planes = 1;
        of.ss_out = c->d_ss;
        of.xn_out = c->ub;
        of.xn_gain = c->w.fc_norm;
        RET(run_gemm_tc(c, x, Mc, F, fc, 1, of, s));
        launch_ulast<bf>(reinterpret_cast<const bf*>(c->ub), (size_t)Mc * H, c->d_ss, H / kTileRows, Mc, t0, Mc,
                         c->d_rows, rows_max, B, H, eps, c->d_ulast, s);
      } else {         // fc, then the normalised rows
        SegRef fc[1] = {{c->w.w_fc, H, nullptr}};
        int splits = 1;
        float* u = reinterpret_cast<float*>(c->ub);
        RET(run_gemm(c, x, Mc, F, fc, 1, &splits, s));
        launch_epi_fcnorm<float>(c->ws, splits, Mc, H, reinterpret_cast<const float*>(c->w.fc_norm), eps, u, s);
        launch_ulast<float>(u, 0, nullptr, 0, 0, t0, Mc, c->d_rows, rows_max, B, H, eps, c->d_ulast, s);
        c->launches += 1;
      }
      c->launches += 1;
    }
  }
  launch_append_commit(c->d_rows, c->st, B, s);
  c->launches += 1;
  CK(cudaGetLastError());
  return DFLASH_OK;
}

template <typename T>
int append_impl(dflash_ctx* c, const void* feats, bool feats_dev, int rows_max, cudaStream_t s) {
  const int B = c->B, F = c->F, H = c->H;
  const dflash_config& g = c->cfg;
  const int total = B * rows_max;
  const int chunk = std::min(total, 4096);
  RET(grow_buffer(&c->ub, &c->ub_cap, (size_t)chunk * H * c->esz, s, "append feature buffer"));
  if (!feats_dev) RET(grow_buffer(&c->stage, &c->stage_cap, (size_t)chunk * F * c->esz, s, "append staging"));
  std::vector<SegRef> kvsegs;
  for (int l = 0; l < c->nl; ++l) {
    const auto* lm = c->bf16 ? &c->lmaps[l] : nullptr;
    kvsegs.push_back({c->w.layers[l].wk, c->kv_dim, lm ? &lm->wk : nullptr});
    kvsegs.push_back({c->w.layers[l].wv, c->kv_dim, lm ? &lm->wv : nullptr});
  }
  SegRef fc[1] = {{c->w.w_fc, H, c->bf16 ? &c->tm_fc : nullptr}};
  T* u = reinterpret_cast<T*>(c->ub);
  int splits = 1;
  for (int t0 = 0; t0 < total; t0 += chunk) {
    const int Mc = std::min(chunk, total - t0);
    const char* src = reinterpret_cast<const char*>(feats) + (size_t)t0 * F * c->esz;
    const void* x = src;
    if (!feats_dev) {
      CK(cudaMemcpyAsync(c->stage, src, (size_t)Mc * F * c->esz, cudaMemcpyHostToDevice, s));
      x = c->stage;
    }
    RET(run_gemm(c, x, Mc, F, fc, 1, &splits, s));
    launch_epi_fcnorm<T>(c->ws, splits, Mc, H, reinterpret_cast<const T*>(c->w.fc_norm), g.rms_eps, u, s);
    RET(run_gemm(c, u, Mc, H, kvsegs.data(), (int)kvsegs.size(), &splits, s));
    launch_epi_ctxkv<T>(c->ws, splits, Mc, t0, rows_max, c->d_rows, c->nl, g.n_kv_heads, c->d, c->d_rope, c->st,
                        c->kv, c->d_flags, s);
  }
  launch_append_commit(c->d_rows, c->st, B, s);
  CK(cudaGetLastError());
  c->launches += 2 * (int64_t)((total + chunk - 1) / chunk) + 1;  // fcnorm + ctxkv per chunk, commit
  return DFLASH_OK;
}

void free_ctx(dflash_ctx* c) {
  cudaDeviceSynchronize();
  if (c->dg.exec) cudaGraphExecDestroy(c->dg.exec);
  if (c->gstream) cudaStreamDestroy(c->gstream);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  void* ptrs[] = {c->d_i32, c->d_kv_base, c->d_flags, c->d_draft, c->d_targets, c->d_rope, c->arena_raw, c->h,
                  c->xn, c->qb, c->ob, c->ab, c->xf, c->ws, c->stage, c->ub, c->attn_ws, c->d_keys,
                  c->d_counters, c->d_ss, c->ybuf, c->d_ss_ctx, c->d_ulast, c->d_plan, c->w16};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  cudaGetLastError();
  delete c;
}

}  // namespace

// dflash_draft_block with the attention's split-KV scratch taken from `scratch`
// and every context workspace frozen at its current size.
int dfl_draft_block_with_scratch(dflash_ctx* c, const int32_t* anchor_ids, int32_t K, int32_t* draft_ids,
                                 float* logits, float* scratch, size_t scratch_floats, void* stream) {
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  c->attn_scratch_ext = scratch;
  c->attn_scratch_ext_floats = scratch_floats;
  c->no_grow = true;
  const int r = dflash_draft_block(c, anchor_ids, K, draft_ids, logits, stream);
  c->attn_scratch_ext = nullptr;
  c->attn_scratch_ext_floats = 0;
  c->no_grow = false;
  return r;
}

int dfl_fail(int code, const char* msg) { return fail(code, "%s", msg); }

struct DraftGraphKey {
  int K;
  const void *anchor, *kseq, *ids, *logits;
};

// Record `body` (the draft just run eagerly, so every workspace it needs
// exists) into a graph for later calls with the same key.  A recording that
// fails leaves drafts eager; the call itself has already succeeded.
template <class Body>
void record_draft(dflash_ctx* c, Body& body, const DraftGraphKey& key) {
  c->dg.valid = false;
  if (c->gstream == nullptr) {
    if (cudaStreamCreateWithFlags(&c->gstream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      c->graph_drafts = false;
      return;
    }
  }
  const int64_t l0 = c->launches;
  const std::string err0 = g_err;
  if (cudaStreamBeginCapture(c->gstream, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaGetLastError();
    c->graph_drafts = false;
    return;
  }
  const int rb = body(c->gstream);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(c->gstream, &g);
  c->dg.launches = c->launches - l0;
  c->launches = l0;   // the capture launched nothing
  g_err = err0;
  cudaGraphExec_t exec = nullptr;
  if (rb != DFLASH_OK || ec != cudaSuccess || g == nullptr || cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    c->graph_drafts = false;
    return;
  }
  cudaGraphDestroy(g);
  if (c->dg.exec) cudaGraphExecDestroy(c->dg.exec);
  c->dg.exec = exec;
  c->dg.K = key.K;
  c->dg.anchor = key.anchor;
  c->dg.kseq = key.kseq;
  c->dg.ids = key.ids;
  c->dg.logits = key.logits;
  c->dg.epoch = g_grow_epoch.load();
  c->dg.valid = true;
}

extern "C" {

const char* dflash_last_error(void) { return g_err.c_str(); }

// A context of the drafter, or (target) of the target model's verify forward,
// which has no fc layer (w_fc, fc_norm unused) and no context K/V GEMM.
static int create_impl(const dflash_config* cfg, const dflash_weights* w, int32_t batch, dflash_ctx** out,
                       bool target) {
  g_err.clear();
  if (!cfg || !w || !out) return fail(DFLASH_ERR_INVALID, "null argument");
  *out = nullptr;
  const dflash_config& g = *cfg;
  if (batch < 1) return fail(DFLASH_ERR_INVALID, "batch must be >= 1");
  if (g.dtype != DFLASH_F32 && g.dtype != DFLASH_BF16) return fail(DFLASH_ERR_INVALID, "dtype must be F32 or BF16");
  if (g.n_layers < 1 || g.n_layers > DFLASH_MAX_LAYERS) return fail(DFLASH_ERR_INVALID, "n_layers out of range");
  if (g.hidden <= 0 || g.n_target_layers <= 0 || g.n_q_heads <= 0 || g.n_kv_heads <= 0 || g.intermediate <= 0 ||
      g.vocab <= 0 || g.k_max < 1)
    return fail(DFLASH_ERR_INVALID, "non-positive dimension");
  if (g.head_dim != 64 && g.head_dim != 128) return fail(DFLASH_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (g.n_q_heads % g.n_kv_heads) return fail(DFLASH_ERR_INVALID, "n_q_heads must be a multiple of n_kv_heads");
  if (g.hidden % 64 || g.intermediate % 64 || (g.n_q_heads * g.head_dim) % 64)
    return fail(DFLASH_ERR_UNSUPPORTED, "hidden, intermediate and n_q_heads*head_dim must be multiples of 64");
  if (g.mask_token_id < 0 || g.mask_token_id >= g.vocab) return fail(DFLASH_ERR_INVALID, "mask_token_id outside vocab");
  if (!(g.rope_theta > 0.f) || !(g.rms_eps >= 0.f)) return fail(DFLASH_ERR_INVALID, "bad rope_theta or rms_eps");
  if (!target && g.n_layers * 2 > kMaxSeg) return fail(DFLASH_ERR_UNSUPPORTED, "too many layers");
  if (g.conditioning < DFLASH_COND_KV || g.conditioning > DFLASH_COND_NONE)
    return fail(DFLASH_ERR_INVALID, "conditioning %d is not a dflash_conditioning", (int)g.conditioning);
  if (g.dtype == DFLASH_BF16 && (g.hidden % 128 || g.intermediate % 128 || g.head_dim != 128))
    return fail(DFLASH_ERR_UNSUPPORTED, "bf16 needs hidden and intermediate multiples of 128 and head_dim 128");
  if ((int64_t)batch * (g.k_max + 1) > (1 << 20)) return fail(DFLASH_ERR_UNSUPPORTED, "batch * (k_max+1) too large");
  auto al = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al(w->embed) || (!target && (!al(w->w_fc) || !al(w->fc_norm))) || !al(w->final_norm) || !al(w->lm_head))
    return fail(DFLASH_ERR_INVALID, "null or unaligned top-level weight");
  for (int l = 0; l < g.n_layers; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    if (!al(lw.wq) || !al(lw.wk) || !al(lw.wv) || !al(lw.wo) || !al(lw.w_gate) || !al(lw.w_up) || !al(lw.w_down) ||
        !al(lw.attn_norm) || !al(lw.mlp_norm))
      return fail(DFLASH_ERR_INVALID, "null or unaligned weight in layer %d", l);
  }
  int dev = 0;
  CK(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3)
    return fail(DFLASH_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", prop.major, prop.minor);

  dflash_ctx* c = new dflash_ctx();
  c->target = target;
  c->cfg = g;
  c->w = *w;
  c->B = batch;
  c->bf16 = g.dtype == DFLASH_BF16;
  c->esz = c->bf16 ? 2 : 4;
  c->num_sms = prop.multiProcessorCount;
  c->H = g.hidden;
  c->F = g.hidden * g.n_target_layers;
  c->I = g.intermediate;
  c->V = g.vocab;
  c->d = g.head_dim;
  c->nl = g.n_layers;
  c->q_dim = g.n_q_heads * g.head_dim;
  c->kv_dim = g.n_kv_heads * g.head_dim;
  c->rows_per_token = (int64_t)c->nl * 2 * g.n_kv_heads;
  c->M_max = batch * (g.k_max + 1);

  auto bail = [&](int code) {
    free_ctx(c);
    return code;
  };
  auto dalloc = [&](void** p, size_t bytes) -> bool {
    if (injected_alloc_failure() || cudaMalloc(p, bytes) != cudaSuccess) {
      cudaGetLastError();
      *p = nullptr;
      return false;
    }
    return true;
  };

  const int B = batch;
  // small state
  if (!dalloc((void**)&c->d_i32, sizeof(int32_t) * (size_t)B * 12) || !dalloc((void**)&c->d_kv_base, 8 * (size_t)B) ||
      !dalloc((void**)&c->d_flags, 16) || !dalloc((void**)&c->d_draft, sizeof(int32_t) * (size_t)B * g.k_max) ||
      !dalloc((void**)&c->d_targets, sizeof(int32_t) * (size_t)B * (g.k_max + 1)) ||
      !dalloc((void**)&c->d_rope, sizeof(uint64_t) * (size_t)(c->d / 2)) ||
      !dalloc((void**)&c->d_keys, sizeof(unsigned long long) * kKeyStride * kKeySlots * (size_t)B * g.k_max) ||
      !dalloc((void**)&c->d_counters, sizeof(unsigned int) * kCounters) ||
      !dalloc((void**)&c->d_ss_ctx, sizeof(float) * (size_t)(c->H / kTileRows + 1) * 128) ||
      (g.conditioning == DFLASH_COND_INPUT && !dalloc((void**)&c->d_ulast, sizeof(float) * (size_t)B * c->H)) ||
      !dalloc((void**)&c->d_plan, sizeof(int32_t) * ((size_t)B * (64 + 3) + 1 + (size_t)c->nl)))
    return bail(fail(DFLASH_ERR_OOM, "state allocation failed"));
  c->d_work = c->d_plan;
  c->d_seq_split = c->d_work + (size_t)B * 64;
  c->d_seq_order = c->d_seq_split + 2 * (size_t)B;
  c->d_n_units = c->d_seq_order + (size_t)B;
  c->d_attn_ctr = reinterpret_cast<uint32_t*>(c->d_n_units + 1);
  c->cond = g.conditioning;
  if (c->d_ulast && cudaMemset(c->d_ulast, 0, sizeof(float) * (size_t)B * c->H) != cudaSuccess)
    return bail(fail(DFLASH_ERR_CUDA, "state initialisation failed"));
  c->d_ctx_len = c->d_i32;
  c->d_kv_len = c->d_i32 + B;
  c->d_anchor = c->d_i32 + 2 * B;
  c->d_cap = c->d_i32 + 3 * B;
  c->d_rows = c->d_i32 + 4 * B;
  c->d_rows_in = c->d_i32 + 5 * B;
  c->d_accept = c->d_i32 + 6 * B;
  c->d_next = c->d_i32 + 7 * B;
  c->d_anchor_in = c->d_i32 + 8 * B;
  c->d_pend_base = c->d_i32 + 9 * B;
  c->d_rblk = c->d_i32 + 10 * B;
  c->d_kseq_in = c->d_i32 + 11 * B;
  c->st = SeqState{c->d_ctx_len, c->d_kv_len,  c->d_anchor, c->d_cap, c->d_kv_base, c->d_pend_base,
                   c->d_rblk,    c->d_ulast, c->cond == DFLASH_COND_KV ? 1 : 0};
  {
    const char* b8 = getenv("DFLASH_BN8");
    c->bn8 = !(b8 && b8[0] == '0');
    const char* fa = getenv("DFLASH_FUSE_APPEND");   // 1: defer small appends' K/V into the next draft
    c->fuse_append = fa && fa[0] == '1';
    const char* lf = getenv("DFLASH_LM_FUSED");   // 1: fused-argmax LM head at every M
    c->lm_fused = lf && lf[0] == '1';
    const char* gp = getenv("DFLASH_GEMM_PAIRS");
    c->gemm_pairs = !(gp && gp[0] == '0');
    const char* gg = getenv("DFLASH_GRAPH");   // 0: no recorded drafts
    c->graph_drafts = !(gg && gg[0] == '0');
    const char* gd = getenv("DFLASH_GEMM_DIRECT");   // 0: single-split tiles also reduce through ws
    c->gemm_direct = !(gd && gd[0] == '0');
    const char* gpe = getenv("DFLASH_GEMM_PERSIST");   // 0: multi-wave one-split GEMMs one tile per CTA
    if (gpe && gpe[0] == '0') c->gemm_persist = false;
    const char* gei = getenv("DFLASH_GEMM_BY_EPI");   // 0: one split-K instance reads the epilogue at run time
    if (gei && gei[0] == '0') c->gemm_by_epi = false;
    const char* ae = getenv("DFLASH_ATTN_EARLY");   // 0: every attention load after the dependency wait
    if (ae && ae[0] == '0') c->attn_early = false;
    const char* gb = getenv("DFLASH_GEMM_BN_MAX");   // widest plain token tile, 64..256 in steps of 16
    if (gb) c->gemm_bn_max = std::max(64, std::min(256, atoi(gb) / 16 * 16));
    const char* gc = getenv("DFLASH_GEMM_CTAS");
    c->gemm_ctas = gc ? std::max(0, std::min(2, atoi(gc))) : 0;
    const char* gs = getenv("DFLASH_GEMM_SMEM_KB");
    c->gemm_smem_kb = gs ? std::max(0, std::min(200, atoi(gs))) : 0;
    const char* au = getenv("DFLASH_ATTN_UMMA");   // 0: the mma.sync attention kernel
    c->attn_umma = !(au && au[0] == '0');
    const char* sp = getenv("DFLASH_SPLIT");        // 0: plain bf16 token operands everywhere
    c->split_ops = !(sp && sp[0] == '0');
    const char* f16 = getenv("DFLASH_F16_OPS");     // 0: no fp16 operands (split bf16 at every M)
    c->f16_ops = !(f16 && f16[0] == '0');
    const char* fm = getenv("DFLASH_F16_MIN_ROWS");
    if (fm) c->f16_min_rows = std::max(1, atoi(fm));
  }
  c->ss_rows = std::max<size_t>((size_t)c->M_max, 4096);
  if (!dalloc((void**)&c->d_ss, sizeof(float) * (size_t)std::max(1, c->H / kTileRows) * c->ss_rows))
    return bail(fail(DFLASH_ERR_OOM, "state allocation failed"));
  if (cudaMemset(c->d_counters, 0, sizeof(unsigned int) * kCounters) != cudaSuccess ||
      cudaMemset(c->d_keys, 0, sizeof(unsigned long long) * kKeyStride * kKeySlots * (size_t)B * g.k_max) != cudaSuccess ||
      cudaMemset(c->d_i32, 0, sizeof(int32_t) * (size_t)B * 12) != cudaSuccess ||
      cudaMemset(c->d_kv_base, 0, 8 * (size_t)B) != cudaSuccess || cudaMemset(c->d_flags, 0, 16) != cudaSuccess)
    return bail(fail(DFLASH_ERR_CUDA, "state init failed"));
  {
    // theta^(-2i/d) in double, then / (2 pi) as a 0.64 fixed-point turn fraction
    std::vector<uint64_t> turns(c->d / 2);
    const long double two_pi = 6.283185307179586476925286766559L;
    for (int i = 0; i < c->d / 2; ++i) {
      const double inv = std::pow((double)g.rope_theta, -2.0 * i / (double)c->d);
      turns[i] = (uint64_t)llroundl(ldexpl((long double)inv / two_pi, 64));
    }
    if (cudaMemcpy(c->d_rope, turns.data(), sizeof(uint64_t) * turns.size(), cudaMemcpyHostToDevice) != cudaSuccess)
      return bail(fail(DFLASH_ERR_CUDA, "rope table upload failed"));
  }

  // KV arena: pool of token slots, each rows_per_token rows of head_dim elements
  int64_t pool = g.kv_pool_tokens > 0
                     ? g.kv_pool_tokens
                     : (int64_t)B * std::max<int64_t>(16384, 4 * next_pow2((int64_t)g.k_max + 1));
  c->buddy.init(pool);
  const size_t arena_bytes = (size_t)c->buddy.pool() * c->rows_per_token * c->d * c->esz;
  const int64_t arena_rows = c->buddy.pool() * c->rows_per_token;
  if (c->bf16 && arena_rows >= ((int64_t)1 << 31))
    return bail(fail(DFLASH_ERR_UNSUPPORTED, "KV arena of %lld rows exceeds the 2^31 rows a tensor map addresses",
                     (long long)arena_rows));
  // the arena sits between two guard bands of a known byte pattern
  // (dflash_check_guards): a write past either end of it shows there
  if (!dalloc(&c->arena_raw, arena_bytes + 2 * kGuardBytes))
    return bail(fail(DFLASH_ERR_OOM, "KV arena of %zu bytes (%lld slots) failed", arena_bytes,
                     (long long)c->buddy.pool()));
  c->arena = static_cast<char*>(c->arena_raw) + kGuardBytes;
  c->arena_bytes = arena_bytes;
  // zero once: every slot attention may touch (including masked tail slots of a tile) holds finite values
  if (cudaMemset(c->arena, 0, arena_bytes) != cudaSuccess ||
      cudaMemset(c->arena_raw, kGuardByte, kGuardBytes) != cudaSuccess ||
      cudaMemset(static_cast<char*>(c->arena) + arena_bytes, kGuardByte, kGuardBytes) != cudaSuccess)
    return bail(fail(DFLASH_ERR_CUDA, "arena memset failed"));
  c->kv = KvArena{c->arena, c->nl, g.n_kv_heads, c->d};
  c->seg_tok.assign(B, 0);
  c->cap.assign(B, 0);
  c->ub_ctx.assign(B, 0);
  c->ub_kv.assign(B, 0);

  // activations (rows padded to a multiple of 256 tokens); the GEMM token
  // operands xn, ob, ab hold two planes (split bf16) on the bf16 path
  const size_t Mp = ((size_t)c->M_max + 255) / 256 * 256;
  const size_t XP = c->bf16 ? 2 : 1;
  if (!dalloc((void**)&c->h, Mp * c->H * sizeof(float)) || !dalloc(&c->xn, XP * Mp * c->H * c->esz) ||
      !dalloc(&c->qb, Mp * c->q_dim * c->esz) || !dalloc(&c->ob, XP * Mp * c->q_dim * c->esz) ||
      !dalloc(&c->ab, XP * Mp * c->I * c->esz) || !dalloc(&c->xf, Mp * c->H * c->esz))
    return bail(fail(DFLASH_ERR_OOM, "activation allocation failed"));
  cudaMemset(c->xn, 0, XP * Mp * c->H * c->esz);
  cudaMemset(c->qb, 0, Mp * c->q_dim * c->esz);
  cudaMemset(c->ob, 0, XP * Mp * c->q_dim * c->esz);
  cudaMemset(c->ab, 0, XP * Mp * c->I * c->esz);
  cudaMemset(c->xf, 0, Mp * c->H * c->esz);

  if (c->bf16) {
    if (!load_encoder()) return bail(fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled unavailable"));
    c->lmaps.resize(c->nl);
    const uint64_t Hb = (uint64_t)c->H * 2;
    int r = target ? DFLASH_OK : tmap_bf16(&c->tm_fc, w->w_fc, c->F, c->H, (uint64_t)c->F * 2, kTileRows);
    if (r == DFLASH_OK && c->d == 128)
      r = tmap_bf16(&c->tm_kv, c->arena, (uint64_t)c->d, (uint64_t)arena_rows, (uint64_t)c->d * 2, 64);
    if (r == DFLASH_OK) r = tmap_bf16(&c->tm_lm, w->lm_head, c->H, c->V, Hb, kTileRows);
    for (int l = 0; l < c->nl && r == DFLASH_OK; ++l) {
      const dflash_layer_weights& lw = w->layers[l];
      auto& m = c->lmaps[l];
      r = tmap_bf16(&m.wq, lw.wq, c->H, c->q_dim, Hb, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wk, lw.wk, c->H, c->kv_dim, Hb, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wv, lw.wv, c->H, c->kv_dim, Hb, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wo, lw.wo, c->q_dim, c->H, (uint64_t)c->q_dim * 2, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wg, lw.w_gate, c->H, c->I, Hb, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wu, lw.w_up, c->H, c->I, Hb, kTileRows);
      if (r == DFLASH_OK) r = tmap_bf16(&m.wd, lw.w_down, c->I, c->H, (uint64_t)c->I * 2, kTileRows);
    }
    if (r != DFLASH_OK) return bail(r);
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(fail(DFLASH_ERR_CUDA, "device sync failed at create"));
  *out = c;
  return DFLASH_OK;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, int32_t batch, dflash_ctx** out) {
  return create_impl(cfg, w, batch, out, false);
}

int dflash_destroy(dflash_ctx* ctx) {
  if (!ctx) return fail(DFLASH_ERR_INVALID, "null context");
  free_ctx(ctx);
  return DFLASH_OK;
}

int dflash_reserve(dflash_ctx* c, int32_t min_capacity, void* stream) {
  g_err.clear();
  if (!c || min_capacity < 0) return fail(DFLASH_ERR_INVALID, "bad argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int b = 0; b < c->B; ++b) RET(ensure_capacity(c, b, min_capacity, s));
  return DFLASH_OK;
}

int dflash_reserve_headroom(dflash_ctx* c, int32_t headroom, void* stream) {
  g_err.clear();
  if (!c || headroom < 0) return fail(DFLASH_ERR_INVALID, "bad argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int b = 0; b < c->B; ++b)
    RET(ensure_capacity(c, b,
                        c->cond == DFLASH_COND_KV ? std::max(c->ub_ctx[b], c->ub_kv[b]) + (int64_t)headroom
                                                  : (int64_t)c->cfg.k_max + 1,
                        s));
  return DFLASH_OK;
}

int dflash_ctx_append(dflash_ctx* c, const void* feats, int32_t rows_max, const int32_t* rows, void* stream) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  if (rows_max < 0) return fail(DFLASH_ERR_INVALID, "rows_max < 0");
  if (rows_max == 0) return DFLASH_OK;
  if (!feats) return fail(DFLASH_ERR_INVALID, "null feats");
  if ((int64_t)c->B * rows_max > (int64_t)1 << 30) return fail(DFLASH_ERR_INVALID, "rows_max too large");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool feats_dev = is_device_ptr(feats);
  if (!feats_dev && is_capturing(s)) return fail(DFLASH_ERR_INVALID, "host feats while the stream is captured");
  if (feats_dev && (reinterpret_cast<uintptr_t>(feats) & 15u))
    return fail(DFLASH_ERR_INVALID, "feats must be 16-byte aligned");
  std::vector<int32_t> host_rows;
  const int32_t* rows_dev = nullptr;
  if (rows) {
    if (!is_device_ptr(rows)) {
      host_rows.assign(rows, rows + c->B);
      for (int b = 0; b < c->B; ++b)
        if (host_rows[b] < 0 || host_rows[b] > rows_max)
          return fail(DFLASH_ERR_INVALID, "rows[%d] = %d outside [0, %d]", b, host_rows[b], rows_max);
    }
    RET(stage_i32(rows, c->d_rows_in, c->B, s, &rows_dev));
  }
  RET(flush_pending(c, s));   // the previous append's K/V first (its rows are about to change)
  const int tr = trace_begin(c, DFLASH_TRACE_APPEND, 0.0, s);
  launch_rows_prep(rows_dev, rows_max, c->B, c->d_rows, c->d_flags, s);
  c->launches += 1;
  for (int b = 0; b < c->B; ++b) {
    const int64_t add = host_rows.empty() ? rows_max : host_rows[b];
    const int64_t kv_after = c->ub_kv[b] + add;
    const int64_t need = c->cond == DFLASH_COND_KV ? std::max(kv_after, c->ub_ctx[b]) + c->cfg.k_max + 1
                                                   : (int64_t)c->cfg.k_max + 1;   // the block's rows only
    RET(ensure_capacity(c, b, need, s));
  }
  int r = c->cond != DFLASH_COND_KV ? append_cond(c, feats, feats_dev, rows_max, s)
          : c->bf16                 ? append_bf16(c, feats, feats_dev, rows_max, s)
                                    : append_impl<float>(c, feats, feats_dev, rows_max, s);
  if (r != DFLASH_OK) return r;
  trace_end(c, tr, s);
  for (int b = 0; b < c->B; ++b) {
    c->ub_kv[b] += host_rows.empty() ? rows_max : host_rows[b];
    c->ub_ctx[b] = std::max(c->ub_ctx[b], c->ub_kv[b]);
  }
  return DFLASH_OK;
}

int dflash_draft_block(dflash_ctx* c, const int32_t* anchor_ids, int32_t K, int32_t* draft_ids, float* logits,
                       void* stream) {
  return dflash_draft_block_k(c, anchor_ids, K, nullptr, draft_ids, logits, stream);
}

int dflash_draft_block_k(dflash_ctx* c, const int32_t* anchor_ids, int32_t K, const int32_t* k_seq,
                         int32_t* draft_ids, float* logits, void* stream) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  if (K < 1 || K > c->cfg.k_max) return fail(DFLASH_ERR_INVALID, "K = %d outside [1, %d]", K, c->cfg.k_max);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int32_t* kseq_dev = nullptr;
  if (k_seq) {
    if (!is_device_ptr(k_seq)) {
      for (int b = 0; b < c->B; ++b)
        if (k_seq[b] < 1 || k_seq[b] > K) return fail(DFLASH_ERR_INVALID, "k_seq[%d] = %d outside [1, %d]", b, k_seq[b], K);
    }
    RET(stage_i32(k_seq, c->d_kseq_in, c->B, s, &kseq_dev));
  }
  for (int b = 0; b < c->B; ++b)
    RET(ensure_capacity(c, b, (c->cond == DFLASH_COND_KV ? c->ub_ctx[b] : 0) + K + 1, s));
  const int32_t* anchor_dev = nullptr;
  if (anchor_ids) {
    if (!is_device_ptr(anchor_ids)) {
      for (int b = 0; b < c->B; ++b)
        if (anchor_ids[b] < 0 || anchor_ids[b] >= c->V)
          return fail(DFLASH_ERR_INVALID, "anchor_ids[%d] = %d outside vocab", b, anchor_ids[b]);
    }
    RET(stage_i32(anchor_ids, c->d_anchor_in, c->B, s, &anchor_dev));
  }
  // logits: the fused LM-head epilogue writes them straight into a device
  // buffer (the caller's, or the workspace when the caller's is host memory)
  float* logits_dev = nullptr;
  const bool logits_host = logits && !is_device_ptr(logits);
  if (logits && c->bf16) {
    if (logits_host) {
      RET(ensure_ws(c, (size_t)c->B * K * c->V, s));
      logits_dev = c->ws;
    } else {
      logits_dev = logits;
    }
  }
  auto body = [&](cudaStream_t st) -> int {
    const int tr = trace_begin(c, DFLASH_TRACE_DRAFT, 0.0, st);
    c->kseq_dev = kseq_dev;   // read by the embedding kernel, which records K_b + 1 per sequence
    int r = !c->bf16 ? draft_impl<float>(c, anchor_dev, K, nullptr, st) : draft_bf16(c, anchor_dev, K, logits_dev, st);
    c->kseq_dev = nullptr;
    if (r != DFLASH_OK) return r;
    if (kseq_dev) {   // ids past a sequence's own K are -1
      launch_mask_drafts(c->d_draft, c->st, c->B, K, st);
      CK(cudaGetLastError());
      c->launches += 1;
    }
    trace_end(c, tr, st);
    RET(copy_out(draft_ids, c->d_draft, sizeof(int32_t) * (size_t)c->B * K, st));
    if (logits && (!c->bf16 || logits_host))
      RET(copy_out(logits, c->ws, sizeof(float) * (size_t)c->B * K * c->V, st));
    return DFLASH_OK;
  };
  const bool graphable = c->graph_drafts && c->bf16 && c->n_pairs <= 0 && !c->fuse_append && !c->pending &&
                         c->attn_scratch_ext == nullptr && !c->no_grow && !is_capturing(s) &&
                         (!anchor_ids || is_device_ptr(anchor_ids)) && (!k_seq || is_device_ptr(k_seq)) &&
                         (!logits || is_device_ptr(logits)) &&
                         (!draft_ids || is_device_ptr(draft_ids) || is_pinned_host(draft_ids));
  DraftGraphKey key{K, anchor_ids, k_seq, draft_ids, logits};
  if (graphable && c->dg.valid && c->dg.K == key.K && c->dg.anchor == key.anchor && c->dg.kseq == key.kseq &&
      c->dg.ids == key.ids && c->dg.logits == key.logits && c->dg.epoch == g_grow_epoch.load()) {
    CK(cudaEventRecord(c->ev_fork, s));
    CK(cudaStreamWaitEvent(c->gstream, c->ev_fork, 0));
    CK(cudaGraphLaunch(c->dg.exec, c->gstream));
    CK(cudaEventRecord(c->ev_join, c->gstream));
    CK(cudaStreamWaitEvent(s, c->ev_join, 0));
    c->launches += c->dg.launches;
    c->replays += 1;
    c->last_K = K;
    return DFLASH_OK;
  }
  RET(body(s));
  c->last_K = K;
  if (graphable) record_draft(c, body, key);   // for the next calls with these arguments
  return DFLASH_OK;
}

int dflash_verify_accept(dflash_ctx* c, const int32_t* target_ids, int32_t* accept_len, int32_t* next_anchor,
                         void* stream) {
  g_err.clear();
  if (!c || !target_ids) return fail(DFLASH_ERR_INVALID, "null argument");
  if (c->last_K < 1) return fail(DFLASH_ERR_INVALID, "verify before any draft");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int K = c->last_K;
  const int32_t* tg = nullptr;
  if (!is_device_ptr(target_ids)) {
    for (int e = 0; e < c->B * (K + 1); ++e)
      if (target_ids[e] < 0 || target_ids[e] >= c->V)
        return fail(DFLASH_ERR_INVALID, "target_ids[%d] = %d outside vocab", e, target_ids[e]);
  }
  RET(stage_i32(target_ids, c->d_targets, (size_t)c->B * (K + 1), s, &tg));
  const int tr = trace_begin(c, DFLASH_TRACE_VERIFY, 0.0, s);
  launch_accept(c->d_draft, tg, c->B, K, c->V, c->st, c->d_accept, c->d_next, c->d_flags, s);
  CK(cudaGetLastError());
  trace_end(c, tr, s);
  c->launches += 1;
  RET(copy_out(accept_len, c->d_accept, sizeof(int32_t) * c->B, s));
  RET(copy_out(next_anchor, c->d_next, sizeof(int32_t) * c->B, s));
  for (int b = 0; b < c->B; ++b) c->ub_ctx[b] += K + 1;
  return DFLASH_OK;
}

int dflash_query_state(dflash_ctx* c, void* stream, int32_t* ctx_len, int32_t* kv_len, int32_t* capacity,
                       int32_t* anchor, uint32_t* device_flags) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (is_capturing(s)) return fail(DFLASH_ERR_INVALID, "query_state while the stream is captured");
  CK(cudaStreamSynchronize(s));
  std::vector<int32_t> buf((size_t)c->B * 4);
  CK(cudaMemcpy(buf.data(), c->d_i32, sizeof(int32_t) * (size_t)c->B * 4, cudaMemcpyDeviceToHost));
  uint32_t flags = 0;
  CK(cudaMemcpy(&flags, c->d_flags, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  CK(cudaMemset(c->d_flags, 0, sizeof(uint32_t)));
  for (int b = 0; b < c->B; ++b) {
    c->ub_ctx[b] = buf[b];
    c->ub_kv[b] = buf[c->B + b];
    if (ctx_len) ctx_len[b] = buf[b];
    if (kv_len) kv_len[b] = buf[c->B + b];
    if (anchor) anchor[b] = buf[2 * c->B + b];
    if (capacity) capacity[b] = buf[3 * c->B + b];
  }
  if (device_flags) *device_flags = flags;
  if (flags) return fail(DFLASH_ERR_DEVICE_FLAG, "device fault bits 0x%x", flags);
  return DFLASH_OK;
}

int dflash_plant_targets(const int32_t* draft_ids, const int32_t* accept_len_plan, const int32_t* fill,
                         int32_t batch, int32_t K, int32_t vocab, int32_t* target_ids, int32_t* step_counter,
                         int32_t n_plans, void* stream) {
  g_err.clear();
  if (!draft_ids || !accept_len_plan || !fill || !target_ids || batch < 1 || K < 1 || vocab < 1)
    return fail(DFLASH_ERR_INVALID, "bad argument");
  if (step_counter && n_plans < 1) return fail(DFLASH_ERR_INVALID, "n_plans must be >= 1");
  launch_plant(draft_ids, accept_len_plan, fill, batch, K, vocab, target_ids, step_counter, n_plans < 1 ? 1 : n_plans,
               reinterpret_cast<cudaStream_t>(stream));
  CK(cudaGetLastError());
  return DFLASH_OK;
}

int dflash_trace_enable(dflash_ctx* c, int32_t n_pairs) {
  g_err.clear();
  if (!c || n_pairs < 0) return fail(DFLASH_ERR_INVALID, "bad argument");
  CK(cudaDeviceSynchronize());
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  c->ev.clear();
  c->trace.clear();
  c->n_pairs = 0;
  c->next_pair = 0;
  for (int i = 0; i < 2 * n_pairs; ++i) {
    cudaEvent_t e;
    CK(cudaEventCreate(&e));
    c->ev.push_back(e);
  }
  c->n_pairs = n_pairs;
  return DFLASH_OK;
}

int dflash_trace_read(dflash_ctx* c, int32_t max, int32_t* kind, float* ms, double* bytes, int32_t* count) {
  g_err.clear();
  if (!c || max < 0 || !count) return fail(DFLASH_ERR_INVALID, "bad argument");
  CK(cudaDeviceSynchronize());
  int n = 0;
  for (const auto& t : c->trace) {
    if (n >= max) break;
    float e = 0.f;
    if (cudaEventElapsedTime(&e, c->ev[2 * t.pair], c->ev[2 * t.pair + 1]) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (kind) kind[n] = t.kind;
    if (ms) ms[n] = e;
    if (bytes) bytes[n] = t.bytes;
    ++n;
  }
  c->trace.clear();
  *count = n;
  return DFLASH_OK;
}

int dflash_read_kv(dflash_ctx* c, int32_t seq, int32_t layer, int32_t kind, int32_t slot0, int32_t n_slots,
                   void* host_out, void* stream) {
  g_err.clear();
  if (!c || !host_out || seq < 0 || seq >= c->B || layer < 0 || layer >= c->nl || (kind != 0 && kind != 1) ||
      slot0 < 0 || n_slots < 0)
    return fail(DFLASH_ERR_INVALID, "bad argument");
  if ((int64_t)slot0 + n_slots > c->cap[seq])
    return fail(DFLASH_ERR_INVALID, "slots [%d, %d) beyond capacity %lld", slot0, slot0 + n_slots,
                (long long)c->cap[seq]);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  RET(flush_pending(c, s));
  CK(cudaStreamSynchronize(s));
  const size_t row_bytes = (size_t)c->d * c->esz;
  for (int h = 0; h < c->cfg.n_kv_heads; ++h) {
    const int64_t row = kv_row(c->kv, c->seg_tok[seq] * c->rows_per_token, (int)c->cap[seq], layer, kind, h, slot0);
    CK(cudaMemcpy(reinterpret_cast<char*>(host_out) + (size_t)h * n_slots * row_bytes,
                  reinterpret_cast<const char*>(c->arena) + row * row_bytes, (size_t)n_slots * row_bytes,
                  cudaMemcpyDeviceToHost));
  }
  return DFLASH_OK;
}

int dflash_launch_count(dflash_ctx* c, int64_t* launches) {
  if (!c || !launches) return fail(DFLASH_ERR_INVALID, "bad argument");
  *launches = c->launches;
  return DFLASH_OK;
}

int dflash_graph_replays(dflash_ctx* c, int64_t* replays) {
  if (!c || !replays) return fail(DFLASH_ERR_INVALID, "bad argument");
  *replays = c->replays;
  return DFLASH_OK;
}

int dflash_set_wait_limit(dflash_ctx* c, uint64_t limit_ns) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  // the limit sits next to the flag word: flags + 2 (8 bytes, 8-byte aligned)
  if (cudaMemcpy(c->d_flags + 2, &limit_ns, sizeof(limit_ns), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return fail(DFLASH_ERR_CUDA, "wait-limit upload failed");
  }
  return DFLASH_OK;
}

int dflash_selftest_wait(dflash_ctx* c, void* stream) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  CK(launch_wait_selftest(c->d_flags, reinterpret_cast<cudaStream_t>(stream)));
  c->launches += 1;
  return DFLASH_OK;
}

int64_t dflash_inject_alloc_failure(int64_t after) {
  return g_alloc_fail_after.exchange(after < 0 ? -1 : after);
}

int dflash_check_guards(dflash_ctx* c, void* stream) {
  g_err.clear();
  if (!c) return fail(DFLASH_ERR_INVALID, "null context");
  if (c->arena_raw == nullptr) return DFLASH_OK;
  std::vector<unsigned char> g(2 * kGuardBytes);
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(g.data(), c->arena_raw, kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(g.data() + kGuardBytes, static_cast<char*>(c->arena) + c->arena_bytes, kGuardBytes,
                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return fail(DFLASH_ERR_CUDA, "guard-band read failed");
  }
  for (size_t i = 0; i < g.size(); ++i)
    if (g[i] != (unsigned char)kGuardByte)
      return fail(DFLASH_ERR_DEVICE_FLAG, "KV arena guard band %s the arena overwritten at byte %zu",
                  i < kGuardBytes ? "before" : "after", i < kGuardBytes ? i : i - kGuardBytes);
  return DFLASH_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- the target side
struct dflash_target {
  dflash_ctx* c;
  int r_last;   // R of the last forward (the bound of the next commit)
};

int dflash_target_create(const dflash_target_config* cfg, const dflash_weights* w, int32_t batch,
                         dflash_target** out) {
  g_err.clear();
  if (!cfg || !w || !out) return fail(DFLASH_ERR_INVALID, "null argument");
  *out = nullptr;
  const dflash_target_config& t = *cfg;
  if (t.r_max < 1) return fail(DFLASH_ERR_INVALID, "r_max must be >= 1");
  if (t.n_feat < 0 || t.n_feat > 8) return fail(DFLASH_ERR_INVALID, "n_feat outside [0, 8]");
  for (int i = 0; i < t.n_feat; ++i)
    if (t.feat_layers[i] < 0 || t.feat_layers[i] >= t.n_layers || (i > 0 && t.feat_layers[i] <= t.feat_layers[i - 1]))
      return fail(DFLASH_ERR_INVALID, "feat_layers must increase strictly inside [0, n_layers)");
  dflash_config g;
  memset(&g, 0, sizeof(g));
  g.hidden = t.hidden;
  g.n_target_layers = 1;
  g.n_layers = t.n_layers;
  g.n_q_heads = t.n_q_heads;
  g.n_kv_heads = t.n_kv_heads;
  g.head_dim = t.head_dim;
  g.intermediate = t.intermediate;
  g.vocab = t.vocab;
  g.rope_theta = t.rope_theta;
  g.rms_eps = t.rms_eps;
  g.mask_token_id = 0;
  g.k_max = t.r_max;   // a forward of R rows is laid out as a block of K + 1 = R rows
  g.dtype = DFLASH_BF16;
  g.kv_pool_tokens = t.kv_pool_tokens;
  g.conditioning = DFLASH_COND_KV;
  dflash_ctx* c = nullptr;
  const int r = create_impl(&g, w, batch, &c, true);
  if (r != DFLASH_OK) return r;
  c->n_feat = t.n_feat;
  for (int i = 0; i < t.n_feat; ++i) c->feat_layers[i] = t.feat_layers[i];
  const char* tp = getenv("DFLASH_TARGET_PLAIN");
  c->target_plain = tp && tp[0] == '1';
  *out = new dflash_target{c, 0};
  return DFLASH_OK;
}

int dflash_target_destroy(dflash_target* t) {
  g_err.clear();
  if (!t) return fail(DFLASH_ERR_INVALID, "null target");
  const int r = dflash_destroy(t->c);
  delete t;
  return r;
}

int dflash_target_forward(dflash_target* t, const int32_t* tokens, int32_t R, int32_t* ids, float* logits,
                          void* feats, void* stream) {
  g_err.clear();
  if (!t || !tokens || !ids) return fail(DFLASH_ERR_INVALID, "null argument");
  dflash_ctx* c = t->c;
  if (R < 1 || R > c->cfg.k_max) return fail(DFLASH_ERR_INVALID, "R = %d outside [1, %d]", R, c->cfg.k_max);
  if (!is_device_ptr(tokens) || !is_device_ptr(ids) || (logits && !is_device_ptr(logits)) ||
      (feats && !is_device_ptr(feats)))
    return fail(DFLASH_ERR_INVALID, "tokens, ids, logits and feats must be device memory");
  if (feats && c->n_feat == 0) return fail(DFLASH_ERR_INVALID, "feats requested but n_feat = 0");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int b = 0; b < c->B; ++b) RET(ensure_capacity(c, b, c->ub_kv[b] + R, s));
  const dflash_ctx::TargetRun run{tokens, ids, logits, reinterpret_cast<__nv_bfloat16*>(feats)};
  c->trun = &run;
  c->kseq_dev = nullptr;
  const int tr = trace_begin(c, DFLASH_TRACE_DRAFT, 0.0, s);
  const int r = draft_bf16(c, nullptr, R - 1, nullptr, s);
  c->trun = nullptr;
  if (r != DFLASH_OK) return r;
  trace_end(c, tr, s);
  CK(cudaGetLastError());
  t->r_last = R;
  return DFLASH_OK;
}

int dflash_target_commit(dflash_target* t, const int32_t* keep, void* stream) {
  g_err.clear();
  if (!t || !keep) return fail(DFLASH_ERR_INVALID, "null argument");
  dflash_ctx* c = t->c;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool dev = is_device_ptr(keep);
  if (!dev)
    for (int b = 0; b < c->B; ++b)
      if (keep[b] < 0 || keep[b] > t->r_last)
        return fail(DFLASH_ERR_INVALID, "keep[%d] = %d outside [0, %d]", b, keep[b], t->r_last);
  const int32_t* keep_dev = nullptr;
  RET(stage_i32(keep, c->d_rows_in, c->B, s, &keep_dev));
  launch_target_commit(keep_dev, c->st, c->B, c->d_flags, s);
  CK(cudaGetLastError());
  c->launches += 1;
  for (int b = 0; b < c->B; ++b) {
    c->ub_kv[b] += dev ? t->r_last : keep[b];
    c->ub_ctx[b] = c->ub_kv[b];
  }
  t->r_last = 0;
  return DFLASH_OK;
}

int dflash_target_query(dflash_target* t, void* stream, int32_t* len, uint32_t* device_flags) {
  if (!t) return fail(DFLASH_ERR_INVALID, "null target");
  return dflash_query_state(t->c, stream, len, nullptr, nullptr, nullptr, device_flags);
}
