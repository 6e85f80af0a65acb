/*
 * dflash.h -- C ABI of the DFlash block-diffusion drafter hot path (GB300, sm_103a).
 *
 * One stateful proposer per context: it projects target hidden features into a
 * static per-sequence draft KV cache, drafts a whole block [anchor ; K masks]
 * in one non-causal forward, and greedily verifies the drafts against the
 * target's argmax tokens, advancing its state by the accepted count only.
 *
 * Pages the operations follow (cited by title and section):
 *   [GDB] "在谷歌TPU上实现3倍加速：UCSD利用扩散式推测解码优化LLM推理"
 *         (AI translation of the Google Developers Blog post on DFlash on TPU)
 *   [KCH] "D-Flash：扩散草稿让大模型推理提速3.5倍的秘密" (summary of the DFlash paper)
 *
 * Conventions shared by every call
 *   - Every call is asynchronous on the given CUDA stream (`stream` is a
 *     cudaStream_t passed as void*; NULL = the legacy default stream) and
 *     returns a dflash_status.  No call exits, traps or asserts on the GPU.
 *   - Buffer arguments may live in device memory or in host memory; the
 *     library tells them apart with cudaPointerGetAttributes.  Host inputs
 *     are copied before the call returns; host outputs are written by a
 *     stream-ordered copy (pinned host memory: valid after the stream is
 *     synchronised; pageable host memory: the copy completes before return).
 *     While a stream is being captured into a CUDA graph, every buffer must be
 *     device memory and no capacity growth may be needed (see dflash_reserve).
 *   - The caller owns all inputs, outputs and the weights; weights are
 *     BORROWED and must outlive the context.  The context owns its state,
 *     its KV arena and its workspaces.
 *   - A context is not thread-safe: use one context per stream.
 *   - Invalid arguments return DFLASH_ERR_INVALID and set dflash_last_error().
 *   - Faults detected on the device (a token id outside [0, V), drafting
 *     before the accepted rows were appended, a KV slot beyond capacity, a
 *     bounded wait that ran out) are latched in a device word, never trapped,
 *     and reported by dflash_query_state as DFLASH_ERR_DEVICE_FLAG.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_MAX_LAYERS 32

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID = 1,      /* bad argument; see dflash_last_error() */
  DFLASH_ERR_OOM = 2,          /* device or pinned allocation failed, or the KV arena is full */
  DFLASH_ERR_CAPACITY = 3,     /* growth needed while a stream is being captured */
  DFLASH_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  DFLASH_ERR_DEVICE_FLAG = 5,  /* a device-side check latched a fault (dflash_query_state) */
  DFLASH_ERR_UNSUPPORTED = 6   /* shape outside what the kernels implement */
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* How the target context conditions a draft ("D-Flash" write-up, sections on the
   target-feature KV injection and on the ablation experiments):
   DFLASH_COND_KV     -- the method: every consumed row's context feature u =
                         RMSNorm(W_fc f) is projected by each draft layer's W_k, W_v
                         into that layer's KV cache, and the block attends to it;
   DFLASH_COND_INPUT  -- input fusion, the ablation's alternative: no context keys;
                         the context feature of each sequence's most recently
                         consumed row is added to the embedding of every block row;
   DFLASH_COND_NONE   -- no target context: the block attends to itself only.
   In every mode ctx_append consumes the rows (kv_len advances, the draft still
   requires kv_len == ctx_len) and positions continue from ctx_len; without K/V
   injection the KV arena holds only the block's rows (capacity k_max + 1). */
typedef enum { DFLASH_COND_KV = 0, DFLASH_COND_INPUT = 1, DFLASH_COND_NONE = 2 } dflash_conditioning;

/* device fault bits reported through dflash_query_state(..., device_flags) */
#define DFLASH_FLAG_BAD_TOKEN      0x1u  /* token id outside [0, V): clamped to 0 */
#define DFLASH_FLAG_NOT_CONSUMED   0x2u  /* draft while kv_len != ctx_len */
#define DFLASH_FLAG_CAPACITY       0x4u  /* KV slot beyond capacity: write skipped */
#define DFLASH_FLAG_WAIT_TIMEOUT   0x8u  /* a bounded mbarrier wait ran out: kernel returned */
#define DFLASH_FLAG_BAD_ROWS       0x10u /* append row count outside [0, rows_max]: clamped */
#define DFLASH_FLAG_BAD_K          0x20u /* per-sequence K outside [1, K]: clamped */
#define DFLASH_FLAG_F16_RANGE      0x40u /* an fp16 GEMM operand (drafts of >= 33 rows) outside
                                            +-65504 or NaN: the value was stored as fp16 inf/NaN */

/* Drafter shape.  All matrix widths must be multiples of 64; head_dim 64 or 128;
   n_q_heads a multiple of n_kv_heads. */
typedef struct dflash_config {
  int32_t hidden;           /* H */
  int32_t n_target_layers;  /* L_t: target-layer features per token, concatenated */
  int32_t n_layers;         /* draft layers, <= DFLASH_MAX_LAYERS */
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;         /* d */
  int32_t intermediate;     /* SwiGLU inner size I */
  int32_t vocab;            /* V (size of the target's LM head and embedding) */
  float rope_theta;
  float rms_eps;
  int32_t mask_token_id;    /* id whose embedding fills the K mask rows */
  int32_t k_max;            /* largest K a draft may use */
  int32_t dtype;            /* dflash_dtype of weights and features; activations follow */
  int64_t kv_pool_tokens;   /* token slots of the KV arena over all sequences; 0 = default:
                               batch * max(16384, 4 * next_pow2(k_max + 1)) */
  int32_t conditioning;     /* dflash_conditioning; DFLASH_ERR_INVALID outside it */
} dflash_config;

/* One draft layer's weights, row-major [out, in] (nn.Linear layout), device memory. */
typedef struct dflash_layer_weights {
  const void* wq;         /* [n_q_heads*d, H] */
  const void* wk;         /* [n_kv_heads*d, H] */
  const void* wv;         /* [n_kv_heads*d, H] */
  const void* wo;         /* [H, n_q_heads*d] */
  const void* w_gate;     /* [I, H] */
  const void* w_up;       /* [I, H] */
  const void* w_down;     /* [H, I] */
  const void* attn_norm;  /* [H] RMSNorm gain before attention */
  const void* mlp_norm;   /* [H] RMSNorm gain before the MLP */
} dflash_layer_weights;

/* All weights, device memory, dtype = config.dtype, 16-byte aligned. */
typedef struct dflash_weights {
  const void* embed;       /* [V, H] token embedding (the target's) */
  const void* w_fc;        /* [H, L_t*H] projection of the concatenated target features */
  const void* fc_norm;     /* [H] RMSNorm gain of the projected context feature */
  const void* final_norm;  /* [H] RMSNorm gain before the LM head */
  const void* lm_head;     /* [V, H] the target's LM head */
  dflash_layer_weights layers[DFLASH_MAX_LAYERS];
} dflash_weights;

typedef struct dflash_ctx dflash_ctx;

/* Create a proposer for `batch` independent sequences on the current device.
 * Allocates the KV arena (config.kv_pool_tokens token slots, each holding the
 * K and V rows of every layer) and the workspaces.  Every sequence starts empty:
 * ctx_len = kv_len = 0, anchor = 0.  Synchronous.  [GDB §用于注意力机制的“双缓存”方案]:
 * the drafter keeps its own static device arrays for the non-causal block. */
int dflash_create(const dflash_config* cfg, const dflash_weights* w, int32_t batch,
                  dflash_ctx** out);

/* Free everything the context owns (synchronises the device first). */
int dflash_destroy(dflash_ctx* ctx);

/* Grow every sequence's KV capacity to at least `min_capacity` token slots
 * (rounded up to a power of two).  Call before capturing a stream into a CUDA
 * graph so that no growth is needed inside the graph. */
int dflash_reserve(dflash_ctx* ctx, int32_t min_capacity, void* stream);

/* Grow each sequence's KV capacity to hold its own context plus `headroom`
 * more token slots (the host's upper bound of the committed length, rounded up
 * to a power of two) -- the per-sequence form of dflash_reserve for ragged
 * batches, so that `headroom` tokens of drafting and appending need no growth.
 * DFLASH_ERR_OOM when the KV pool cannot hold it. */
int dflash_reserve_headroom(dflash_ctx* ctx, int32_t headroom, void* stream);

/* Context append.  [KCH §系统架构]: the L_t target features of a token are
 * concatenated and projected by fc to one target context feature; [KCH §创新二]:
 * that feature goes through every draft layer's own K and V projections and is
 * stored as persistent context KV.  Computes, for sequence b and row r < rows[b]:
 *     u = RMSNorm(W_fc x_{b,r}) * fc_norm
 *     K_l = RoPE(W_k^l u, kv_len_b + r),  V_l = W_v^l u      (every layer l)
 * stored at KV slot kv_len_b + r; then kv_len_b += rows[b] and
 * ctx_len_b = max(ctx_len_b, kv_len_b).  [GDB §智能上下文管理]: kv_len counts
 * exactly the context consumed so far.
 *   feats:    [batch, rows_max, L_t*H] (dtype), row r of sequence b at
 *             (b*rows_max + r)*L_t*H; rows r >= rows[b] are padding and ignored.
 *   rows_max: padded rows per sequence (>= 0).
 *   rows:     int32 [batch], each in [0, rows_max] (host or device; a device
 *             array such as accept_len+1 needs no host synchronisation), or
 *             NULL = rows_max for every sequence.
 * Capacity grows to a power of two (>= 64) covering kv_len + rows_max. */
int dflash_ctx_append(dflash_ctx* ctx, const void* feats, int32_t rows_max,
                      const int32_t* rows, void* stream);

/* One block-diffusion draft: one non-causal forward over [anchor ; K masks] for
 * every sequence ([KCH §系统架构, §创新一]; [GDB §用于注意力机制的“双缓存”方案]).
 * Block row j of sequence b sits at position ctx_len_b + j and sees all
 * kv_len_b context keys and all K+1 block keys (no mask, GQA, RoPE); each
 * draft layer is pre-norm attention + SwiGLU MLP; the K mask rows go through
 * the final RMSNorm and the LM head, and d_j is the greedy argmax (lowest id
 * on ties).  The block's own K/V occupy slots kv_len_b .. kv_len_b + K until
 * the next append overwrites them.
 *   anchor_ids: int32 [batch] (host or device) that replaces the held anchors,
 *               or NULL to use the anchors left by dflash_verify_accept.
 *   K:          1 .. k_max.
 *   draft_ids:  out int32 [batch, K] (host or device), or NULL.
 *   logits:     out float [batch, K, V] (host or device), or NULL to skip.
 * A bf16 draft records its launches into a CUDA graph the first time it sees a
 * set of arguments (K and these pointers, device or pinned-host outputs) and
 * replays it on a private stream, ordered after and before `stream` by events,
 * while the arguments and the context's workspaces stay the same; inside a
 * caller's stream capture, with host anchors or with tracing on it launches
 * eagerly (environment DFLASH_GRAPH=0: always).
 * A bf16 draft of 33 rows or more (B * (K + 1); environment DFLASH_F16_MIN_ROWS
 * moves the threshold) with head_dim 128 feeds the tensor cores fp16 token
 * operands (11 significant bits) instead of split bf16 ones (about 16), against
 * fp16 copies of the layer and
 * LM-head weights, which the first such draft makes (one allocation of the
 * weights' size, kept until dflash_destroy; the weights must not change
 * afterwards); without the memory, inside a stream capture, in
 * dflash_draft_block_noalloc or with DFLASH_F16_OPS=0 it keeps split bf16. */
int dflash_draft_block(dflash_ctx* ctx, const int32_t* anchor_ids, int32_t K,
                       int32_t* draft_ids, float* logits, void* stream);

/* The same draft with a block length per sequence (K may differ per sequence
 * without any rebuild; [KCH §创新一] drafts a block of masks, and nothing in
 * the method ties the sequences of a batch to one block length).  Sequence b
 * drafts K_b = k_seq[b] masks: its block rows j <= K_b see its kv_len_b
 * context keys and its own K_b + 1 block keys, exactly as a draft of K = K_b;
 * the layout is still K + 1 rows per sequence, the rows past K_b are computed
 * and discarded.
 *   k_seq:     int32 [batch], each in [1, K] (host: checked, DFLASH_ERR_INVALID;
 *              device: clamped, DFLASH_FLAG_BAD_K), or NULL = K for all.
 *   draft_ids: [batch, K]; entries k >= K_b are -1.  logits rows k >= K_b are
 *              not meaningful.
 * The next dflash_verify_accept compares sequence b's first K_b drafts (its
 * target row still has K + 1 entries; entries past K_b are ignored). */
int dflash_draft_block_k(dflash_ctx* ctx, const int32_t* anchor_ids, int32_t K, const int32_t* k_seq,
                         int32_t* draft_ids, float* logits, void* stream);

/* Same draft as dflash_draft_block, for callers that must not allocate device
 * memory while drafting (a loop recorded by stream capture in global mode, where
 * cudaMalloc is an error; a process whose device memory is carved up once at
 * start-up).  The pages have no counterpart: this is a deployment variant.
 * The attention's split-KV scratch comes from a static device array of 8 MiB
 * (2M floats) held by every GPU that loads the library.  A draft needs
 * batch x kv_heads x splits x rows_pad x 129 floats of it (rows_pad: the query
 * rows of a KV head, G x (K + 1), rounded up to 128 on the tensor-core path);
 * when the split count the draft would choose does not fit, it runs with as
 * many splits as fit (one split needs none), so its ids and logits agree with
 * dflash_draft_block's up to the fp32 summation order of the split merge.  A
 * draft that would need any context workspace to grow (run one
 * dflash_draft_block with the same K and batch first) fails with
 * DFLASH_ERR_CAPACITY and allocates nothing.  The first call on a device (or
 * on a new context of it) looks up the array's device address (with lazy
 * module loading this is also when the array's 8 MiB appear on that device),
 * so make it before any stream capture.  All calls share the array: calls that
 * overlap on the GPU (other streams, other contexts) race on it.  Arguments and
 * results as for dflash_draft_block. */
int dflash_draft_block_noalloc(dflash_ctx* ctx, const int32_t* anchor_ids, int32_t K,
                               int32_t* draft_ids, float* logits, void* stream);

/* Greedy verify-and-accept of the last draft.  [GDB §克服自回归瓶颈]: the target
 * checks all drafts in one parallel forward; [GDB §弥合 TPU 推理中的元数据鸿沟]:
 * the proposer's positions advance by the truly accepted count only.
 *   target_ids:  int32 [batch, K+1] (host or device): g_0..g_K, g_{j-1} being the
 *                target's argmax where d_j was proposed, g_K the bonus.
 *   accept_len:  out int32 [batch]: n_b = max{n <= K : d_j == g_{j-1} for all j <= n}.
 *   next_anchor: out int32 [batch]: g_{n_b}, also held as the next anchor.
 * On the device: ctx_len_b += n_b + 1.  The n_b + 1 committed rows (anchor and
 * accepted drafts) are expected from the next dflash_ctx_append. */
int dflash_verify_accept(dflash_ctx* ctx, const int32_t* target_ids,
                         int32_t* accept_len, int32_t* next_anchor, void* stream);

/* Synchronise `stream`, then copy the per-sequence state to host arrays of
 * [batch] (any may be NULL) and return the latched device fault bits (cleared
 * by this call).  Returns DFLASH_ERR_DEVICE_FLAG when any bit was set. */
int dflash_query_state(dflash_ctx* ctx, void* stream, int32_t* ctx_len, int32_t* kv_len,
                       int32_t* capacity, int32_t* anchor, uint32_t* device_flags);

/* Message of the last failing call on this thread ("" if none). */
const char* dflash_last_error(void);

/* Tracing.  With n_pairs > 0, every later tensor-core / CUDA-core GEMM launch
 * and every ctx_append / draft_block / verify_accept call is bracketed by a
 * pair of CUDA events taken round-robin from a pool of n_pairs (0 disables and
 * frees the pool).  Events recorded while a stream is captured become graph
 * nodes and are re-recorded on every replay. */
#define DFLASH_TRACE_GEMM    0   /* one GEMM launch; bytes = weights + activations + fp32 output */
#define DFLASH_TRACE_APPEND  1   /* one dflash_ctx_append call */
#define DFLASH_TRACE_DRAFT   2   /* one dflash_draft_block call */
#define DFLASH_TRACE_VERIFY  3   /* one dflash_verify_accept call */
#define DFLASH_TRACE_ENGINE  4   /* one draft-engine launch (the whole bf16 draft forward after the embedding);
                                    bytes = every weight once + the context K/V read */
int dflash_trace_enable(dflash_ctx* ctx, int32_t n_pairs);
/* Synchronise the device and report the traced events recorded since
 * dflash_trace_enable, oldest first, at most `max` of them: kind
 * (DFLASH_TRACE_*), elapsed milliseconds and algorithmic bytes (GEMMs only).
 * *count receives the number written.  The pairs are then free for reuse. */
int dflash_trace_read(dflash_ctx* ctx, int32_t max, int32_t* kind, float* ms, double* bytes,
                      int32_t* count);

/* Copy KV rows of one sequence to host memory (synchronises `stream`): slots
 * [slot0, slot0 + n_slots) of layer `layer`, kind 0 = K (after RoPE) or 1 = V,
 * for every KV head, as [n_kv_heads][n_slots][head_dim] elements of the
 * context dtype.  Slots must lie inside the sequence's capacity. */
int dflash_read_kv(dflash_ctx* ctx, int32_t seq, int32_t layer, int32_t kind, int32_t slot0,
                   int32_t n_slots, void* host_out, void* stream);

/* Number of kernels this context has launched (or captured) so far. */
int dflash_launch_count(dflash_ctx* ctx, int64_t* launches);

/* Number of drafts this context has served by replaying a recorded graph
 * (see dflash_draft_block); a diagnostic, like dflash_launch_count. */
int dflash_graph_replays(dflash_ctx* ctx, int64_t* replays);

/* Synthetic-input harness, not part of the method: plants target ids that
 * force accepted lengths.  For each b with L = plan row p of accept_len_plan:
 *   g[b][j] = d[b][j] for j < L;  g[b][L] = (d[b][L] + 1) mod V if L < K;
 *   every other g[b][j] = fill[p][b][j].
 * draft_ids [B, K]; accept_len_plan [n_plans, B]; fill [n_plans, B, K+1];
 * target_ids out [B, K+1]; all int32 device memory.  With step_counter NULL
 * the plan row is 0; otherwise it is *step_counter mod n_plans and the kernel
 * increments *step_counter (so a captured step walks through the plans). */
int dflash_plant_targets(const int32_t* draft_ids, const int32_t* accept_len_plan,
                         const int32_t* fill, int32_t batch, int32_t K, int32_t vocab,
                         int32_t* target_ids, int32_t* step_counter, int32_t n_plans,
                         void* stream);

/* ---------------------------------------------------------------- the target side
 * The other half of the speculative loop: the target model's verify forward.
 * [GDB §克服自回归瓶颈]: the target checks a whole block of drafted tokens in one
 * parallel forward; [GDB §"K-Flat" 突破]: verifying 1024 tokens costs about as
 * much as 16, the time going to the weights; [GDB §用于注意力机制的"双缓存"方案]:
 * the target keeps its own KV cache, apart from the drafter's.  The target is a
 * pre-norm decoder of the drafter's layer shape (RMSNorm, GQA with rotate-half
 * RoPE, SwiGLU, final RMSNorm, LM head) with causal attention; bf16, head_dim
 * 128.  Weights: a dflash_weights whose embed, final_norm, lm_head and
 * layers[0 .. n_layers) are used (w_fc and fc_norm are not). */
typedef struct dflash_target dflash_target;   /* opaque */

typedef struct dflash_target_config {
  int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, intermediate, vocab;
  float rope_theta, rms_eps;
  int32_t r_max;            /* largest R of a forward (rows per sequence) */
  int32_t n_feat;           /* layers whose outputs are exported as features, 0 .. 8 */
  int32_t feat_layers[8];   /* their indices, strictly increasing, < n_layers */
  int64_t kv_pool_tokens;   /* KV arena token slots over all sequences; 0 = default */
} dflash_target_config;

int dflash_target_create(const dflash_target_config* cfg, const dflash_weights* w, int32_t batch,
                         dflash_target** out);
int dflash_target_destroy(dflash_target* t);

/* Forward of R new tokens per sequence at positions len_b .. len_b + R - 1:
 * row j attends to the len_b cached positions and to rows 0 .. j (causal).
 *   tokens: int32 [batch, R], device memory (ids outside [0, V) are clamped to 0
 *           and latch DFLASH_FLAG_BAD_TOKEN).
 *   R:      1 .. r_max.
 *   ids:    out int32 [batch, R], device: the greedy id (lowest on ties) of every
 *           row -- row j predicts position len_b + j + 1, so for a verify block
 *           [anchor, d_1 .. d_K] these are g_0 .. g_K of dflash_verify_accept.
 *   logits: out float [batch, R, V], device, or NULL.
 *   feats:  out bf16 [batch, R, n_feat * hidden], device, or NULL: the residual
 *           stream after each feature layer, concatenated in layer order (the
 *           drafter's ctx_append rows, with L_t = n_feat).
 * The rows' K/V are written at slots len_b .. len_b + R - 1 and stay provisional
 * until dflash_target_commit. */
int dflash_target_forward(dflash_target* t, const int32_t* tokens, int32_t R, int32_t* ids, float* logits,
                          void* feats, void* stream);

/* Keep the first keep[b] rows of the last forward as cache: len_b += keep[b]
 * ([GDB §弥合 TPU 推理中的元数据鸿沟]: the state advances by the accepted count,
 * here accept_len + 1).  keep: int32 [batch], host (checked against the last R)
 * or device (clamped to [0, R], DFLASH_FLAG_BAD_ROWS). */
int dflash_target_commit(dflash_target* t, const int32_t* keep, void* stream);

/* Synchronise `stream`; len: host int32 [batch] of committed lengths (or NULL);
 * returns DFLASH_ERR_DEVICE_FLAG with the latched bits in *device_flags. */
int dflash_target_query(dflash_target* t, void* stream, int32_t* len, uint32_t* device_flags);

/* ---------------------------------------------------------------- failure detection
 * (bounded device waits, allocation failures, KV arena guard bands).  The
 * method's description has no counterpart for these: they are the library's
 * own error-handling surface.
 *
 * Time limit of every bounded wait in this context's kernels (mbarrier and
 * cross-CTA counter waits), in nanoseconds; 0 restores the default of 2 s.  A
 * wait that runs out latches DFLASH_FLAG_WAIT_TIMEOUT, its kernel unwinds
 * (in-flight copies land, tensor memory is freed) and the context stays usable
 * once dflash_query_state has returned the flag.  Synchronous; do not call it
 * while a kernel of the context runs. */
int dflash_set_wait_limit(dflash_ctx* ctx, uint64_t limit_ns);

/* Self-test of the bounded waits: launches one kernel on `stream` whose single
 * wait is on an mbarrier that nothing arrives at, so it can only end by running
 * out of the context's wait limit; it then latches DFLASH_FLAG_WAIT_TIMEOUT
 * (read it with dflash_query_state) and returns.  It holds one SM for the
 * length of the limit: set a short one first. */
int dflash_selftest_wait(dflash_ctx* ctx, void* stream);

/* Allocation-failure injection (process-wide test hook): with after >= 0 the
 * after-th next device allocation the library makes (0: the very next one)
 * fails as if the device were out of memory, once -- the call that made it
 * returns DFLASH_ERR_OOM and frees what it had taken; after < 0 disables it.
 * Returns the previous setting (the allocations still to succeed, or -1). */
int64_t dflash_inject_alloc_failure(int64_t after);

/* Synchronise `stream` and check the guard bands of 4096 bytes of 0xA5 on both
 * sides of the KV arena: DFLASH_OK, or DFLASH_ERR_DEVICE_FLAG naming the band
 * and the first byte written where no kernel may write. */
int dflash_check_guards(dflash_ctx* ctx, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
