// Host-side declarations shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dfl {

// Lo-plane offset that marks a GEMM token operand stored as one fp16 plane
// (instead of split bf16, hi + lo planes that many elements apart).
constexpr size_t kF16Plane = ~(size_t)0;

// Launch with programmatic stream serialisation (the kernel may begin while
// the previous kernel in the stream drains; it orders itself with
// griddepcontrol.wait).  pdl_enabled() is false when DFLASH_PDL=0.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kMaxSeg = 32;      // weight segments one GEMM may concatenate
constexpr int kTileRows = 128;   // weight rows per tensor-core tile (MMA M)
constexpr int kTileK = 64;       // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kKeyStride = 16;   // u64 between two argmax key slots (one 128-byte line each)
constexpr int kKeySlots = 32;    // argmax key slots per token (LM-head CTAs spread over them)

// Per-sequence proposer state in device memory (arrays of [batch]).
struct SeqState {
  int32_t* ctx_len;   // committed tokens = position of the anchor (RoPE offset)
  int32_t* kv_len;    // context rows whose K/V are stored ("consumed")
  int32_t* anchor;    // next anchor token
  int32_t* cap;       // KV capacity in token slots (power of two)
  int64_t* kv_base;   // first arena row of the sequence's KV segment
  int32_t* pend_base; // kv_len before the last append = slot of its first row
  int32_t* rblk;      // block rows of the last draft: K_b + 1 (K_b <= K, per sequence)
  // How the target context conditions the draft: ctx_kv = 1 -- every consumed
  // row's K/V in every layer (the block's rows follow at slots kv_len ..);
  // ctx_kv = 0 -- no context keys (the block's rows at slots 0 .. R-1, attention
  // over the block only), and with input fusion u_last [B][H] (fp32) is added to
  // every block row's embedding (null otherwise).
  const float* u_last;
  int32_t ctx_kv;
};

// First KV slot of sequence b's block rows (the context length attention sees).
__host__ __device__ __forceinline__ int block_base(const SeqState& st, int b) { return st.ctx_kv ? st.kv_len[b] : 0; }

// Addressing of the KV arena: rows of head_dim elements; the K (s=0) or V
// (s=1) row of layer l, KV head h, slot p of sequence b is
//   kv_base[b] + ((l * 2 + s) * n_kv + h) * cap[b] + p.
struct KvArena {
  void* base;
  int n_layers, n_kv, head_dim;
};

__host__ __device__ inline int64_t kv_row(const KvArena& a, int64_t base, int cap, int l, int s, int h, int p) {
  return base + ((int64_t)(l * 2 + s) * a.n_kv + h) * (int64_t)cap + p;
}

// One GEMM Y[t][n] = sum_k X[t][k] W[n][k] over concatenated weight segments.
struct GemmSegs {
  const void* w[kMaxSeg];
  int rows[kMaxSeg];
  int n;
};

// Epilogues of the tensor-core GEMM.  Split-K partial sums always go to
// ws[split][t][n]; for every epilogue but EPI_PARTIAL the CTAs of a tile (or
// gate/up tile pair) meet on a counter once all partials have landed, and each
// then sums, in split order, and finishes its own slice of the tokens.
enum GemmEpi : int {
  EPI_PARTIAL = 0,  // partial sums only (a separate kernel reduces them)
  EPI_ARGMAX = 1,   // LM head, one split: packed (logit, lowest id) keys; the last CTA writes the ids
  EPI_QKV = 2,      // q -> RoPE -> q_out; k -> RoPE -> KV slot; v -> KV slot (block rows)
  EPI_RESID = 3,    // h += y; per-tile sums of squares and bf16(h * gain) of the new rows
  EPI_SILU = 4,     // gate/up tile pairs -> silu(gate) * up -> a_out
  EPI_Y_SS = 5,     // y -> optional fp32 rows; per-tile sums of squares and bf16(y * gain)
  EPI_CTXKV = 6,    // context rows: k -> RoPE -> KV slot; v -> KV slot (every layer)
};

// What a tensor-core GEMM's epilogue needs: shape, split-K partials, and the
// inputs and outputs of each epilogue kind (shared by the stand-alone GEMM
// kernel's instances).
struct EpiArgs {
  int epi;                      // GemmEpi
  int x_planes;                 // token operand planes: 1 (plain bf16) or 2 (split hi + lo, see split_bf16)
  int op16;                     // 1: one fp16 plane against fp16 weights (x_planes 1); operands written as fp16
  int M;                        // tokens
  int N;                        // output columns (sum of segment rows)
  int nkb;                      // 64-wide k-blocks of K
  int splits;                   // split-K factor
  int nseg;
  int seg_rows[kMaxSeg];
  int seg_tile0[kMaxSeg + 1];   // prefix sums of 128-row tiles
  int seg_col0[kMaxSeg + 1];    // prefix sums of rows (= output column offsets)
  float* ws;                    // [splits][M][N] fp32 partial sums
  uint32_t* flags;

  // RMSNorm folded in: the token operand holds bf16(h * gain), and the reduced
  // outputs of token t are multiplied by 1/sqrt(ss_t / K + eps), with
  // ss_t = sum_i ss_in[i * ss_ld + t] (ss_in null: no scale; EPI_QKV, EPI_CTXKV,
  // EPI_SILU, EPI_ARGMAX)
  const float* ss_in;
  int n_ss, ss_ld;
  float eps;

  unsigned int* counters;       // arrival / departure counters, zero between launches
  unsigned long long* argmax_keys;
  float* logits;                // EPI_ARGMAX: optional fp32 logits [B][R-1][N] of the mask rows
  int32_t* ids;                 // EPI_ARGMAX: argmax ids [B][R-1]; token t = b*R + j, anchor rows (j = 0) skipped
  float* h;                     // EPI_RESID: residual stream [M][N]; EPI_Y_SS: optional output [M][N]
  float* ss_out;                // EPI_RESID / EPI_Y_SS: [n_tiles][M] per-tile sums of squares
  __nv_bfloat16* xn_out;        // EPI_RESID / EPI_Y_SS: optional split bf16 of v * xn_gain [2][M][N], the next norm's input
  const __nv_bfloat16* xn_gain; // [N] gain of that norm
  __nv_bfloat16* q_out;         // EPI_QKV: [M][q rows]
  __nv_bfloat16* a_out;         // EPI_SILU: split bf16 [2][M][I]
  SeqState st;
  KvArena kv;
  const uint64_t* rope_turns;       // RoPE frequencies [head_dim / 2]
  int layer, R;                 // EPI_QKV / EPI_ARGMAX: layer, block rows per sequence
  const int32_t* rows;          // EPI_CTXKV: valid rows per sequence
  int rows_max, t0;             // EPI_CTXKV: padded rows per sequence, first flat row of this chunk
  int half_tiles;               // EPI_SILU: tiles per gate (or up) segment
  // EPI_SILU: tiles alternate between the two segments (tile 2i = gate rows
  // 128i.., tile 2i+1 = up rows 128i..) so that the two CTAs of a pair are at
  // most t_tiles apart in launch order and so resident together
  int interleave2;
  // EPI_QKV with the pending context rows of an append (fuse_ctx = 1): token
  // tile 0 (BN rows) holds the m_blk block rows, token tile 1 (the next BN rows)
  // the m_ctx = B * rows_max context rows u of the append (rows, rows_max as for
  // EPI_CTXKV), whose folded norm sums are ss_ctx[i * ss_ctx_ld + row]; their
  // K/V go to slots pend_base[b] + rr, their Q is not written
  int fuse_ctx, m_blk, m_ctx;
  const float* ss_ctx;
  int ss_ctx_ld;
};

// Parameters of the stand-alone tensor-core GEMM (passed by value as a grid constant).
struct TcGemmParams : EpiArgs {
  CUtensorMap tm_w[kMaxSeg];
  CUtensorMap tm_x;             // tokens [x_planes][M][K] bf16 (3D map, box 64 x BN x 1)
  CUtensorMap tm_x2;            // fuse_ctx: the context rows [x_planes][m_ctx][K], same box
  int BN;                       // token tile (MMA N = x_planes * BN, multiple of 16, <= 256)
  int tt;                       // token tiles per CTA (weights staged once, one MMA per tile)
  int stages;
  int kb_per_split;             // 64-wide k-blocks per split
  int direct;                   // 1: one split; the epilogue reads the sums from tensor memory
                                //    (no partials in ws, no counters)
  int wpair;                    // 1 (EPI_SILU, direct, tt = 1): CTA y computes gate tile y and up
                                //    tile y (two weight boxes per stage, two accumulators)
  int p_tiles, p_ttiles;        // persistent instance: tiles, token tiles per weight tile
  int late_trigger;             // 1: the dependent launch is released after the dependency wait
                                //    (its pre-wait reads may then see every earlier kernel's writes)
};


// Parameters of the tensor-core attention (bf16, head_dim 128).
struct AttnTcParams {
  CUtensorMap tm_kv;            // KV arena as [rows, 128] bf16, 64 x 64 boxes, 128-byte swizzle
  const __nv_bfloat16* q;       // [M, n_q * 128], rotated queries
  __nv_bfloat16* o;             // split bf16 [2][M][n_q * 128], M = B * R
  float* part_o;                // [B, n_kv, n_splits, rows_pad, 128] (n_splits > 1)
  float* part_lse;              // [B, n_kv, n_splits, rows_pad], log2 domain
  SeqState st;
  KvArena kv;
  int layer, R, n_q, n_kv, G;   // G = n_q / n_kv query heads per KV head
  int rows, rows_pad, n_qtiles, n_splits;
  float scale_log2;             // d^-1/2 * log2(e)
  uint32_t* flags;
  size_t o_plane;               // elements between the hi and lo planes of o (M * n_q * 128)
};
// tcgen05 attention (head_dim 128, 128 % G == 0): query tiles of JT = 128 / G
// block rows x G heads, loaded through tm_q = q viewed as [M][n_q][128] with
// 64 x G x JT boxes; partials in the same layout as AttnTcParams
// (row gq * R + j, rows_pad >= G * R).
struct AttnUParams {
  CUtensorMap tm_kv;            // KV arena as [rows, 128] bf16, 64 x 64 boxes, 128-byte swizzle
  CUtensorMap tm_q;             // rotated queries, 3-D view, 128-byte swizzle
  __nv_bfloat16* o;             // split bf16 [2][M][n_q * 128]
  // partials of sequence b (S_b > 1 splits, first partial group pg_b): row
  // ((pg_b * n_kv + hk * S_b) + split) * rows_pad + rq of [groups * n_kv * rows_pad][128]
  float* part_o;
  float* part_lse;              // [groups * n_kv * rows_pad], log2 domain
  SeqState st;
  KvArena kv;
  int layer, R, n_q, n_kv, G, JT;
  int rows_pad, n_qtiles;
  int n_splits;                 // grid mode: every sequence's split count (pg_b = b * n_splits)
  int causal;                   // 1: block row j sees positions <= block_base + j only
  const int32_t* seq_order;     // grid mode: sequence of grid row z (longest context first), or null: z
  // persistent schedule (null work: grid mode, one item per CTA)
  const int32_t* work;          // units (b << 8 | split) in processing order
  const int32_t* seq_split;     // [B][2]: S_b, pg_b
  const int32_t* n_units;       // number of units
  uint32_t* item_ctr;           // this launch's item counter (zero at launch)
  float scale_log2;
  uint32_t* flags;
  size_t o_plane;
  // grid mode: the predecessor (the layer's QKV GEMM) released this launch
  // after its own dependency wait and writes no K/V below block_base, so the
  // first K/V tiles below it may be loaded before this kernel's wait
  int early_kv;
};
size_t attn_umma_smem_bytes();
cudaError_t launch_attention_umma(const AttnUParams& p, int B, int grid, cudaStream_t s);
// seq_split null: every sequence has S splits, partial group b * S; else the
// per-sequence S_b and pg_b of the persistent schedule (S the largest expected,
// sequences with one split are skipped: their output is written directly)
cudaError_t launch_attn_merge(const float* part_o, const float* part_lse, int n_kv, int S, int rows, int rows_pad,
                              int R, int G, int n_q, __nv_bfloat16* o, size_t o_plane, int B, cudaStream_t s,
                              uint32_t* flags, const int32_t* seq_split = nullptr);
// The attention schedule of one draft (all layers): order[k] = the sequence of
// rank k by decreasing context (ties by index); for the persistent kernel, per sequence b,
// T_b = ceil(L_b / 64) tiles of the live length L_b, S_b = ceil(T_b / c) KV
// splits (at most s_max, none empty) with c >= chunk grown until the splits of
// multi-split sequences fit max_groups partial groups; units (b, split) ordered
// by tiles per split, most first; the per-layer item counters zeroed.
void launch_attn_plan(SeqState st, int B, int chunk, int s_max, int max_groups, int32_t* work, int32_t* seq_split,
                      int32_t* n_units, int32_t* order, uint32_t* ctrs, int n_ctrs, cudaStream_t s);
int attn_plan_max_batch();   // largest batch one plan CTA takes (shared-memory tables)
size_t attn_tc_smem_bytes();
cudaError_t launch_attention_tc(const AttnTcParams& p, int n_consumer_warps, int B, cudaStream_t s);
void launch_argmax_finalize(unsigned long long* keys, int rows, int32_t* ids, cudaStream_t s);

size_t gemm_tc_smem_bytes(int BN, int stages, int x_planes, int tt, int w_boxes = 1);
size_t gemm_tc_persist_smem_bytes(int BN, int stages, int w_boxes);
cudaError_t launch_gemm_tc_persist(const TcGemmParams& p, int grid, cudaStream_t s);
// epi / by_epi: the split-K one-tile GEMM has one instance per epilogue (the
// one in p.epi); -1 / false take the instance that reads it from the parameters
int gemm_tc_resident_ctas(int tt, bool direct, size_t smem, int n_cols, int epi = -1);
cudaError_t launch_gemm_tc(const TcGemmParams& p, int n_tiles, int splits, int t_tiles, int stages,
                           cudaStream_t s, bool by_epi = true);

template <typename T>
cudaError_t launch_gemm_simt(const T* x, int ldx, int M, int K, const GemmSegs& segs, int N, float* ws,
                             int splits, int k_per_split, cudaStream_t s);

// ---- element-wise and epilogue kernels (dtype T = float or __nv_bfloat16)
template <typename T>
void launch_embed(const T* E, const int32_t* anchor_in, SeqState st, int B, int R, int H, int V, int mask_id,
                  float* h, uint32_t* flags, float* ss, const int32_t* kseq, cudaStream_t s);
template <typename T>
void launch_embed_norm(const T* E, const int32_t* anchor_in, SeqState st, int B, int R, int H, int V, int mask_id,
                       const T* gain, float eps, float* h, T* xn, size_t lo_plane, uint32_t* flags,
                       const int32_t* kseq, cudaStream_t s, const int32_t* tokens = nullptr);
template <typename T>
void launch_epi_residual_norm(const float* ws, int splits, int M, int H, float* h, const T* gain, float eps, T* y,
                              int R, int sel_K, cudaStream_t s);
template <typename T>
void launch_rmsnorm(const float* h, const T* gain, T* out, int rows, int H, float eps, int sel_R, int sel_K,
                    cudaStream_t s);
template <typename T>
void launch_epi_qkv(const float* ws, int splits, int M, int R, int layer, int n_q, int n_kv, int d,
                    const uint64_t* rope_turns, SeqState st, KvArena kv, T* q_out, uint32_t* flags, cudaStream_t s);
void launch_epi_residual(const float* ws, int splits, int M, int H, float* h, cudaStream_t s);
template <typename T>
void launch_epi_silu(const float* ws, int splits, int M, int I, T* out, cudaStream_t s);
template <typename T>
void launch_epi_fcnorm(const float* ws, int splits, int M, int H, const T* gain, float eps, T* u,
                       cudaStream_t s);
template <typename T>
void launch_epi_ctxkv(const float* ws, int splits, int Mc, int t0, int rows_max, const int32_t* rows,
                      int n_layers, int n_kv, int d, const uint64_t* rope_turns, SeqState st, KvArena kv,
                      uint32_t* flags, cudaStream_t s);
void launch_rows_prep(const int32_t* rows_in, int rows_max, int B, int32_t* rows_out, uint32_t* flags,
                      cudaStream_t s);
void launch_mask_drafts(int32_t* drafts, SeqState st, int B, int K, cudaStream_t s);
void launch_append_commit(const int32_t* rows, SeqState st, int B, cudaStream_t s);
template <typename T>
void launch_ulast(const T* u, size_t lo_plane, const float* ss, int n_ss, int ss_ld, int t0, int Mc,
                  const int32_t* rows, int rows_max, int B, int H, float eps, float* u_last, cudaStream_t s);
void launch_argmax(float* ws, int splits, int rows, int V, int32_t* ids, cudaStream_t s);
void launch_lm_argmax(const float* ws, int splits, int M, int V, int R, const float* ss, int n_ss, int ss_ld, int H, float eps,
                      float* logits, unsigned long long* keys, unsigned int* counter, int32_t* ids, int n_mask,
                      cudaStream_t s);
void launch_accept(const int32_t* drafts, const int32_t* targets, int B, int K, int V, SeqState st,
                   int32_t* accept_len, int32_t* next_anchor, uint32_t* flags, cudaStream_t s);
void launch_plant(const int32_t* d, const int32_t* L, const int32_t* fill, int B, int K, int V, int32_t* g,
                  int32_t* counter, int n_plans, cudaStream_t s);
void launch_arena_copy(void* arena, size_t esz, int head_dim, int64_t src_row0, int64_t dst_row0, int src_cap,
                       int dst_cap, int groups, int rows, cudaStream_t s);
void launch_set_seq(SeqState st, int b, int64_t kv_base, int cap, cudaStream_t s);
void launch_reset_state(SeqState st, int B, cudaStream_t s);

template <typename T>
void launch_attention(const T* q, SeqState st, KvArena kv, int layer, int B, int R, int n_q, int n_kv, int d,
                      T* o, uint32_t* flags, cudaStream_t s, int causal = 0);
// target forward: greedy ids are per row; features of a layer copied out; commit
void launch_feat_copy(const float* h, int M, int H, int n_feat, int fi, __nv_bfloat16* feats, cudaStream_t s);
void launch_target_commit(const int32_t* keep, SeqState st, int B, uint32_t* flags, cudaStream_t s);

// The failure-detection self-test kernel (one wait that nothing ends; it runs
// out after the context's wait limit and latches DFLASH_FLAG_WAIT_TIMEOUT).
cudaError_t launch_wait_selftest(uint32_t* flags, cudaStream_t s);

// bf16 -> fp16 copy of n elements; *bad |= 1 where a value is outside fp16's range.
cudaError_t launch_bf16_to_f16(const __nv_bfloat16* x, void* y, size_t n, uint32_t* bad, cudaStream_t s);

}  // namespace dfl
