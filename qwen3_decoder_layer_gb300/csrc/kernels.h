// Internal launch interface between the host runtime (runtime.cpp) and the
// CUDA kernels.  Plain structs of device pointers and sizes; no torch types.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

enum DType { DT_F32 = 0, DT_BF16 = 1 };
enum WFmt { W_DT = 0, W_U8 = 1 };  // weights in the model dtype, or affine int8 codes
enum Epi { EPI_STORE = 0, EPI_STORE_F32 = 1, EPI_RESIDUAL = 2, EPI_SWIGLU = 3,
           EPI_STORE_RF32 = 4 /* rounded to the model dtype, stored as fp32 (output head) */,
           EPI_QKROPE = 5 /* q|k|v rows: per-head q/k RMSNorm + RoPE, q to q_out, k and v to the caches */ };

struct LaunchCtx {
  cudaStream_t stream;
  bool pdl;      // programmatic dependent launch attribute on every launch
  int num_sms;
};

// h_out = R(h_in + pend) (pend may be NULL: h_out = h_in); y = RMSNorm(h_out) * gain.
// h_out may alias h_in.  y may be NULL.  One block per row.
struct NormArgs {
  const void* h_in;
  const void* pend;
  void* h_out;
  void* y;
  const void* gain;
  int rows, hidden;
  float eps;
};
cudaError_t launch_add_rmsnorm(const LaunchCtx& c, int dt, const NormArgs& a);

// Per-head RMSNorm of q and k, RoPE of q and k at each row's position, and
// the cache append of k and v.  q_out dt [T, H, D]; caches: layer base of
// sequence 0, sequence stride `seq_stride` elements, [KV][capacity][D] inside.
struct QkRopeArgs {
  const void* qkv;
  int T, H, KV, D;
  void* q_out;
  void* kcache;
  void* vcache;
  long long seq_stride;
  int capacity;
  const void* q_gain;
  const void* k_gain;
  const float* cos_t;  // [capacity][D]
  const float* sin_t;
  const int* row_seq;  // [T]
  const int* row_pos;  // [T]
  float eps;
  // bf16 models: the same table as bf16 pairs (cos | sin << 16) of the D/2
  // frequencies, [capacity][D/2] (every cos / sin value is a bf16 value)
  const uint32_t* cs_bf16;
};
cudaError_t launch_qk_rope_cache(const LaunchCtx& c, int dt, const QkRopeArgs& a);

// Weight-streaming GEMV for a few rows: out[t, n] = sum_k x[t, k] W[n, k].
struct GemvArgs {
  int T;       // rows of x (shared weights, 1..4) or slots (gather mode)
  int K;       // input features
  int N;       // outputs per row (EPI_SWIGLU: pairs; the weight has 2N rows, gate first)
  const void* w;
  const void* scale;   // W_U8 only: bf16 [rows, K/group]
  const void* bias;
  int group;
  // gather mode (MoE experts): slot b uses the matrix w + slot_expert[b] * w_stride
  // and x row b / slot_div.  slot_expert == NULL: one matrix shared by all T rows.
  const int* slot_expert;
  long long w_stride;
  int slot_div;
  int x_rows;          // rows of x staged in shared memory
  const void* x;       // dt [x_rows, K]
  int epilogue;        // Epi
  void* out;
  int ldo;
};
cudaError_t launch_gemv(const LaunchCtx& c, int dt, int wfmt, const GemvArgs& a);
size_t gemv_smem_bytes(const GemvArgs& a);

// Tiled CUDA-core GEMM C[M, N] = A[M, K] B[N, K]^T with fp32 accumulation.
// Grouped mode (tile_start != NULL): rows are sorted by group; group g owns
// sorted rows row_off[g] .. row_off[g] + row_cnt[g] and its own weight matrix
// w + g * w_stride; tile_start is the prefix sum of its row tiles.
struct GemmArgs {
  int M, N, K;
  const void* a;
  int lda;
  const int* a_rows;   // A row of output row m (NULL = m)
  const void* w;
  const void* scale;
  const void* bias;
  int group;
  long long w_stride;
  const int* tile_start;
  const int* row_off;
  const int* row_cnt;
  int n_groups;
  int max_tiles;       // grouped: upper bound of row tiles (grid size)
  int epilogue;
  void* out;
  int ldo;
  const int* c_rows;   // output row of row m (NULL = m)
};
cudaError_t launch_gemm_simt(const LaunchCtx& c, int dt, int wfmt, const GemmArgs& a);
int gemm_simt_tile_m();

// Skinny GEMM for 1..64 rows (batched decode with int8 or fp32 weights):
// out[M, N] = a[M, K] w[N, K]^T, K split over up to 8 CTAs; each split's
// partial tile goes to its own slice of an fp32 workspace (gemm_skinny_ws_floats
// floats) and the last CTA of a tile sums the slices in order; counters (one
// per 64 output columns) are zero between calls.
struct SkinnyArgs {
  int M, N, K;
  const void* a;
  int lda;
  const void* w;
  const void* scale;
  const void* bias;
  int group;
  int epilogue;
  void* out;
  int ldo;
  float* ws;
  int* counters;
  int ktiles_per_split;  // set by the launcher
  int* err;              // device error flag (tensor-core variant's bounded waits)
};
bool gemm_skinny_supported(int M, int N, int K);
size_t gemm_skinny_ws_floats(int M, int N, int epilogue);
int gemm_skinny_tiles(int N);
cudaError_t launch_gemm_skinny(const LaunchCtx& c, int dt, int wfmt, SkinnyArgs a);
// Tensor-core form for affine int8 weights, bf16 activations and 1..32 rows
// (integer codes through tcgen05.mma, group scale and bias in the epilogue);
// groups must be whole multiples of 64.  Same arguments and workspace.
bool gemm_w8_tc_supported(int M, int N, int K, int group, int epilogue);
cudaError_t launch_gemm_w8_tc(const LaunchCtx& c, SkinnyArgs a);

// Tensor-core (tcgen05 / TMEM / TMA) bf16 GEMM: out[M, N] = a[M, K] w[N, K]^T
// with EPI_STORE, EPI_RESIDUAL (out += R(.), in place) or EPI_SWIGLU (w has
// 2N rows, gate first).  Dense bf16 weights only.
struct GemmTcArgs {
  int M, N, K;
  const void* a;
  int lda;
  const void* w;
  void* out;
  int ldo;
  int epilogue;
  int* err;
  // grouped mode (tile_start != NULL): rows sorted by group; group g owns rows
  // row_off[g] .. + row_cnt[g] of a, its weight rows start at g * w_group_rows
  // of w, tile_start is the prefix sum of its 128-row tiles (tile_start[n_groups]
  // = total); output row of sorted row m is c_rows[m] (NULL = m).
  const int* tile_start;
  const int* row_off;
  const int* row_cnt;
  int n_groups;
  int max_tiles_m;       // upper bound of tile_start[n_groups] (grid size)
  long long w_group_rows;
  long long w_rows_total;
  const int* c_rows;
  // EPI_QKROPE: the head layout, gains, RoPE table, caches and row positions
  // (rope.qkv unused: the q|k|v rows never leave the kernel)
  QkRopeArgs rope;
  // split k (one row tile, EPI_STORE / RESIDUAL / SWIGLU): splits > 1 ranges
  // of k-steps, each item's fp32 accumulator to part [splits][M][N/ncol*256];
  // launch_gemm_tc_reduce then adds them in range order and applies the epilogue
  int splits;
  float* part;
};
bool gemm_tc_supported(int M, int N, int K, int epilogue);
// split k for GEMMs of one 128-row tile with few column tiles: the number of
// k ranges (1 = none), the partial-tile floats they need, and the reduction
int gemm_tc_splits(int M, int N, int K, int epilogue, int num_sms);
size_t gemm_tc_part_floats(int M, int N, int epilogue, int splits);
cudaError_t launch_gemm_tc_reduce(const LaunchCtx& c, const GemmTcArgs& a);
// the q|k|v GEMM with the fused q/k RMSNorm + RoPE + cache-append epilogue
bool gemm_tc_qkrope_supported(int M, int H, int KV, int D);
cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmTcArgs& a);

// Attention over the cache.  Work: query blocks (rows of one sequence at
// consecutive positions) x key chunks x kv heads; each item writes a partial
// (max, sum, unnormalised output) and the last item of a (query block, kv
// head) combines them.
struct AttnQBlock {
  int seq, row0, nrows, pos0, n_chunks, part_base;
  int seg_row0, seg_pos0, seg_n, pad;  // the block's sequence rows in this call (new keys)
};
struct AttnItem {
  int qb, chunk;
};
struct AttnArgs {
  const void* q;
  const void* kc;
  const void* vc;
  long long seq_stride;
  int capacity, H, KV, D;
  float scale;
  const AttnQBlock* qblocks;
  const AttnItem* items;
  const int* n_items;  // device scalar
  int chunk;           // keys per chunk
  int nq_max;          // query vectors per block (rows x G), partial stride
  float* part_o;       // [parts * KV][nq_max][D]
  float* part_ml;      // [parts * KV][nq_max][2]
  int* counters;       // [n_qblocks * KV], zero between calls
  void* out;           // dt [T, H * D]
  int grid_x;          // persistent grid width
};
cudaError_t launch_attention_prefill(const LaunchCtx& c, int dt, const AttnArgs& a);
// chunk size and query-vector limit the prefill attention kernel is built for
int attn_prefill_chunk();
int attn_prefill_nq_max();

// Tensor-core (tcgen05) causal attention for bf16 prefill: one CTA per
// (128-row query tile, q head); qblocks are 128-row tiles of one sequence.
// q: bf16 [T, H * D] after RMSNorm + RoPE; kc / vc: the layer's cache of
// sequence 0, sequences seq_stride elements apart, [KV][capacity][D] inside.
struct AttnTcArgs {
  const AttnQBlock* qblocks;
  int n_qblocks;
  int T, H, KV, D, capacity, max_seqs;
  long long seq_stride;
  const void* q;
  const void* kc;
  const void* vc;
  void* out;           // bf16 [T, H * D]
  float scale_log2;    // log2(e) / sqrt(D)
  int* err;
};
bool attn_tc_supported(int D);
int attn_tc_rows();
cudaError_t launch_attn_tc(const LaunchCtx& c, const AttnTcArgs& a);

// MoE router: softmax over all experts, top-k by logit (ties to the lower
// index), optional renormalisation; per-expert counts (atomics) if counts != NULL.
struct RouterArgs {
  const float* logits;  // [T, E]
  int T, E, k, norm;
  int* idx;             // [T, k]
  float* w;             // [T, k]
  int* counts;          // [E] (zeroed by the caller's scan kernel of the previous use)
};
cudaError_t launch_router_topk(const LaunchCtx& c, const RouterArgs& a);
// Router logits of many rows, fp32 and unrounded: out[t][e] = sum_k y[t][k] W[e][k]
// (y [M][ldy] and W [E][K] in the model dtype).  The k range may be split:
// `part` holds the partial tiles ([max_splits][M][E] floats), `counters` one
// int per 32 x 128 output tile, zero between calls (the kernel restores it);
// part == NULL computes each output in one range.
struct RouterLogitsArgs {
  int M, E, K;
  const void* y;
  int ldy;
  const void* w;
  float* out;
  int ldo;
  float* part;
  int* counters;
  int max_splits;
};
bool router_logits_supported(int dt, int E, int K);
cudaError_t launch_router_logits(const LaunchCtx& c, int dt, const RouterLogitsArgs& a);
constexpr int kRouterMaxSplits = 8;
int router_logits_tiles(int M, int E);

// Exclusive scan of expert counts -> row offsets and tile prefix; zeroes cursors.
struct MoeScanArgs {
  int* counts;   // [E] read, then zeroed for the next call
  int E, bm;
  int* row_off;     // [E]
  int* row_cnt;     // [E]
  int* tile_start;  // [E + 1]
  int* cursor;      // [E] zeroed
};
cudaError_t launch_moe_scan(const LaunchCtx& c, const MoeScanArgs& a);

// Place each (token, slot) at its expert's next free sorted row.
struct MoeScatterArgs {
  const int* idx;
  int T, k;
  const int* row_off;
  int* cursor;
  int* sorted_tok;  // [T k] token of each sorted row
  int* sorted_src;  // [T k] flat (token * k + slot) of each sorted row
};
cudaError_t launch_moe_scatter(const LaunchCtx& c, const MoeScatterArgs& a);

// Gather rows into sorted order: out[r] = x[rows[r]] (dt, row length K).
struct MoeGatherArgs {
  const void* x;
  const int* rows;
  int n, K;
  void* out;
};
cudaError_t launch_moe_gather(const LaunchCtx& c, int dt, const MoeGatherArgs& a);

// pend[t] = R(sum_i w[t, i] z[t k + i]) in fp32; written to `out`, or, when
// h != NULL, added to the residual in place (h = R(h + pend)) with the row's
// sum of squares added to sumsq_out[t] (which must be zero beforehand).
struct MoeCombineArgs {
  const void* z;
  const float* w;
  int T, k, hidden;
  void* out;
  void* h;
  double* sumsq_out;
};
cudaError_t launch_moe_combine(const LaunchCtx& c, int dt, const MoeCombineArgs& a);

// ---------------------------------------------------------------- decode path (T <= 4)
enum Prologue { PRO_X = 0, PRO_FULL = 1, PRO_SUMSQ = 2 };

// GEMV whose weight rows stream through per-warp shared-memory rings filled by
// TMA bulk copies; the first copies are issued before waiting on the previous
// kernel.  Prologues: PRO_X: x given (dt [T, K]); PRO_FULL: h = R(x + pend)
// (pend optional), block 0 stores h, RMSNorm with a block reduction, block 0
// also zeroes sumsq_zero[0 .. sumsq_zero_n); PRO_SUMSQ: RMSNorm of h from the
// precomputed sum of squares sumsq_in[t].  EPI_RESIDUAL updates out (= h) in
// place and adds the squares of the updated rows to sumsq_out[t].
struct Gemv2Args {
  int T, K, N;
  const void* w;
  const void* scale;
  const void* bias;
  int group;
  int prologue;
  const void* x;
  const void* pend;
  void* h;
  const void* gain;
  float eps;
  const double* sumsq_in;
  double* sumsq_zero;
  int sumsq_zero_n;
  int epilogue;
  void* out;
  int ldo;
  double* sumsq_out;
  int stages;          // ring slots per warp
  int nwarps;          // warps per block
  int* err;
  const void* pf;      // L2 prefetch (before the wait) of the next kernel's operand
  size_t pf_bytes;
  void* x_out;         // PRO_SUMSQ (optional): block 0 also stores the normalised rows [T][K]
};
cudaError_t launch_gemv2(const LaunchCtx& c, int dt, int wfmt, const Gemv2Args& a);
// Ring slots per warp (return value, 0 = does not fit) and warps per block
// (*nwarps) for a linear of K inputs at T rows; `coresident` keeps a block to
// half an SM so that two kernels' blocks share it.
int gemv2_plan(int dt, int wfmt, int T, int K, int group, bool pair, int* nwarps, bool coresident);

// Decode attention with the q/k RMSNorm, RoPE and cache append fused in:
// items as in AttnArgs; K/V chunks stream into a shared-memory ring by TMA;
// keys appended in this call are computed from qkv inside the kernel (the
// item that owns the row also writes them to the cache).
struct AttnDecArgs {
  const void* qkv;
  int H, KV, D;
  const void* q_gain;
  const void* k_gain;
  const float* cos_t;
  const float* sin_t;
  float eps;
  void* kc;
  void* vc;
  long long seq_stride;
  int capacity;
  int n_seqs;          // sequences in the cache (its outer extent)
  float scale;
  const AttnQBlock* qblocks;
  const AttnItem* items;
  const int* n_items;
  float* part_o;
  float* part_ml;
  int nq_max;
  int* counters;
  void* out;
  int grid_x;
  int nq;              // largest query-vector count (rows x G) of any query block, <= attn_decode2_nq_max()
  int runs;            // 1: blocks walk contiguous item ranges (more items than blocks); 0: one item per block
  int cluster;         // > 1: one query block per cluster of this many CTAs (grid_x = cluster x query blocks),
                       // partials merged through distributed shared memory; items and partial buffers unused
  int* err;
  const void* pf;      // L2 prefetches (before the wait) of the next kernels' operands
  size_t pf_bytes;
  const void* pf2;
  size_t pf2_bytes;
};
cudaError_t launch_attn_decode2(const LaunchCtx& c, int dt, const AttnDecArgs& a);
int attn_decode2_chunk(int dt);
int attn_decode2_nq_max();
// Cluster variant: keys a cluster of `cl` CTAs takes for nq query vectors, and
// how many such clusters (grid cl * clusters_x by kv) can be resident at once.
int attn_decode_cluster_keys(int dt, int nq, int cl);
int attn_decode_cluster_capacity(int dt, int D, int nq, int cl, int kv, int clusters_x);


// Embedding rows: out[t] = table[ids[t]] (dt rows of `hidden`); ids on the device.
struct EmbedArgs {
  const void* table;
  const int* ids;
  int n, hidden;
  void* out;
};
cudaError_t launch_embed_gather(const LaunchCtx& c, int dt, const EmbedArgs& a);

// L2 normalisation of one dt row of `hidden` into out, each step rounded to
// the model dtype: sq = R(v v), ss = R(sum sq), n = R(sqrt ss), out = R(v / n).
struct L2PoolArgs {
  const void* row;
  int hidden;
  void* out;
};
cudaError_t launch_l2_pool(const LaunchCtx& c, int dt, const L2PoolArgs& a);

// One CTA waits on an mbarrier that nothing completes, with the bounded wait
// every kernel here uses (mbar_wait); it gives up after its limit, records
// kWaitProbeCode in *err and returns.
constexpr int kWaitProbeCode = 99;
cudaError_t launch_wait_probe(cudaStream_t s, int* err);

// out = RMSNorm(h) * gain with the sum of squares of each row precomputed.
struct NormApplyArgs {
  const void* h;
  const double* sumsq;
  const void* gain;
  void* out;
  int T, hidden;
  float eps;
};
cudaError_t launch_norm_apply(const LaunchCtx& c, int dt, const NormApplyArgs& a);

// Shared launch helper: cudaLaunchKernelEx with the PDL attribute when asked.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, const LaunchCtx& c,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = c.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace q3
