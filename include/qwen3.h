/*
 * qwen3.h -- C ABI of the GB300 (sm_103a) Qwen3 decoder-stack forward.
 *
 * What it computes (page titles as the pages give them):
 *   maya2_mlx/backbone.py, class Backbone, `forward`: per layer
 *     h = h + pend (one rounding); y = RMSNorm(h); qkv = y @ [Wq;Wk;Wv]^T;
 *     per-head RMSNorm of q and k; RoPE in fp32 on a cos/sin table (one
 *     rounding); append k (post-RoPE) and v to a static KV cache; GQA attention
 *     over keys 0..pos with an fp32 softmax (one rounding); h = h + o_proj(a);
 *     y2 = RMSNorm(h); pend = down(silu(g) * u) with silu in fp32 rounded once;
 *     and after the last layer out = RMSNorm(h + pend).
 *   @mlx-bun/inference qwen3-moe.ts, `Qwen3MoeSparseMoeBlock.forward`: for MoE
 *     layers the MLP is replaced by router softmax over all experts, top-k,
 *     renormalisation (norm_topk_prob) and a weighted sum of SwiGLU experts.
 *
 * Conventions
 *   - Every device pointer is a plain CUDA device address on the device that
 *     was current at qwen3_create.  Tensors are dense, row-major, contiguous.
 *   - "dt" is the model dtype: fp32 (QWEN3_DTYPE_F32) or bf16 (QWEN3_DTYPE_BF16).
 *   - Linear weights are nn.Linear [out, in] row-major.  The q|k|v rows and
 *     the gate|up rows are concatenated (one fused projection each).
 *   - Streams are cudaStream_t passed as void* (NULL = legacy default stream).
 *     All device work is enqueued on the given stream; nothing synchronises
 *     except qwen3_create, qwen3_destroy and qwen3_profile_read.
 *   - Every call returns a qwen3_status.  Arguments are validated on the host
 *     before any launch or state change; on error the cache, lengths and
 *     outputs are unchanged and qwen3_last_error() says why.
 *   - Weights, inputs and outputs are owned by the caller and must stay alive
 *     (weights: until qwen3_destroy; x/out: until the stream work completes).
 *     The KV cache, RoPE table and workspaces are owned by the library.
 */
#ifndef QWEN3_GB300_H
#define QWEN3_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QWEN3_API __attribute__((visibility("default")))
#else
#define QWEN3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QWEN3_OK = 0,
  QWEN3_E_ARG = 1,          /* null pointer, size out of range, bad config field */
  QWEN3_E_DTYPE = 2,        /* dtype other than fp32 / bf16 (Backbone.__init__ raises the same) */
  QWEN3_E_CAPACITY = 3,     /* a position would reach or pass `capacity` (Backbone.forward raises) */
  QWEN3_E_POSITION = 4,     /* rows of a sequence do not continue its cache contiguously */
  QWEN3_E_SEQ = 5,          /* sequence id outside [0, max_seqs) or rows of a sequence split */
  QWEN3_E_OOM = 6,          /* device allocation failed */
  QWEN3_E_CUDA = 7,         /* a CUDA runtime call failed (message in qwen3_last_error) */
  QWEN3_E_UNSUPPORTED = 8,  /* a valid but unimplemented combination */
  QWEN3_E_DEVICE = 9        /* no usable CUDA device / wrong architecture */
} qwen3_status;

#define QWEN3_DTYPE_F32 0
#define QWEN3_DTYPE_BF16 1

#define QWEN3_WEIGHTS_DENSE 0       /* linears stored in dt */
#define QWEN3_WEIGHTS_INT8 1        /* affine int8: W = scale * q + bias per group (see qwen3_linear) */

typedef struct qwen3_handle qwen3_handle;   /* opaque, library-owned */

/* Model and cache shape.  Field names follow the Hugging Face Qwen3 config. */
typedef struct {
  int32_t num_layers;        /* num_hidden_layers */
  int32_t hidden;            /* hidden_size; multiple of 64, <= 8192 */
  int32_t n_heads;           /* num_attention_heads */
  int32_t n_kv_heads;        /* num_key_value_heads; divides n_heads */
  int32_t head_dim;          /* 64 or 128 */
  int32_t intermediate;      /* intermediate_size of dense MLP layers; multiple of 64 */
  float rms_eps;             /* rms_norm_eps */
  double rope_theta;         /* rope_theta */
  int32_t capacity;          /* static KV-cache positions per sequence */
  int32_t max_seqs;          /* independent sequences held by the cache */
  int32_t dtype;             /* QWEN3_DTYPE_F32 or QWEN3_DTYPE_BF16 */
  int32_t weight_format;     /* QWEN3_WEIGHTS_DENSE or QWEN3_WEIGHTS_INT8 (every linear but the router) */
  int32_t group_size;        /* int8 group along the input dim (64); multiple of 16 */
  int32_t num_experts;       /* 0 = dense stack */
  int32_t top_k;             /* num_experts_per_tok */
  int32_t moe_intermediate;  /* moe_intermediate_size; multiple of 64 */
  int32_t norm_topk_prob;    /* renormalise the top-k weights to sum to 1 */
  int32_t decoder_sparse_step; /* layer i is MoE iff (i+1) % step == 0 and i not in mlp_only_layers */
  const int32_t* mlp_only_layers; /* optional list of dense layers in a MoE stack (copied at create) */
  int32_t n_mlp_only_layers;
} qwen3_config;

/* One linear layer.  Dense: `w` is dt [out, in]; scale = bias = NULL.
 * Int8 (weight_format QWEN3_WEIGHTS_INT8): `w` is uint8 codes [out, in];
 * `scale` and `bias` are bf16 [out, in / group_size]; the weight is
 * W[o, i] = scale[o, i/group] * w[o, i] + bias[o, i/group], dequantised in
 * fp32 inside the kernels (maya2_mlx/backbone.py keeps fused exports quantised
 * with the same groups as the parts). */
typedef struct {
  const void* w;
  const void* scale;
  const void* bias;
} qwen3_linear;

/* Borrowed device pointers of one decoder layer.  The norm gains, the router
 * and every linear's w must be 16-byte aligned (a misaligned or missing one
 * makes qwen3_create return QWEN3_E_ARG). */
typedef struct {
  const void* in_norm;       /* dt [hidden]  input_layernorm gain */
  const void* post_norm;     /* dt [hidden]  post_attention_layernorm gain */
  const void* q_norm;        /* dt [head_dim] */
  const void* k_norm;        /* dt [head_dim] */
  qwen3_linear qkv;          /* [(n_heads + 2 n_kv_heads) head_dim, hidden], rows q | k | v */
  qwen3_linear o;            /* [hidden, n_heads head_dim] */
  qwen3_linear gate_up;      /* dense layers: [2 intermediate, hidden], rows gate | up */
  qwen3_linear down;         /* dense layers: [hidden, intermediate] */
  const void* router;        /* MoE layers: dt [num_experts, hidden] (the `gate` Linear; never quantised) */
  qwen3_linear exp_gate_up;  /* MoE layers: [num_experts, 2 moe_intermediate, hidden], per expert rows gate | up */
  qwen3_linear exp_down;     /* MoE layers: [num_experts, hidden, moe_intermediate] */
  /* Expert linears follow weight_format like the others: dense dt, or int8
   * codes with bf16 scale / bias [num_experts, rows, in / group_size] (the
   * stacked quantised expert matrices of qwen3-moe.ts QuantizedSwitchLinear). */
} qwen3_layer_weights;

/* Validate a config on the host only (no device work).  QWEN3_OK or the
 * reason it is rejected. */
QWEN3_API qwen3_status qwen3_check_config(const qwen3_config* cfg);

/* Create a stack on the current CUDA device: validates the config and the
 * weight pointers, allocates the KV cache [max_seqs][num_layers][n_kv_heads]
 * [capacity][head_dim] (dt, zeroed) for K and for V, builds the RoPE table on
 * the host (inv_freq_i = theta^(-2i/D) rounded to dt, angle p*inv_freq in
 * double, cos/sin rounded to dt, stored fp32 -- the table Backbone.__init__
 * describes) and uploads it.  `layers` has num_layers entries; the struct
 * array is copied, the device pointers in it are borrowed.  Synchronous. */
QWEN3_API qwen3_status qwen3_create(const qwen3_config* cfg, const qwen3_layer_weights* layers,
                          const void* final_norm, qwen3_handle** out);

/* Free everything the handle owns (synchronises the device first). */
QWEN3_API void qwen3_destroy(qwen3_handle* h);

/* Backbone.reset: zero the cache of sequence `seq_id` (or of all sequences if
 * seq_id == -1) on `stream` and set its length to 0. */
QWEN3_API qwen3_status qwen3_reset(qwen3_handle* h, int32_t seq_id, void* stream);

/* Backbone.forward for T rows that may belong to several sequences.
 *   x         dt [T, hidden] device: input hidden rows (read only)
 *   seq_ids   int32 [T] HOST: sequence of each row; the rows of one sequence
 *             must be consecutive in x
 *   positions int32 [T] HOST: position of each row; the rows of sequence s
 *             must be length(s), length(s)+1, ... in order (contiguous append),
 *             all < capacity
 *   out       dt [T, hidden] device: final-norm hidden states (may alias x)
 * Each row attends to the keys 0..position of its own sequence (causal, keys
 * appended in this call included).  On success the lengths advance at once
 * (host side); the device work completes in stream order. */
QWEN3_API qwen3_status qwen3_forward(qwen3_handle* h, const void* x, int32_t T, const int32_t* seq_ids,
                           const int32_t* positions, void* out, void* stream);

/* One MoE block (qwen3-moe.ts Qwen3MoeSparseMoeBlock.forward) of layer `layer`
 * on given rows, without touching the cache:
 *   y         dt [T, hidden] device: the block input (post-attention RMSNorm output)
 *   out       dt [T, hidden] device: sum_k w_k * expert_k(y), rounded once
 *   topk_idx  int32 [T, top_k] device: chosen experts, by router logit
 *             descending, ties to the lower index
 *   topk_w    fp32 [T, top_k] device: their (renormalised) softmax weights
 * QWEN3_E_ARG if `layer` is not a MoE layer. */
QWEN3_API qwen3_status qwen3_moe_layer(qwen3_handle* h, int32_t layer, const void* y, int32_t T, void* out,
                             int32_t* topk_idx, float* topk_w, void* stream);

/* qwen3_moe_layer for callers that must not allocate.  The paper has no
 * counterpart: this entry point exists for the library's users.
 *
 * qwen3_moe_layer grows the handle's workspace with cudaMalloc when a call
 * needs more room than any earlier one.  Some callers cannot allow that: a
 * serving engine that reserves nearly all of the GPU's memory for its own pool
 * at start-up (a later cudaMalloc may fail), a host program that runs inside
 * another framework's allocator and must not take memory behind its back, and
 * latency-bound loops where cudaFree's implicit device-wide synchronisation
 * would stall every stream.  This variant computes the same result as
 * qwen3_moe_layer (same arguments, same kernels) with all of its scratch --
 * router logits, expert histogram and permutation, expert activations and
 * per-slot expert outputs -- in one fixed 4 MiB array in device memory that
 * is part of the library: it calls no cudaMalloc, cudaFree or other
 * allocating routine.  Every GPU that loads the library holds those 4 MiB
 * until the process exits.
 *
 * Limit: the scratch must fit in 4 MiB; for the 128-expert, top-8,
 * moe_intermediate 768, hidden 2048 bf16 model that is up to 91 rows.  A
 * larger T returns QWEN3_E_ARG with the row count that fits in
 * qwen3_last_error, before any work is enqueued.  QWEN3_E_ARG too when the
 * handle's device is not the current device; QWEN3_E_UNSUPPORTED while
 * QWEN3_OPT_PROFILE is on (profiling records events).
 *
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture.
 *
 * Sharing: every call on a device, from any handle or thread, uses the same
 * array, which keeps the previous call's contents; each call clears the part
 * that must start at zero on its own stream.  Calls whose GPU work can overlap
 * (different streams without an ordering between them) race on the array and
 * give wrong results: order them on one stream or with events. */
QWEN3_API qwen3_status qwen3_moe_layer_static(qwen3_handle* h, int32_t layer, const void* y, int32_t T, void* out,
                                    int32_t* topk_idx, float* topk_w, void* stream);

/* Embedding rows (maya2_mlx/backbone.py, Backbone.embed_tokens: the rows of
 * the embedding table at the token ids, in the model dtype):
 *   table  dt [vocab, hidden] device, caller-owned, 16-byte aligned
 *   ids    int32 [n] HOST, each in [0, vocab) (checked before any work:
 *          QWEN3_E_ARG names the first bad id)
 *   out    dt [n, hidden] device
 * out[t] = table[ids[t]].  The ids are copied to the device on `stream`. */
QWEN3_API qwen3_status qwen3_embed(qwen3_handle* h, const void* table, int32_t vocab, const int32_t* ids, int32_t n,
                         void* out, void* stream);

/* Output head (maya2_mlx/backbone.py, Backbone.cb0_logits: the product with
 * the head's matrix in the model dtype, then fp32; @mlx-bun/inference
 * qwen3-moe.ts / qwen3.ts: a separate lm_head, or the tied embedding's
 * asLinear):
 *   w       dt [n_out, hidden] device (the head's nn.Linear weight, or the
 *           embedding table for a tied head), 16-byte aligned
 *   x       dt [T, hidden] device: final-norm hidden states
 *   logits  fp32 [T, n_out] device
 * logits[t, o] = fp32(R(sum_k x[t, k] w[o, k])): accumulated in fp32, rounded
 * once to the model dtype, widened exactly.  Any n_out (e.g. 2049). */
QWEN3_API qwen3_status qwen3_head(qwen3_handle* h, const void* w, int32_t n_out, const void* x, int32_t T,
                        float* logits, void* stream);

/* Pooled sentence vector (@mlx-bun/inference qwen3.ts, embedPooled): clears
 * sequence `seq` (as qwen3_reset), runs the stack over the T rows of x at
 * positions 0..T-1 of that sequence, and writes the last row's final-norm
 * hidden state v divided by its L2 norm:
 *   out = R(v / R(sqrt(R(sum_k R(v_k^2)))))   (each array operation of the page
 *   rounded to the model dtype; the sum accumulated in fp32)
 *   x    dt [T, hidden] device (embedded tokens, the pooling token last)
 *   out  dt [hidden] device
 * T must be in [1, capacity] (QWEN3_E_CAPACITY otherwise).  Sequence `seq`
 * ends holding these T positions. */
QWEN3_API qwen3_status qwen3_embed_pooled(qwen3_handle* h, const void* x, int32_t T, int32_t seq, void* out,
                                void* stream);

/* Device bytes held by the handle's grow-only workspace (everything the
 * handle allocates after qwen3_create apart from pinned host staging). */
QWEN3_API qwen3_status qwen3_workspace_bytes(const qwen3_handle* h, int64_t* bytes);

/* Device pointers of one (sequence, layer) cache slab: K and V, each dt
 * [n_kv_heads][capacity][head_dim], K post-RoPE.  Owned by the library; valid
 * until qwen3_destroy.  Used to pre-fill a cache, then qwen3_set_length. */
QWEN3_API qwen3_status qwen3_cache_view(qwen3_handle* h, int32_t seq, int32_t layer, void** k, void** v);

/* Set / read a sequence's length (positions already in its cache). */
QWEN3_API qwen3_status qwen3_set_length(qwen3_handle* h, int32_t seq, int32_t length);
QWEN3_API qwen3_status qwen3_get_length(const qwen3_handle* h, int32_t seq, int32_t* length);

/* Options. */
#define QWEN3_OPT_CUDA_GRAPHS 1   /* 1 (default) = replay a captured graph per row count for decode-sized calls */
#define QWEN3_OPT_PROFILE 2       /* 1 = launch directly and time every kernel with CUDA events */
#define QWEN3_OPT_PDL 3           /* 1 (default) = programmatic dependent launch between kernels */
#define QWEN3_OPT_TENSOR_CORES 4  /* 1 (default) = tcgen05 for bf16 prefill linears and attention, MoE expert GEMMs, and int8 linears of 5..32 rows; 0 = CUDA cores */
#define QWEN3_OPT_L2_PREFETCH 5   /* decode kernels prefetch weights into L2 ahead of their kernel: 0 (default) = off;
                                     1 = each kernel the next one's; 2 = attention o_proj's and gate|up's, o_proj
                                     down's, down the next qkv's */
#define QWEN3_OPT_CLUSTER_ATTENTION 8 /* 1 (default) = decode attention of few sequences on thread-block clusters
                                         (partials merged in distributed shared memory); 0 = split-K with a global merge */
#define QWEN3_OPT_GEMV_CORESIDENT 9 /* 1 = decode GEMV blocks take at most half an SM, so the next kernel's blocks
                                       stream their weights while these finish; 0 (default) = one block per SM */
#define QWEN3_OPT_FAIL_ALLOC 7    /* failure injection: n > 0 makes the n-th next workspace allocation fail as if
                                     cudaMalloc had (QWEN3_E_OOM, no state change); 0 (default) = off */
QWEN3_API qwen3_status qwen3_set_option(qwen3_handle* h, int32_t option, int64_t value);

/* Kernel timing collected while QWEN3_OPT_PROFILE is on (synchronises the
 * device).  Entry `i` (0 <= i < *count) reports a kernel name, its launch
 * count and total milliseconds since the last qwen3_profile_reset. */
QWEN3_API qwen3_status qwen3_profile_read(qwen3_handle* h, int32_t i, const char** name, int64_t* launches,
                                double* total_ms, int32_t* count);
QWEN3_API qwen3_status qwen3_profile_reset(qwen3_handle* h);

/* Device-side failure report: synchronises, then returns QWEN3_E_DEVICE with
 * *code != 0 (and clears it) if a kernel gave up a bounded wait for data it
 * was owed (a TMA copy that never completed), QWEN3_OK with *code = 0
 * otherwise.  Kernels never trap; they record the code and return. */
QWEN3_API qwen3_status qwen3_device_error(qwen3_handle* h, int32_t* code);

/* Self test of the device-side failure report: enqueues one kernel that
 * waits for an mbarrier nothing completes, with the same bounded wait the
 * library's kernels use; after its limit (about a second) it records code 99
 * and returns, so the next qwen3_device_error reports QWEN3_E_DEVICE with
 * code 99 and the context stays usable.  No counterpart on the pages. */
QWEN3_API qwen3_status qwen3_selftest_bounded_wait(qwen3_handle* h, void* stream);

/* Number of kernel launches made by the last successful qwen3_forward. */
QWEN3_API int64_t qwen3_last_launch_count(const qwen3_handle* h);

/* Human-readable text of the last error on this handle ("" if none). */
QWEN3_API const char* qwen3_last_error(const qwen3_handle* h);
QWEN3_API const char* qwen3_status_string(qwen3_status s);

#ifdef __cplusplus
}
#endif
#endif /* QWEN3_GB300_H */
