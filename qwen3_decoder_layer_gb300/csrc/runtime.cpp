// Host runtime behind the C ABI of include/qwen3.h: configuration and
// argument validation (before any state change, as Backbone.forward raises
// before mutating), ownership of the static KV cache and the RoPE table,
// workspaces, the per-call launch plan, CUDA-graph replay and kernel timing.
//
// Plan of one qwen3_forward (maya2_mlx/backbone.py, Backbone.forward), per layer:
//   T <= 4 rows ("decode"):  GEMV(qkv, prologue h = R(h + pend), RMSNorm)
//                            -> q/k norm + RoPE + cache append -> attention
//                            -> GEMV(o, epilogue h = R(h + R(.)))
//                            -> GEMV(gate|up, prologue RMSNorm, epilogue SiLU*up) -> GEMV(down)
//   T > 4 rows ("prefill"):  add+RMSNorm -> GEMM(qkv) -> q/k norm + RoPE + cache
//                            -> attention -> GEMM(o, residual) -> RMSNorm
//                            -> GEMM(gate|up, SiLU*up) -> GEMM(down)
//   MoE layers replace the MLP with RMSNorm -> router logits (fp32) -> top-k
//   -> experts (gathered GEMVs for few rows, sorted grouped GEMMs otherwise)
//   -> weighted combine (@mlx-bun/inference qwen3-moe.ts Qwen3MoeSparseMoeBlock).
// and finally add + RMSNorm with the final norm into `out`.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "kernels.h"
#include "qwen3.h"

using namespace q3;

namespace {

struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
};

struct ProfEvent {
  const char* name;
  cudaEvent_t a, b;
};

struct GraphKey {
  int T;
  int kind;
  const void* x;
  const void* out;
  bool operator<(const GraphKey& o) const {
    if (T != o.T) return T < o.T;
    if (kind != o.kind) return kind < o.kind;
    if (x != o.x) return x < o.x;
    return out < o.out;
  }
};

}  // namespace

struct qwen3_handle {
  qwen3_config cfg{};
  std::vector<int32_t> mlp_only;
  std::vector<qwen3_layer_weights> layers;
  const void* final_norm = nullptr;
  int device = 0, num_sms = 0;
  size_t esz = 0;
  int dt = 0, wfmt = 0;
  void* kcache = nullptr;
  void* vcache = nullptr;
  size_t seq_stride = 0;    // elements between sequences in a cache
  size_t layer_stride = 0;  // elements between layers
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  uint32_t* rope_cs16 = nullptr;  // bf16 models: (cos | sin << 16) per (position, frequency)
  std::vector<int32_t> lengths;
  std::string err;
  // options
  bool use_graphs = true, profile = false, pdl = true, use_tc = true;
  int l2_prefetch = 0;  // off: measured faster on the batch-1 decode step (the prefetches compete with the loads)
  bool cluster_attn = true;   // decode attention on thread-block clusters where it fits
  bool coresident = false;    // decode GEMVs sized for two blocks per SM
  int64_t fail_alloc_in = 0;  // test hook: the n-th next workspace allocation fails (0 = off)
  std::map<int64_t, int> cluster_cap;  // resident clusters of the decode-attention cluster kernel, by launch shape
  // workspace buffers (grow only)
  DevBuf hA, hB, pend, y, qkv, q, attn, mbuf, logits, idx, wts, counts, row_off, row_cnt, tile_start,
      cursor, sorted_tok, sorted_src, mexp, zexp, part_o, part_ml, counters, desc, sumsq, dev_err, skws,
      skcnt, ysort, ids, pool_rows, rlpart, rlcnt, tcpart;
  int ws_generation = 0;
  // descriptor staging (pinned ring)
  static constexpr int kRing = 4;
  void* pinned[kRing] = {};
  size_t pinned_bytes[kRing] = {};
  cudaEvent_t pinned_ev[kRing] = {};
  int ring_pos = 0;
  // graphs
  cudaStream_t gstream = nullptr;
  cudaEvent_t ev_in = nullptr, ev_out = nullptr;
  std::map<GraphKey, std::pair<cudaGraphExec_t, int>> graphs;  // exec, ws generation
  // profiling
  std::vector<ProfEvent> prof_pending;
  std::vector<cudaEvent_t> ev_pool;
  std::map<std::string, std::pair<int64_t, double>> prof_acc;
  std::vector<std::string> prof_names;
  int64_t launches = 0;
  int64_t last_launches = 0;
};

namespace {

qwen3_status fail(qwen3_handle* h, qwen3_status s, const std::string& msg) {
  if (h) h->err = msg;
  return s;
}

qwen3_status cuda_fail(qwen3_handle* h, cudaError_t e, const char* what) {
  return fail(h, QWEN3_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool is_moe_layer(const qwen3_handle* h, int layer) {
  const qwen3_config& c = h->cfg;
  if (c.num_experts <= 0) return false;
  for (int32_t l : h->mlp_only)
    if (l == layer) return false;
  return (layer + 1) % c.decoder_sparse_step == 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Round a double to the model dtype, ties to even: x = m * 2^e with
// 0.5 <= |m| < 1; keep 8 (bf16) or 24 (fp32) significant bits of m.
double round_to_dtype(double x, int dt) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e = 0;
  const double m = std::frexp(x, &e);
  const int bits = dt == QWEN3_DTYPE_BF16 ? 8 : 24;
  return std::ldexp(std::nearbyint(std::ldexp(m, bits)), e - bits);
}

qwen3_status ensure(qwen3_handle* h, DevBuf& b, size_t bytes, bool zero = false) {
  if (bytes <= b.bytes) return QWEN3_OK;
  size_t nb = std::max(bytes, b.bytes + b.bytes / 2);
  nb = (nb + 255) & ~size_t(255);
  void* p = nullptr;
  const bool injected = h->fail_alloc_in > 0 && --h->fail_alloc_in == 0;
  if (injected || cudaMalloc(&p, nb) != cudaSuccess) {
    cudaGetLastError();
    return fail(h, QWEN3_E_OOM, std::string(injected ? "(injected) " : "") + "device allocation of " +
                                    std::to_string(nb) + " bytes failed");
  }
  if (zero) cudaMemset(p, 0, nb);
  if (b.p) {
    cudaDeviceSynchronize();
    cudaFree(b.p);
  }
  b.p = p;
  b.bytes = nb;
  h->ws_generation++;
  return QWEN3_OK;
}

// ---------------------------------------------------------------- profiling
cudaEvent_t pool_event(qwen3_handle* h) {
  if (!h->ev_pool.empty()) {
    cudaEvent_t e = h->ev_pool.back();
    h->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  cudaEventCreate(&e);
  return e;
}

struct Launcher {
  qwen3_handle* h;
  LaunchCtx ctx;
  int count = 0;
};

// Every kernel launch of a forward goes through here so that profiling can
// bracket it with events and the launch count is known.
template <typename F>
cudaError_t launch(Launcher& L, const char* name, F&& fn) {
  qwen3_handle* h = L.h;
  cudaEvent_t a = nullptr, b = nullptr;
  if (h->profile) {
    a = pool_event(h);
    b = pool_event(h);
    cudaEventRecord(a, L.ctx.stream);
  }
  cudaError_t e = fn();
  L.count++;
  if (h->profile) {
    cudaEventRecord(b, L.ctx.stream);
    h->prof_pending.push_back({name, a, b});
  }
  return e;
}

}  // namespace

// ======================================================================
// C ABI
// ======================================================================
extern "C" {

const char* qwen3_status_string(qwen3_status s) {
  switch (s) {
    case QWEN3_OK: return "ok";
    case QWEN3_E_ARG: return "invalid argument";
    case QWEN3_E_DTYPE: return "dtype must be fp32 or bf16";
    case QWEN3_E_CAPACITY: return "context exceeds capacity";
    case QWEN3_E_POSITION: return "positions do not continue the cache";
    case QWEN3_E_SEQ: return "bad sequence id";
    case QWEN3_E_OOM: return "out of device memory";
    case QWEN3_E_CUDA: return "CUDA error";
    case QWEN3_E_UNSUPPORTED: return "unsupported configuration";
    case QWEN3_E_DEVICE: return "no usable device";
  }
  return "unknown status";
}

const char* qwen3_last_error(const qwen3_handle* h) { return h ? h->err.c_str() : "null handle"; }

qwen3_status qwen3_check_config(const qwen3_config* c) {
  if (!c) return QWEN3_E_ARG;
  if (c->dtype != QWEN3_DTYPE_F32 && c->dtype != QWEN3_DTYPE_BF16) return QWEN3_E_DTYPE;
  if (c->num_layers < 1 || c->hidden < 64 || c->hidden % 64 || c->hidden > 8192) return QWEN3_E_ARG;
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) return QWEN3_E_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return QWEN3_E_UNSUPPORTED;
  if (c->n_heads / c->n_kv_heads > 16) return QWEN3_E_UNSUPPORTED;
  if ((c->n_heads * c->head_dim) % 64 || c->n_heads * c->head_dim > 8192) return QWEN3_E_UNSUPPORTED;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 1.0)) return QWEN3_E_ARG;
  if (c->capacity < 1 || c->max_seqs < 1) return QWEN3_E_ARG;
  if (c->weight_format != QWEN3_WEIGHTS_DENSE && c->weight_format != QWEN3_WEIGHTS_INT8) return QWEN3_E_ARG;
  if (c->weight_format == QWEN3_WEIGHTS_INT8) {
    if (c->dtype != QWEN3_DTYPE_BF16) return QWEN3_E_UNSUPPORTED;
    if (c->group_size < 16 || c->group_size % 16 || c->hidden % c->group_size) return QWEN3_E_ARG;
  }
  if (c->num_experts < 0) return QWEN3_E_ARG;
  const bool has_dense = c->num_experts == 0 || c->decoder_sparse_step != 1 || c->n_mlp_only_layers > 0;
  if (has_dense) {
    if (c->intermediate < 64 || c->intermediate % 64 || c->intermediate > 16384) return QWEN3_E_ARG;
    if (c->weight_format == QWEN3_WEIGHTS_INT8 && c->intermediate % c->group_size) return QWEN3_E_ARG;
  }
  if (c->num_experts > 0) {
    if (c->num_experts > 256 || c->top_k < 1 || c->top_k > c->num_experts || c->top_k > 32) return QWEN3_E_ARG;
    if (c->moe_intermediate < 64 || c->moe_intermediate % 64 || c->moe_intermediate > 8192) return QWEN3_E_ARG;
    if (c->decoder_sparse_step < 1) return QWEN3_E_ARG;
    if (c->weight_format == QWEN3_WEIGHTS_INT8 && c->moe_intermediate % c->group_size) return QWEN3_E_ARG;
    if (c->n_mlp_only_layers < 0 || (c->n_mlp_only_layers > 0 && !c->mlp_only_layers)) return QWEN3_E_ARG;
  }
  const double cache_elems = 2.0 * c->max_seqs * c->num_layers * c->n_kv_heads * (double)c->capacity * c->head_dim;
  if (cache_elems > 1.2e12) return QWEN3_E_ARG;
  return QWEN3_OK;
}

qwen3_status qwen3_create(const qwen3_config* cfg, const qwen3_layer_weights* layers, const void* final_norm,
                          qwen3_handle** out) {
  if (!out) return QWEN3_E_ARG;
  *out = nullptr;
  qwen3_status st = qwen3_check_config(cfg);
  if (st != QWEN3_OK) return st;
  if (!layers || !final_norm) return QWEN3_E_ARG;
  qwen3_handle* h = new qwen3_handle();
  h->cfg = *cfg;
  if (cfg->n_mlp_only_layers > 0) h->mlp_only.assign(cfg->mlp_only_layers, cfg->mlp_only_layers + cfg->n_mlp_only_layers);
  h->cfg.mlp_only_layers = nullptr;
  h->layers.assign(layers, layers + cfg->num_layers);
  h->final_norm = final_norm;
  h->dt = cfg->dtype == QWEN3_DTYPE_BF16 ? DT_BF16 : DT_F32;
  h->wfmt = cfg->weight_format == QWEN3_WEIGHTS_INT8 ? W_U8 : W_DT;
  h->esz = cfg->dtype == QWEN3_DTYPE_BF16 ? 2 : 4;
  const bool int8 = cfg->weight_format == QWEN3_WEIGHTS_INT8;
  auto bad = [&](const char* what, int l) {
    h->err = std::string("layer ") + std::to_string(l) + ": " + what;
    return QWEN3_E_ARG;
  };
  if (!aligned16(final_norm)) { delete h; return QWEN3_E_ARG; }
  for (int l = 0; l < cfg->num_layers; ++l) {
    const qwen3_layer_weights& w = layers[l];
    qwen3_status s = QWEN3_OK;
    auto lin_ok = [&](const qwen3_linear& L) {
      if (!L.w || !aligned16(L.w)) return false;
      if (int8 && (!L.scale || !L.bias)) return false;
      return true;
    };
    if (!w.in_norm || !w.post_norm || !w.q_norm || !w.k_norm || !aligned16(w.in_norm) || !aligned16(w.post_norm) ||
        !aligned16(w.q_norm) || !aligned16(w.k_norm))
      s = bad("missing or misaligned norm gain", l);
    else if (!lin_ok(w.qkv) || !lin_ok(w.o)) s = bad("missing attention weights", l);
    else if (is_moe_layer(h, l)) {
      if (!w.router || !aligned16(w.router) || !lin_ok(w.exp_gate_up) || !lin_ok(w.exp_down))
        s = bad("missing MoE weights", l);
    } else if (!lin_ok(w.gate_up) || !lin_ok(w.down)) {
      s = bad("missing MLP weights", l);
    }
    if (s != QWEN3_OK) {
      qwen3_status r = s;
      delete h;
      return r;
    }
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    delete h;
    return QWEN3_E_DEVICE;
  }
  cudaGetDevice(&h->device);
  cudaDeviceProp prop;
  cudaGetDeviceProperties(&prop, h->device);
  if (prop.major < 10) {
    delete h;
    return QWEN3_E_DEVICE;
  }
  h->num_sms = prop.multiProcessorCount;
  const qwen3_config& c = h->cfg;
  h->layer_stride = (size_t)c.n_kv_heads * c.capacity * c.head_dim;
  h->seq_stride = h->layer_stride * c.num_layers;
  const size_t cache_bytes = h->seq_stride * c.max_seqs * h->esz;
  if (cudaMalloc(&h->kcache, cache_bytes) != cudaSuccess || cudaMalloc(&h->vcache, cache_bytes) != cudaSuccess) {
    cudaGetLastError();
    qwen3_destroy(h);
    return QWEN3_E_OOM;
  }
  cudaMemset(h->kcache, 0, cache_bytes);
  cudaMemset(h->vcache, 0, cache_bytes);
  // RoPE table: inv_freq_i = theta^(-2i/D) rounded to dt; angle p * inv_freq in
  // double; cos / sin rounded to dt; both halves of a row repeat the frequencies.
  const int D = c.head_dim, half = D / 2;
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = round_to_dtype(std::pow(c.rope_theta, -2.0 * i / D), c.dtype);
  std::vector<float> cs((size_t)c.capacity * D), sn((size_t)c.capacity * D);
  for (int p = 0; p < c.capacity; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * inv[i];
      const float cv = (float)round_to_dtype(std::cos(ang), c.dtype);
      const float sv = (float)round_to_dtype(std::sin(ang), c.dtype);
      cs[(size_t)p * D + i] = cs[(size_t)p * D + i + half] = cv;
      sn[(size_t)p * D + i] = sn[(size_t)p * D + i + half] = sv;
    }
  if (cudaMalloc(&h->rope_cos, cs.size() * 4) != cudaSuccess ||
      cudaMalloc(&h->rope_sin, sn.size() * 4) != cudaSuccess) {
    cudaGetLastError();
    qwen3_destroy(h);
    return QWEN3_E_OOM;
  }
  cudaMemcpy(h->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
  cudaMemcpy(h->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
  if (c.dtype == QWEN3_DTYPE_BF16) {
    // the table's bf16 values (exact: each was rounded to bf16 above), one
    // (cos, sin) pair per frequency, for the q|k|v GEMM epilogue
    std::vector<uint32_t> cs16((size_t)c.capacity * half);
    auto bits = [](float v) {
      uint32_t u;
      std::memcpy(&u, &v, 4);
      return u >> 16;
    };
    for (int p = 0; p < c.capacity; ++p)
      for (int i = 0; i < half; ++i)
        cs16[(size_t)p * half + i] = bits(cs[(size_t)p * D + i]) | (bits(sn[(size_t)p * D + i]) << 16);
    if (cudaMalloc(&h->rope_cs16, cs16.size() * 4) != cudaSuccess) {
      cudaGetLastError();
      qwen3_destroy(h);
      return QWEN3_E_OOM;
    }
    cudaMemcpy(h->rope_cs16, cs16.data(), cs16.size() * 4, cudaMemcpyHostToDevice);
  }
  h->lengths.assign(c.max_seqs, 0);
  for (int i = 0; i < qwen3_handle::kRing; ++i) cudaEventCreateWithFlags(&h->pinned_ev[i], cudaEventDisableTiming);
  cudaStreamCreateWithFlags(&h->gstream, cudaStreamNonBlocking);
  cudaEventCreateWithFlags(&h->ev_in, cudaEventDisableTiming);
  cudaEventCreateWithFlags(&h->ev_out, cudaEventDisableTiming);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    qwen3_destroy(h);
    return QWEN3_E_CUDA;
  }
  *out = h;
  return QWEN3_OK;
}

void qwen3_destroy(qwen3_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.second.first);
  DevBuf* bufs[] = {&h->hA, &h->hB, &h->pend, &h->y, &h->qkv, &h->q, &h->attn, &h->mbuf, &h->logits, &h->idx,
                    &h->wts, &h->counts, &h->row_off, &h->row_cnt, &h->tile_start, &h->cursor, &h->sorted_tok,
                    &h->sorted_src, &h->mexp, &h->zexp, &h->part_o, &h->part_ml, &h->counters, &h->desc, &h->sumsq, &h->dev_err,
                    &h->skws, &h->skcnt, &h->ysort, &h->ids, &h->pool_rows, &h->rlpart, &h->rlcnt,
                    &h->tcpart};
  for (DevBuf* b : bufs)
    if (b->p) cudaFree(b->p);
  for (int i = 0; i < qwen3_handle::kRing; ++i) {
    if (h->pinned[i]) cudaFreeHost(h->pinned[i]);
    if (h->pinned_ev[i]) cudaEventDestroy(h->pinned_ev[i]);
  }
  for (auto& p : h->prof_pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : h->ev_pool) cudaEventDestroy(e);
  if (h->gstream) cudaStreamDestroy(h->gstream);
  if (h->ev_in) cudaEventDestroy(h->ev_in);
  if (h->ev_out) cudaEventDestroy(h->ev_out);
  if (h->kcache) cudaFree(h->kcache);
  if (h->vcache) cudaFree(h->vcache);
  if (h->rope_cos) cudaFree(h->rope_cos);
  if (h->rope_sin) cudaFree(h->rope_sin);
  if (h->rope_cs16) cudaFree(h->rope_cs16);
  delete h;
}

qwen3_status qwen3_reset(qwen3_handle* h, int32_t seq, void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (seq < -1 || seq >= h->cfg.max_seqs) return fail(h, QWEN3_E_SEQ, "sequence id out of range");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = h->seq_stride * h->esz;
  const int s0 = seq < 0 ? 0 : seq, s1 = seq < 0 ? h->cfg.max_seqs : seq + 1;
  for (int i = s0; i < s1; ++i) {
    cudaError_t e1 = cudaMemsetAsync(static_cast<char*>(h->kcache) + i * bytes, 0, bytes, s);
    cudaError_t e2 = cudaMemsetAsync(static_cast<char*>(h->vcache) + i * bytes, 0, bytes, s);
    if (e1 != cudaSuccess || e2 != cudaSuccess) return cuda_fail(h, e1 != cudaSuccess ? e1 : e2, "reset");
    h->lengths[i] = 0;
  }
  return QWEN3_OK;
}

qwen3_status qwen3_cache_view(qwen3_handle* h, int32_t seq, int32_t layer, void** k, void** v) {
  if (!h || !k || !v) return QWEN3_E_ARG;
  if (seq < 0 || seq >= h->cfg.max_seqs) return fail(h, QWEN3_E_SEQ, "sequence id out of range");
  if (layer < 0 || layer >= h->cfg.num_layers) return fail(h, QWEN3_E_ARG, "layer out of range");
  const size_t off = (seq * h->seq_stride + layer * h->layer_stride) * h->esz;
  *k = static_cast<char*>(h->kcache) + off;
  *v = static_cast<char*>(h->vcache) + off;
  return QWEN3_OK;
}

qwen3_status qwen3_set_length(qwen3_handle* h, int32_t seq, int32_t length) {
  if (!h) return QWEN3_E_ARG;
  if (seq < 0 || seq >= h->cfg.max_seqs) return fail(h, QWEN3_E_SEQ, "sequence id out of range");
  if (length < 0 || length > h->cfg.capacity) return fail(h, QWEN3_E_CAPACITY, "length exceeds capacity");
  h->lengths[seq] = length;
  return QWEN3_OK;
}

qwen3_status qwen3_get_length(const qwen3_handle* h, int32_t seq, int32_t* length) {
  if (!h || !length) return QWEN3_E_ARG;
  if (seq < 0 || seq >= h->cfg.max_seqs) return QWEN3_E_SEQ;
  *length = h->lengths[seq];
  return QWEN3_OK;
}

qwen3_status qwen3_set_option(qwen3_handle* h, int32_t option, int64_t value) {
  if (!h) return QWEN3_E_ARG;
  if (option != QWEN3_OPT_FAIL_ALLOC && !h->graphs.empty()) {  // captured launches follow the old options
    cudaDeviceSynchronize();
    for (auto& g : h->graphs) cudaGraphExecDestroy(g.second.first);
    h->graphs.clear();
  }
  switch (option) {
    case QWEN3_OPT_CUDA_GRAPHS: h->use_graphs = value != 0; return QWEN3_OK;
    case QWEN3_OPT_PROFILE: h->profile = value != 0; return QWEN3_OK;
    case QWEN3_OPT_PDL: h->pdl = value != 0; return QWEN3_OK;
    case QWEN3_OPT_TENSOR_CORES: h->use_tc = value != 0; return QWEN3_OK;
    case QWEN3_OPT_L2_PREFETCH:
      if (value < 0 || value > 2) return fail(h, QWEN3_E_ARG, "QWEN3_OPT_L2_PREFETCH takes 0, 1 or 2");
      h->l2_prefetch = (int)value;
      return QWEN3_OK;
    case QWEN3_OPT_CLUSTER_ATTENTION: h->cluster_attn = value != 0; return QWEN3_OK;
    case QWEN3_OPT_GEMV_CORESIDENT: h->coresident = value != 0; return QWEN3_OK;
    case QWEN3_OPT_FAIL_ALLOC:
      if (value < 0) return fail(h, QWEN3_E_ARG, "QWEN3_OPT_FAIL_ALLOC takes a count >= 0");
      h->fail_alloc_in = value;
      return QWEN3_OK;
  }
  return fail(h, QWEN3_E_ARG, "unknown option");
}

qwen3_status qwen3_profile_reset(qwen3_handle* h) {
  if (!h) return QWEN3_E_ARG;
  cudaDeviceSynchronize();
  for (auto& p : h->prof_pending) {
    h->ev_pool.push_back(p.a);
    h->ev_pool.push_back(p.b);
  }
  h->prof_pending.clear();
  h->prof_acc.clear();
  h->prof_names.clear();
  return QWEN3_OK;
}

qwen3_status qwen3_profile_read(qwen3_handle* h, int32_t i, const char** name, int64_t* launches, double* total_ms,
                                int32_t* count) {
  if (!h) return QWEN3_E_ARG;
  if (!h->prof_pending.empty()) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "profile sync");
    for (auto& p : h->prof_pending) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, p.a, p.b);
      auto& acc = h->prof_acc[p.name];
      acc.first += 1;
      acc.second += ms;
      h->ev_pool.push_back(p.a);
      h->ev_pool.push_back(p.b);
    }
    h->prof_pending.clear();
    h->prof_names.clear();
    for (auto& kv : h->prof_acc) h->prof_names.push_back(kv.first);
  }
  if (count) *count = (int32_t)h->prof_names.size();
  if (i < 0 || i >= (int32_t)h->prof_names.size()) return QWEN3_OK;
  const auto& acc = h->prof_acc[h->prof_names[i]];
  if (name) *name = h->prof_names[i].c_str();
  if (launches) *launches = acc.first;
  if (total_ms) *total_ms = acc.second;
  return QWEN3_OK;
}

int64_t qwen3_last_launch_count(const qwen3_handle* h) { return h ? h->last_launches : 0; }

}  // extern "C"

// ======================================================================
// forward
// ======================================================================
namespace {

enum AttnKind { ATTN_DECODE = 0, ATTN_PREFILL = 1, ATTN_TC = 2 };  // decode kernel; SIMT / tcgen05 prefill

struct Plan {
  int T = 0;
  bool gemv = false;           // T <= 4: weight-streaming GEMVs for the linears
  int attn = ATTN_DECODE;      // attention kernel
  int rows_per_block = 1;
  int chunk = 64;
  int nq_max = 16;
  int max_nq = 1;              // largest rows x G of any query block
  int max_keys = 0;            // most keys any query block attends to
  int cluster = 0;             // decode attention: CTAs per cluster (0 = the item / run kernels)
  int n_qblocks = 0, n_items = 0, n_parts = 0;
  std::vector<int32_t> blob;   // row_seq[T] row_pos[T] n_items qblocks items
  size_t off_rowseq = 0, off_rowpos = 0, off_nitems = 0, off_qb = 0, off_items = 0;
};

constexpr int kQbInts = sizeof(AttnQBlock) / sizeof(int32_t);

// Validate rows and build the attention work list (host only; no state change).
qwen3_status build_plan(qwen3_handle* h, int T, const int32_t* seq_ids, const int32_t* positions, Plan& P) {
  const qwen3_config& c = h->cfg;
  const int G = c.n_heads / c.n_kv_heads;
  struct Seg { int seq, row0, n, pos0; };
  std::vector<Seg> segs;
  std::vector<char> seen(c.max_seqs, 0);
  for (int t = 0; t < T; ++t) {
    const int s = seq_ids[t];
    if (s < 0 || s >= c.max_seqs) return fail(h, QWEN3_E_SEQ, "row " + std::to_string(t) + ": sequence id out of range");
    if (segs.empty() || segs.back().seq != s) {
      if (seen[s]) return fail(h, QWEN3_E_SEQ, "rows of sequence " + std::to_string(s) + " are not consecutive");
      seen[s] = 1;
      segs.push_back({s, t, 0, h->lengths[s]});
    }
    Seg& g = segs.back();
    const int expect = g.pos0 + g.n;
    if (expect >= c.capacity)
      return fail(h, QWEN3_E_CAPACITY, "context " + std::to_string(expect + 1) + " exceeds capacity " +
                                           std::to_string(c.capacity));
    if (positions[t] != expect)
      return fail(h, QWEN3_E_POSITION, "row " + std::to_string(t) + " of sequence " + std::to_string(s) +
                                           " at position " + std::to_string(positions[t]) + ", expected " +
                                           std::to_string(expect));
    g.n++;
  }
  P.T = T;
  P.gemv = T <= 4;
  int max_rows = 0;
  for (auto& g : segs) max_rows = std::max(max_rows, g.n);
  // the decode kernel takes up to 4 rows per sequence, in query blocks of nq_max / G rows
  P.attn = (max_rows <= 4 && G <= attn_decode2_nq_max()) ? ATTN_DECODE : ATTN_PREFILL;
  if (P.attn == ATTN_PREFILL && h->dt == DT_BF16 && h->use_tc && attn_tc_supported(c.head_dim)) P.attn = ATTN_TC;
  P.nq_max = P.attn == ATTN_DECODE ? attn_decode2_nq_max() : attn_prefill_nq_max();
  P.chunk = P.attn == ATTN_DECODE ? attn_decode2_chunk(h->dt) : attn_prefill_chunk();
  // tcgen05 attention: 128-row query tiles, each walking all of its keys (one "chunk")
  P.rows_per_block = P.attn == ATTN_TC ? attn_tc_rows() : P.nq_max / G;
  std::vector<int32_t> qb, items;
  int parts = 0, nqb = 0;
  for (auto& g : segs) {
    for (int r = 0; r < g.n; r += P.rows_per_block) {
      const int nr = std::min(P.rows_per_block, g.n - r);
      P.max_nq = std::max(P.max_nq, nr * G);
      const int last_pos = g.pos0 + r + nr - 1;
      P.max_keys = std::max(P.max_keys, last_pos + 1);
      const int nch = P.attn == ATTN_TC ? 1 : (last_pos + 1 + P.chunk - 1) / P.chunk;
      qb.insert(qb.end(), {g.seq, g.row0 + r, nr, g.pos0 + r, nch, parts, g.row0, g.pos0, g.n, 0});
      for (int ch = 0; ch < nch; ++ch) items.insert(items.end(), {nqb, ch});
      parts += nch;
      nqb++;
    }
  }
  P.n_qblocks = nqb;
  P.n_items = (int)items.size() / 2;
  P.n_parts = parts;
  P.blob.clear();
  P.off_rowseq = 0;
  P.blob.insert(P.blob.end(), seq_ids, seq_ids + T);
  P.off_rowpos = P.blob.size();
  P.blob.insert(P.blob.end(), positions, positions + T);
  P.off_nitems = P.blob.size();
  P.blob.push_back(P.n_items);
  while (P.blob.size() % 4) P.blob.push_back(0);
  P.off_qb = P.blob.size();
  P.blob.insert(P.blob.end(), qb.begin(), qb.end());
  // room for T query blocks so that the item list sits at an offset fixed by T
  P.blob.resize(P.off_qb + (size_t)kQbInts * std::max(T, nqb), 0);
  P.off_items = P.blob.size();
  P.blob.insert(P.blob.end(), items.begin(), items.end());
  return QWEN3_OK;
}

struct Bufs {  // raw pointers for one forward
  void *hA, *hB, *pend, *y, *qkv, *q, *attn, *m;
  float *logits, *wts, *part_o, *part_ml;
  int *idx, *counts, *row_off, *row_cnt, *tile_start, *cursor, *sorted_tok, *sorted_src, *counters, *err;
  void *mexp, *zexp, *ysort;
  float* rlpart;  // router logits: split-k partial tiles (NULL: one k range)
  int* rlcnt;     // router logits: per-tile arrival counters (kept zero by the kernel)
  float* tcpart;  // split-k partial tiles of the tensor-core GEMM (one row tile)
  size_t tcpart_floats;
  double* sumsq;
  int32_t* desc;
};

qwen3_status ensure_workspace(qwen3_handle* h, const Plan& P, int T) {
  const qwen3_config& c = h->cfg;
  const size_t e = h->esz;
  const size_t Tz = (size_t)std::max(T, 1);
  qwen3_status s;
#define ENS(buf, bytes, zero) \
  if ((s = ensure(h, h->buf, (bytes), zero)) != QWEN3_OK) return s;
  ENS(hA, Tz * c.hidden * e, false);
  ENS(hB, Tz * c.hidden * e, false);
  ENS(pend, Tz * c.hidden * e, false);
  ENS(y, Tz * c.hidden * e, false);
  ENS(qkv, Tz * (c.n_heads + 2 * c.n_kv_heads) * c.head_dim * e, false);
  ENS(q, Tz * c.n_heads * c.head_dim * e, false);
  ENS(attn, Tz * c.n_heads * c.head_dim * e, false);
  ENS(mbuf, Tz * std::max(c.intermediate, 64) * e, false);
  ENS(sumsq, Tz * (2 * (size_t)c.num_layers + 1) * sizeof(double), true);
  ENS(dev_err, 64, true);
  if (!P.gemv && T <= 64) {  // skinny GEMM split-K workspace (kept zero by the kernel)
    const size_t nmax = std::max({(size_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim, (size_t)c.hidden,
                                  2 * (size_t)c.intermediate});
    ENS(skws, gemm_skinny_ws_floats(64, (int)nmax, EPI_STORE) * 4, false);
    ENS(skcnt, (size_t)gemm_skinny_tiles((int)nmax) * 4, true);
  }
  // attention partials: sized for the worst case of this row count when graphs replay it
  size_t parts = (size_t)std::max(P.n_parts, 1);
  if (P.gemv) parts = std::max(parts, (size_t)std::max(P.n_qblocks, T) * ((c.capacity + P.chunk - 1) / P.chunk));
  ENS(part_o, parts * c.n_kv_heads * P.nq_max * c.head_dim * 4, false);
  ENS(part_ml, parts * c.n_kv_heads * P.nq_max * 2 * 4, false);
  ENS(counters, (size_t)std::max(P.n_qblocks, T) * c.n_kv_heads * 4, true);
  if (c.num_experts > 0) {
    const size_t slots = Tz * c.top_k;
    ENS(logits, Tz * c.num_experts * 4, false);
    ENS(idx, slots * 4, false);
    ENS(wts, slots * 4, false);
    ENS(counts, (size_t)c.num_experts * 4, true);
    ENS(row_off, (size_t)c.num_experts * 4, false);
    ENS(row_cnt, (size_t)c.num_experts * 4, false);
    ENS(tile_start, (size_t)(c.num_experts + 1) * 4, false);
    ENS(cursor, (size_t)c.num_experts * 4, true);
    ENS(sorted_tok, slots * 4, false);
    ENS(sorted_src, slots * 4, false);
    ENS(mexp, slots * c.moe_intermediate * e, false);
    ENS(zexp, slots * c.hidden * e, false);
    if (h->dt == DT_BF16 && T > 4) ENS(ysort, slots * c.hidden * e, false);  // rows in expert order (tensor-core path)
    if (T > 4) {
      ENS(rlpart, (size_t)kRouterMaxSplits * Tz * c.num_experts * 4, false);
      ENS(rlcnt, (size_t)router_logits_tiles(T, c.num_experts) * 4, true);
    }
  }
  if (!P.gemv && T <= 128 && h->use_tc && h->dt == DT_BF16) {
    // split-k partial tiles for the dense linears of one 128-row tile
    const int hid = c.hidden, qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim, hd = c.n_heads * c.head_dim;
    const int shapes[4][3] = {{qkv, hid, EPI_STORE}, {hid, hd, EPI_RESIDUAL}, {c.intermediate, hid, EPI_SWIGLU},
                              {hid, c.intermediate, EPI_STORE}};
    size_t fl = 0;
    for (const auto& sh : shapes)
      fl = std::max(fl, gemm_tc_part_floats(T, sh[0], sh[2], gemm_tc_splits(T, sh[0], sh[1], sh[2], h->num_sms)));
    if (fl) ENS(tcpart, fl * sizeof(float), false);
  }
  ENS(desc, P.blob.size() * 4 + 64, false);
#undef ENS
  return QWEN3_OK;
}

Bufs bufs_of(qwen3_handle* h) {
  Bufs b;
  b.hA = h->hA.p; b.hB = h->hB.p; b.pend = h->pend.p; b.y = h->y.p; b.qkv = h->qkv.p; b.q = h->q.p;
  b.attn = h->attn.p; b.m = h->mbuf.p;
  b.logits = (float*)h->logits.p; b.wts = (float*)h->wts.p; b.part_o = (float*)h->part_o.p;
  b.part_ml = (float*)h->part_ml.p; b.idx = (int*)h->idx.p; b.counts = (int*)h->counts.p;
  b.row_off = (int*)h->row_off.p; b.row_cnt = (int*)h->row_cnt.p; b.tile_start = (int*)h->tile_start.p;
  b.cursor = (int*)h->cursor.p; b.sorted_tok = (int*)h->sorted_tok.p; b.sorted_src = (int*)h->sorted_src.p;
  b.counters = (int*)h->counters.p; b.err = (int*)h->dev_err.p; b.mexp = h->mexp.p; b.zexp = h->zexp.p;
  b.ysort = h->ysort.p; b.rlpart = (float*)h->rlpart.p; b.rlcnt = (int*)h->rlcnt.p;
  b.tcpart = (float*)h->tcpart.p; b.tcpart_floats = h->tcpart.bytes / sizeof(float);
  b.sumsq = (double*)h->sumsq.p; b.desc = (int32_t*)h->desc.p;
  return b;
}

// Upload the plan descriptor through a pinned staging ring.
qwen3_status upload_plan(qwen3_handle* h, const Plan& P, cudaStream_t s) {
  const size_t bytes = P.blob.size() * 4;
  const int i = h->ring_pos;
  h->ring_pos = (h->ring_pos + 1) % qwen3_handle::kRing;
  cudaEventSynchronize(h->pinned_ev[i]);
  if (h->pinned_bytes[i] < bytes) {
    if (h->pinned[i]) cudaFreeHost(h->pinned[i]);
    h->pinned[i] = nullptr;
    const size_t nb = std::max(bytes, (size_t)4096) * 2;
    if (cudaHostAlloc(&h->pinned[i], nb, cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      h->pinned_bytes[i] = 0;
      return fail(h, QWEN3_E_OOM, "pinned host allocation failed");
    }
    h->pinned_bytes[i] = nb;
  }
  std::memcpy(h->pinned[i], P.blob.data(), bytes);
  cudaError_t e = cudaMemcpyAsync(h->desc.p, h->pinned[i], bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "descriptor upload");
  cudaEventRecord(h->pinned_ev[i], s);
  return QWEN3_OK;
}

// MoE block on y [T, hidden].  The weighted expert sum goes to `out`, or,
// when h_res is given, is added to the residual h_res in place with the
// rows' sums of squares added to sumsq_out (zero beforehand).  idx/w receive the routing.
// norm_sumsq (decode, T <= 4, with h_res): y is not there yet but is the
// layer's post-attention RMSNorm of h_res with these sums of squares; the
// router GEMV forms it in its prologue and stores it to y for the experts.
cudaError_t moe_block(qwen3_handle* h, Launcher& L, int layer, const void* y, int T, void* out, void* h_res,
                      double* sumsq_out, int* idx, float* w, const Bufs& B, const double* norm_sumsq = nullptr) {
  const qwen3_config& c = h->cfg;
  const qwen3_layer_weights& W = h->layers[layer];
  const int E = c.num_experts, k = c.top_k, mI = c.moe_intermediate, hid = c.hidden;
  const int dt = h->dt;
  const int xw = W.exp_gate_up.scale ? h->wfmt : W_DT;  // expert weight format
  cudaError_t e;
  // router logits, fp32, not rounded
  if (T <= 4 && norm_sumsq && h_res) {
    // RMSNorm prologue from the residual epilogue's sums of squares; block 0
    // stores the normalised rows for the expert GEMVs
    Gemv2Args g{};
    g.T = T; g.K = hid; g.N = E; g.w = W.router; g.prologue = PRO_SUMSQ; g.h = h_res; g.gain = W.post_norm;
    g.eps = c.rms_eps; g.sumsq_in = norm_sumsq; g.x_out = const_cast<void*>(y); g.epilogue = EPI_STORE_F32;
    g.out = B.logits; g.ldo = E; g.err = B.err;
    g.stages = gemv2_plan(dt, W_DT, T, hid, c.group_size, false, &g.nwarps, false);
    g.nwarps = std::min(g.nwarps, 4);  // one weight row per warp: E / 4 blocks
    e = launch(L, "gemv_router", [&] { return launch_gemv2(L.ctx, dt, W_DT, g); });
  } else if (T <= 4) {
    GemvArgs g{};
    g.T = T; g.K = hid; g.N = E; g.w = W.router; g.x_rows = T; g.x = y;
    g.epilogue = EPI_STORE_F32; g.out = B.logits; g.ldo = E;
    e = launch(L, "gemv_router", [&] { return launch_gemv(L.ctx, dt, W_DT, g); });
  } else {
    GemmArgs g{};
    g.M = T; g.N = E; g.K = hid; g.a = y; g.lda = hid; g.w = W.router; g.epilogue = EPI_STORE_F32;
    g.out = B.logits; g.ldo = E;
    if (router_logits_supported(dt, E, hid)) {
      RouterLogitsArgs r{};
      r.M = T; r.E = E; r.K = hid; r.y = y; r.ldy = hid; r.w = W.router; r.out = B.logits; r.ldo = E;
      r.part = B.rlpart; r.counters = B.rlcnt; r.max_splits = kRouterMaxSplits;
      e = launch(L, "router_logits", [&] { return launch_router_logits(L.ctx, dt, r); });
    } else
      e = launch(L, "gemm_router", [&] { return launch_gemm_simt(L.ctx, dt, W_DT, g); });
  }
  if (e != cudaSuccess) return e;
  const int sort_from = (64 + k - 1) / k;  // qwen3-moe.ts: sorted experts from ceil(64 / topK) rows
  const bool unsorted = T < sort_from && (size_t)T * k * mI * 4 <= 200 * 1024 && T * k <= 64;
  RouterArgs r{};
  r.logits = B.logits; r.T = T; r.E = E; r.k = k; r.norm = c.norm_topk_prob; r.idx = idx; r.w = w;
  r.counts = unsorted ? nullptr : B.counts;
  e = launch(L, "router_topk", [&] { return launch_router_topk(L.ctx, r); });
  if (e != cudaSuccess) return e;
  const int slots = T * k;
  if (unsorted) {
    GemvArgs g{};
    g.T = slots; g.K = hid; g.N = mI; g.w = W.exp_gate_up.w; g.scale = W.exp_gate_up.scale;
    g.bias = W.exp_gate_up.bias; g.group = c.group_size; g.slot_expert = idx;
    g.w_stride = (long long)2 * mI * hid; g.slot_div = k; g.x_rows = T; g.x = y;
    g.epilogue = EPI_SWIGLU; g.out = B.mexp; g.ldo = mI;
    e = launch(L, "gemv_expert_gate_up", [&] { return launch_gemv(L.ctx, dt, xw, g); });
    if (e != cudaSuccess) return e;
    GemvArgs d{};
    d.T = slots; d.K = mI; d.N = hid; d.w = W.exp_down.w; d.scale = W.exp_down.scale; d.bias = W.exp_down.bias;
    d.group = c.group_size; d.slot_expert = idx; d.w_stride = (long long)hid * mI;
    d.slot_div = 1; d.x_rows = slots; d.x = B.mexp; d.epilogue = EPI_STORE; d.out = B.zexp;
    d.ldo = hid;
    e = launch(L, "gemv_expert_down", [&] { return launch_gemv(L.ctx, dt, xw, d); });
    if (e != cudaSuccess) return e;
  } else {
    // tensor-core grouped GEMMs (bf16 experts whose shapes fit the 128 x 256 tiles), else CUDA cores
    const bool tc = h->use_tc && dt == DT_BF16 && xw == W_DT && B.ysort && mI % (128) == 0 && hid % 256 == 0 &&
                    gemm_tc_supported(slots, mI, hid, EPI_SWIGLU) && gemm_tc_supported(slots, hid, mI, EPI_STORE);
    const int BM = tc ? 128 : gemm_simt_tile_m();
    MoeScanArgs sc{};
    sc.counts = B.counts; sc.E = E; sc.bm = BM; sc.row_off = B.row_off; sc.row_cnt = B.row_cnt;
    sc.tile_start = B.tile_start; sc.cursor = B.cursor;
    e = launch(L, "moe_scan", [&] { return launch_moe_scan(L.ctx, sc); });
    if (e != cudaSuccess) return e;
    MoeScatterArgs sa{};
    sa.idx = idx; sa.T = T; sa.k = k; sa.row_off = B.row_off; sa.cursor = B.cursor; sa.sorted_tok = B.sorted_tok;
    sa.sorted_src = B.sorted_src;
    e = launch(L, "moe_scatter", [&] { return launch_moe_scatter(L.ctx, sa); });
    if (e != cudaSuccess) return e;
    const int max_tiles = (slots + BM - 1) / BM + E;
    if (tc) {
      MoeGatherArgs ga{};
      ga.x = y; ga.rows = B.sorted_tok; ga.n = slots; ga.K = hid; ga.out = B.ysort;
      e = launch(L, "moe_gather", [&] { return launch_moe_gather(L.ctx, dt, ga); });
      if (e != cudaSuccess) return e;
      GemmTcArgs t{};
      t.M = slots; t.N = mI; t.K = hid; t.a = B.ysort; t.lda = hid; t.w = W.exp_gate_up.w; t.out = B.mexp;
      t.ldo = mI; t.epilogue = EPI_SWIGLU; t.err = B.err; t.tile_start = B.tile_start; t.row_off = B.row_off;
      t.row_cnt = B.row_cnt; t.n_groups = E; t.max_tiles_m = max_tiles; t.w_group_rows = 2LL * mI;
      t.w_rows_total = 2LL * mI * E;
      e = launch(L, "gemm_tc_expert_gate_up", [&] { return launch_gemm_tc(L.ctx, t); });
      if (e != cudaSuccess) return e;
      GemmTcArgs d{};
      d.M = slots; d.N = hid; d.K = mI; d.a = B.mexp; d.lda = mI; d.w = W.exp_down.w; d.out = B.zexp; d.ldo = hid;
      d.epilogue = EPI_STORE; d.err = B.err; d.tile_start = B.tile_start; d.row_off = B.row_off;
      d.row_cnt = B.row_cnt; d.n_groups = E; d.max_tiles_m = max_tiles; d.w_group_rows = hid;
      d.w_rows_total = (long long)hid * E; d.c_rows = B.sorted_src;
      e = launch(L, "gemm_tc_expert_down", [&] { return launch_gemm_tc(L.ctx, d); });
      if (e != cudaSuccess) return e;
    } else {
    GemmArgs g{};
    g.M = slots; g.N = mI; g.K = hid; g.a = y; g.lda = hid; g.a_rows = B.sorted_tok; g.w = W.exp_gate_up.w;
    g.scale = W.exp_gate_up.scale; g.bias = W.exp_gate_up.bias; g.group = c.group_size;
    g.w_stride = (long long)2 * mI * hid; g.tile_start = B.tile_start; g.row_off = B.row_off;
    g.row_cnt = B.row_cnt; g.n_groups = E; g.max_tiles = max_tiles; g.epilogue = EPI_SWIGLU; g.out = B.mexp;
    g.ldo = mI;
    e = launch(L, "gemm_expert_gate_up", [&] { return launch_gemm_simt(L.ctx, dt, xw, g); });
    if (e != cudaSuccess) return e;
    GemmArgs d{};
    d.M = slots; d.N = hid; d.K = mI; d.a = B.mexp; d.lda = mI; d.w = W.exp_down.w; d.scale = W.exp_down.scale;
    d.bias = W.exp_down.bias; d.group = c.group_size; d.w_stride = (long long)hid * mI;
    d.tile_start = B.tile_start; d.row_off = B.row_off; d.row_cnt = B.row_cnt; d.n_groups = E;
    d.max_tiles = max_tiles; d.epilogue = EPI_STORE; d.out = B.zexp; d.ldo = hid; d.c_rows = B.sorted_src;
    e = launch(L, "gemm_expert_down", [&] { return launch_gemm_simt(L.ctx, dt, xw, d); });
    if (e != cudaSuccess) return e;
    }
  }
  MoeCombineArgs cb{};
  cb.z = B.zexp; cb.w = w; cb.T = T; cb.k = k; cb.hidden = hid; cb.out = out; cb.h = h_res; cb.sumsq_out = sumsq_out;
  return launch(L, "moe_combine", [&] { return launch_moe_combine(L.ctx, dt, cb); });
}

// Decode attention with one query block per thread-block cluster when every
// (query block, kv head) gets its own cluster, all of them resident at once,
// and each query block's keys fit the cluster's shared memory: the largest of
// 16, 12 or 8 CTAs per cluster that fits (on a 152-SM GB300, seven 16-CTA
// clusters of this kernel are resident at once, eight of 12, fifteen of 8).
int decode_cluster_size(qwen3_handle* h, const Plan& P) {
  if (P.attn != ATTN_DECODE || P.n_qblocks < 1) return 0;
  const qwen3_config& c = h->cfg;
  for (int cl : {16, 12, 8}) {
    if ((int64_t)P.n_qblocks * c.n_kv_heads * cl > h->num_sms) continue;
    if (P.max_keys > attn_decode_cluster_keys(h->dt, P.max_nq, cl)) continue;
    const int nqb = P.max_nq <= 1 ? 1 : P.max_nq <= 2 ? 2 : P.max_nq <= 4 ? 4 : 8;
    const int64_t key = ((int64_t)cl << 40) | ((int64_t)nqb << 32) | ((int64_t)P.n_qblocks << 16) | c.n_kv_heads;
    auto it = h->cluster_cap.find(key);
    if (it == h->cluster_cap.end())
      it = h->cluster_cap.emplace(key, attn_decode_cluster_capacity(h->dt, c.head_dim, P.max_nq, cl, c.n_kv_heads,
                                                                    P.n_qblocks)).first;
    if (it->second >= P.n_qblocks * c.n_kv_heads) return cl;
  }
  return 0;
}

// q/k RMSNorm + RoPE + cache append of layer l's q|k|v rows (B.qkv) for the
// prefill attention kernels: queries to B.q, keys and values to the caches.
QkRopeArgs qk_rope_args(qwen3_handle* h, const Plan& P, int l, const Bufs& B) {
  const qwen3_config& c = h->cfg;
  const qwen3_layer_weights& W = h->layers[l];
  QkRopeArgs r{};
  r.qkv = B.qkv; r.T = P.T; r.H = c.n_heads; r.KV = c.n_kv_heads; r.D = c.head_dim; r.q_out = B.q;
  r.kcache = static_cast<char*>(h->kcache) + (size_t)l * h->layer_stride * h->esz;
  r.vcache = static_cast<char*>(h->vcache) + (size_t)l * h->layer_stride * h->esz;
  r.seq_stride = (long long)h->seq_stride; r.capacity = c.capacity; r.q_gain = W.q_norm; r.k_gain = W.k_norm;
  r.cos_t = h->rope_cos; r.sin_t = h->rope_sin; r.row_seq = B.desc + P.off_rowseq; r.row_pos = B.desc + P.off_rowpos;
  r.eps = c.rms_eps; r.cs_bf16 = h->rope_cs16;
  return r;
}

// Attention of layer l for the plan's kernel (qk_done: the q|k|v GEMM's
// epilogue already normalised, rotated and appended the rows).
cudaError_t enqueue_attention(qwen3_handle* h, Launcher& L, const Plan& P, int l, const Bufs& B,
                              const void* pf = nullptr, size_t pf_bytes = 0, const void* pf2 = nullptr,
                              size_t pf2_bytes = 0, bool qk_done = false) {
  const qwen3_config& c = h->cfg;
  const qwen3_layer_weights& W = h->layers[l];
  const int dt = h->dt, KV = c.n_kv_heads, D = c.head_dim;
  char* kc = static_cast<char*>(h->kcache) + (size_t)l * h->layer_stride * h->esz;
  char* vc = static_cast<char*>(h->vcache) + (size_t)l * h->layer_stride * h->esz;
  const int32_t* row_seq = B.desc + P.off_rowseq;
  const int32_t* row_pos = B.desc + P.off_rowpos;
  const int32_t* n_items = B.desc + P.off_nitems;
  const AttnQBlock* qbs = reinterpret_cast<const AttnQBlock*>(B.desc + P.off_qb);
  const AttnItem* items = reinterpret_cast<const AttnItem*>(B.desc + P.off_items);
  const float scale = (float)(1.0 / std::sqrt((double)D));
  cudaError_t e;
  if (P.attn == ATTN_DECODE) {
    AttnDecArgs a{};
    a.qkv = B.qkv; a.H = c.n_heads; a.KV = KV; a.D = D; a.q_gain = W.q_norm; a.k_gain = W.k_norm;
    a.cos_t = h->rope_cos; a.sin_t = h->rope_sin; a.eps = c.rms_eps; a.kc = kc; a.vc = vc;
    a.seq_stride = (long long)h->seq_stride; a.capacity = c.capacity; a.n_seqs = c.max_seqs; a.scale = scale;
    a.qblocks = qbs;
    a.items = items; a.n_items = n_items; a.part_o = B.part_o; a.part_ml = B.part_ml; a.nq_max = P.nq_max;
    a.counters = B.counters; a.out = B.attn; a.err = B.err;
    a.grid_x = std::max(1, (h->num_sms + KV - 1) / KV);
    a.nq = P.max_nq;
    a.runs = P.n_items > a.grid_x;
    if (P.cluster > 1) {
      a.cluster = P.cluster;
      a.grid_x = P.cluster * P.n_qblocks;
      a.runs = 0;
    }
    a.pf = pf; a.pf_bytes = pf_bytes; a.pf2 = pf2; a.pf2_bytes = pf2_bytes;
    return launch(L, a.cluster > 1 ? "attn_decode_cluster" : "attn_decode",
                  [&] { return launch_attn_decode2(L.ctx, dt, a); });
  }
  if (!qk_done) {
    const QkRopeArgs r = qk_rope_args(h, P, l, B);
    e = launch(L, "qk_rope_cache", [&] { return launch_qk_rope_cache(L.ctx, dt, r); });
    if (e != cudaSuccess) return e;
  }
  if (P.attn == ATTN_TC) {
    AttnTcArgs t{};
    t.qblocks = qbs; t.n_qblocks = P.n_qblocks; t.T = P.T; t.H = c.n_heads; t.KV = KV; t.D = D;
    t.capacity = c.capacity; t.max_seqs = c.max_seqs; t.seq_stride = (long long)h->seq_stride;
    t.q = B.q; t.kc = kc; t.vc = vc; t.out = B.attn;
    t.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    t.err = B.err;
    return launch(L, "attn_tc", [&] { return launch_attn_tc(L.ctx, t); });
  }
  AttnArgs a{};
  a.q = B.q; a.kc = kc; a.vc = vc; a.seq_stride = (long long)h->seq_stride; a.capacity = c.capacity;
  a.H = c.n_heads; a.KV = KV; a.D = D; a.scale = scale; a.qblocks = qbs; a.items = items; a.n_items = n_items;
  a.chunk = P.chunk; a.nq_max = P.nq_max; a.part_o = B.part_o; a.part_ml = B.part_ml; a.counters = B.counters;
  a.out = B.attn;
  a.grid_x = std::max(1, std::min((h->num_sms * 8 + KV - 1) / KV, P.n_items));
  return launch(L, "attn_prefill", [&] { return launch_attention_prefill(L.ctx, dt, a); });
}

// Decode plan (T <= 4): five kernels per dense layer.  The residual stream
// lives in hA and is updated in place; sumsq holds, per row, the sum of
// squares of h entering each RMSNorm: slot 2l (input norm of layer l >= 1),
// 2l + 1 (post-attention norm of layer l), 2L (final norm).
cudaError_t enqueue_decode(qwen3_handle* h, Launcher& L, const Plan& P, const void* x, void* out, const Bufs& B) {
  const qwen3_config& c = h->cfg;
  const int T = P.T, hid = c.hidden, H = c.n_heads, KV = c.n_kv_heads, D = c.head_dim, I = c.intermediate;
  const int NL = c.num_layers;
  const int dt = h->dt, wf = h->wfmt;
  const int qkv_rows = (H + 2 * KV) * D;
  void* hres = B.hA;
  auto slot = [&](int s) { return B.sumsq + (size_t)s * T; };
  auto wfmt_of = [&](const qwen3_linear& lin) { return lin.scale ? wf : W_DT; };
  // bytes of a linear's weight matrix (the codes for int8), for L2 prefetch
  auto lin_bytes = [&](const qwen3_linear& lin, int rows, int K) {
    return (size_t)rows * K * (lin.scale ? 1 : h->esz);
  };
  // L2 prefetch of weights ahead of their kernels: 1 = each kernel asks for
  // the next one's; 2 = the attention kernel (far below the HBM rate) asks
  // for o_proj's and gate|up's, o_proj for down's, down for the next qkv's.
  const int pf_mode = h->l2_prefetch;
  const bool pf_on = pf_mode == 1;
  cudaError_t e;
  for (int l = 0; l < NL; ++l) {
    const qwen3_layer_weights& W = h->layers[l];
    {
      Gemv2Args g{};
      g.T = T; g.K = hid; g.N = qkv_rows; g.w = W.qkv.w; g.scale = W.qkv.scale; g.bias = W.qkv.bias;
      g.group = c.group_size; g.gain = W.in_norm; g.eps = c.rms_eps; g.h = hres; g.epilogue = EPI_STORE;
      g.out = B.qkv; g.ldo = qkv_rows; g.err = B.err;
      if (l == 0) {
        g.prologue = PRO_FULL; g.x = x; g.pend = nullptr; g.sumsq_zero = slot(1); g.sumsq_zero_n = 2 * NL * T;
      } else {
        g.prologue = PRO_SUMSQ; g.sumsq_in = slot(2 * l);
      }
      g.stages = gemv2_plan(dt, wfmt_of(W.qkv), T, hid, c.group_size, false, &g.nwarps, h->coresident);
      e = launch(L, "gemv_qkv", [&] { return launch_gemv2(L.ctx, dt, wfmt_of(W.qkv), g); });
      if (e != cudaSuccess) return e;
    }
    const bool moe = is_moe_layer(h, l);
    if (pf_mode == 2 && !moe)
      e = enqueue_attention(h, L, P, l, B, W.o.w, lin_bytes(W.o, hid, H * D), W.gate_up.w,
                            lin_bytes(W.gate_up, 2 * I, hid));
    else
      e = enqueue_attention(h, L, P, l, B, pf_mode ? W.o.w : nullptr, lin_bytes(W.o, hid, H * D));
    if (e != cudaSuccess) return e;
    {
      Gemv2Args g{};
      g.T = T; g.K = H * D; g.N = hid; g.w = W.o.w; g.scale = W.o.scale; g.bias = W.o.bias; g.group = c.group_size;
      g.prologue = PRO_X; g.x = B.attn; g.epilogue = EPI_RESIDUAL; g.out = hres; g.ldo = hid;
      g.sumsq_out = slot(2 * l + 1); g.err = B.err;
      if (pf_on && !moe) { g.pf = W.gate_up.w; g.pf_bytes = lin_bytes(W.gate_up, 2 * I, hid); }
      if (pf_mode == 2 && !moe) { g.pf = W.down.w; g.pf_bytes = lin_bytes(W.down, hid, I); }
      g.stages = gemv2_plan(dt, wfmt_of(W.o), T, H * D, c.group_size, false, &g.nwarps, h->coresident);
      e = launch(L, "gemv_o", [&] { return launch_gemv2(L.ctx, dt, wfmt_of(W.o), g); });
      if (e != cudaSuccess) return e;
    }
    if (moe) {
      // the post-attention RMSNorm runs in the router GEMV's prologue
      e = moe_block(h, L, l, B.y, T, nullptr, hres, slot(2 * l + 2), B.idx, B.wts, B, slot(2 * l + 1));
      if (e != cudaSuccess) return e;
      continue;
    }
    {
      Gemv2Args g{};
      g.T = T; g.K = hid; g.N = I; g.w = W.gate_up.w; g.scale = W.gate_up.scale; g.bias = W.gate_up.bias;
      g.group = c.group_size; g.prologue = PRO_SUMSQ; g.h = hres; g.gain = W.post_norm; g.eps = c.rms_eps;
      g.sumsq_in = slot(2 * l + 1); g.epilogue = EPI_SWIGLU; g.out = B.m; g.ldo = I; g.err = B.err;
      if (pf_on) { g.pf = W.down.w; g.pf_bytes = lin_bytes(W.down, hid, I); }
      g.stages = gemv2_plan(dt, wfmt_of(W.gate_up), T, hid, c.group_size, true, &g.nwarps, h->coresident);
      e = launch(L, "gemv_gate_up", [&] { return launch_gemv2(L.ctx, dt, wfmt_of(W.gate_up), g); });
      if (e != cudaSuccess) return e;
    }
    {
      Gemv2Args g{};
      g.T = T; g.K = I; g.N = hid; g.w = W.down.w; g.scale = W.down.scale; g.bias = W.down.bias;
      g.group = c.group_size; g.prologue = PRO_X; g.x = B.m; g.epilogue = EPI_RESIDUAL; g.out = hres; g.ldo = hid;
      g.sumsq_out = slot(2 * l + 2); g.err = B.err;
      if (pf_mode && l + 1 < NL) { g.pf = h->layers[l + 1].qkv.w; g.pf_bytes = lin_bytes(h->layers[l + 1].qkv, qkv_rows, hid); }
      g.stages = gemv2_plan(dt, wfmt_of(W.down), T, I, c.group_size, false, &g.nwarps, h->coresident);
      e = launch(L, "gemv_down", [&] { return launch_gemv2(L.ctx, dt, wfmt_of(W.down), g); });
      if (e != cudaSuccess) return e;
    }
  }
  NormApplyArgs n{};
  n.h = hres; n.sumsq = slot(2 * NL); n.gain = h->final_norm; n.out = out; n.T = T; n.hidden = hid;
  n.eps = c.rms_eps;
  return launch(L, "norm_apply", [&] { return launch_norm_apply(L.ctx, dt, n); });
}

// Kernel names of one linear under each GEMM it may run on (profiling keys).
struct LinNames {
  const char *tc, *w8tc, *skinny, *simt;
};
constexpr LinNames kQkv{"gemm_tc_qkv", "gemm_w8tc_qkv", "gemm_skinny_qkv", "gemm_qkv"};
constexpr LinNames kO{"gemm_tc_o", "gemm_w8tc_o", "gemm_skinny_o", "gemm_o"};
constexpr LinNames kGateUp{"gemm_tc_gate_up", "gemm_w8tc_gate_up", "gemm_skinny_gate_up", "gemm_gate_up"};
constexpr LinNames kDown{"gemm_tc_down", "gemm_w8tc_down", "gemm_skinny_down", "gemm_down"};

// A prefill linear: the tcgen05 GEMM for dense bf16 weights on shapes its
// tile takes, the CUDA-core GEMM otherwise (fp32, int8, ragged N).
cudaError_t linear_gemm(qwen3_handle* h, Launcher& L, const LinNames& nm, int wfmt, const GemmArgs& g,
                        const Bufs& B) {
  if (h->use_tc && h->dt == DT_BF16 && wfmt == W_DT && !g.a_rows && !g.c_rows && !g.tile_start &&
      gemm_tc_supported(g.M, g.N, g.K, g.epilogue)) {
    GemmTcArgs t{};
    t.M = g.M; t.N = g.N; t.K = g.K; t.a = g.a; t.lda = g.lda; t.w = g.w; t.out = g.out; t.ldo = g.ldo;
    t.epilogue = g.epilogue; t.err = B.err;
    // one row tile and few column tiles: split k over the SMs, then add the
    // partial tiles in range order
    const int S = B.tcpart ? gemm_tc_splits(g.M, g.N, g.K, g.epilogue, h->num_sms) : 1;
    if (S > 1 && gemm_tc_part_floats(g.M, g.N, g.epilogue, S) <= B.tcpart_floats) {
      t.splits = S;
      t.part = B.tcpart;
    }
    cudaError_t e = launch(L, nm.tc, [&] { return launch_gemm_tc(L.ctx, t); });
    if (e != cudaSuccess || t.splits < 2) return e;
    return launch(L, "gemm_tc_reduce", [&] { return launch_gemm_tc_reduce(L.ctx, t); });
  }
  if (g.M <= 64 && !g.a_rows && !g.c_rows && !g.tile_start && gemm_skinny_supported(g.M, g.N, g.K) && h->skws.p) {
    SkinnyArgs k{};
    k.M = g.M; k.N = g.N; k.K = g.K; k.a = g.a; k.lda = g.lda; k.w = g.w; k.scale = g.scale; k.bias = g.bias;
    k.group = g.group; k.epilogue = g.epilogue; k.out = g.out; k.ldo = g.ldo;
    k.ws = static_cast<float*>(h->skws.p); k.counters = static_cast<int*>(h->skcnt.p); k.err = B.err;
    if (h->use_tc && h->dt == DT_BF16 && wfmt == W_U8 && gemm_w8_tc_supported(g.M, g.N, g.K, g.group, g.epilogue))
      return launch(L, nm.w8tc, [&] { return launch_gemm_w8_tc(L.ctx, k); });
    return launch(L, nm.skinny, [&] { return launch_gemm_skinny(L.ctx, h->dt, wfmt, k); });
  }
  return launch(L, nm.simt, [&] { return launch_gemm_simt(L.ctx, h->dt, wfmt, g); });
}

// Prefill plan (T > 4): add+RMSNorm kernels, tiled GEMMs, ping-pong residual.
cudaError_t enqueue_prefill(qwen3_handle* h, Launcher& L, const Plan& P, const void* x, void* out, const Bufs& B) {
  const qwen3_config& c = h->cfg;
  const int T = P.T, hid = c.hidden, H = c.n_heads, KV = c.n_kv_heads, D = c.head_dim, I = c.intermediate;
  const int dt = h->dt, wf = h->wfmt;
  const int qkv_rows = (H + 2 * KV) * D;
  auto wfmt_of = [&](const qwen3_linear& lin) { return lin.scale ? wf : W_DT; };
  cudaError_t e;
  const void* h_in = x;   // residual stream entering the layer
  void* h_cur = B.hA;     // residual stream of the current layer
  bool have_pend = false;
  for (int l = 0; l < c.num_layers; ++l) {
    const qwen3_layer_weights& W = h->layers[l];
    NormArgs n{};
    n.h_in = h_in; n.pend = have_pend ? B.pend : nullptr; n.h_out = h_cur; n.y = B.y; n.gain = W.in_norm;
    n.rows = T; n.hidden = hid; n.eps = c.rms_eps;
    e = launch(L, "add_rmsnorm", [&] { return launch_add_rmsnorm(L.ctx, dt, n); });
    if (e != cudaSuccess) return e;
    // bf16 on tensor cores: q/k RMSNorm, RoPE and the cache append run in the
    // q|k|v GEMM's epilogue (the rows never reach global memory) when the
    // tiles fill at least one wave, so that most epilogues overlap the next
    // tile's MMAs; with fewer tiles every epilogue is exposed and the separate
    // kernel is faster (4 x 512-row chunks: 116k against 124k tok/s)
    const int qkv_tiles = ((T + 127) / 128) * (qkv_rows / 256);
    const bool qk_fused = P.attn != ATTN_DECODE && h->use_tc && dt == DT_BF16 && wfmt_of(W.qkv) == W_DT &&
                          qkv_tiles >= h->num_sms && gemm_tc_qkrope_supported(T, H, KV, D) &&
                          gemm_tc_supported(T, qkv_rows, hid, EPI_QKROPE);
    if (qk_fused) {
      GemmTcArgs t{};
      t.M = T; t.N = qkv_rows; t.K = hid; t.a = B.y; t.lda = hid; t.w = W.qkv.w; t.out = nullptr; t.ldo = qkv_rows;
      t.epilogue = EPI_QKROPE; t.err = B.err; t.rope = qk_rope_args(h, P, l, B);
      e = launch(L, "gemm_tc_qkv_rope", [&] { return launch_gemm_tc(L.ctx, t); });
    } else {
      GemmArgs g{};
      g.M = T; g.N = qkv_rows; g.K = hid; g.a = B.y; g.lda = hid; g.w = W.qkv.w; g.scale = W.qkv.scale;
      g.bias = W.qkv.bias; g.group = c.group_size; g.epilogue = EPI_STORE; g.out = B.qkv; g.ldo = qkv_rows;
      e = linear_gemm(h, L, kQkv, wfmt_of(W.qkv), g, B);
    }
    if (e != cudaSuccess) return e;
    e = enqueue_attention(h, L, P, l, B, nullptr, 0, nullptr, 0, qk_fused);
    if (e != cudaSuccess) return e;
    GemmArgs go{};
    go.M = T; go.N = hid; go.K = H * D; go.a = B.attn; go.lda = H * D; go.w = W.o.w; go.scale = W.o.scale;
    go.bias = W.o.bias; go.group = c.group_size; go.epilogue = EPI_RESIDUAL; go.out = h_cur; go.ldo = hid;
    e = linear_gemm(h, L, kO, wfmt_of(W.o), go, B);
    if (e != cudaSuccess) return e;
    NormArgs n2{};
    n2.h_in = h_cur; n2.pend = nullptr; n2.h_out = h_cur; n2.y = B.y; n2.gain = W.post_norm; n2.rows = T;
    n2.hidden = hid; n2.eps = c.rms_eps;
    e = launch(L, "add_rmsnorm", [&] { return launch_add_rmsnorm(L.ctx, dt, n2); });
    if (e != cudaSuccess) return e;
    if (is_moe_layer(h, l)) {
      e = moe_block(h, L, l, B.y, T, B.pend, nullptr, nullptr, B.idx, B.wts, B);
      if (e != cudaSuccess) return e;
    } else {
      GemmArgs gu{};
      gu.M = T; gu.N = I; gu.K = hid; gu.a = B.y; gu.lda = hid; gu.w = W.gate_up.w; gu.scale = W.gate_up.scale;
      gu.bias = W.gate_up.bias; gu.group = c.group_size; gu.epilogue = EPI_SWIGLU; gu.out = B.m; gu.ldo = I;
      e = linear_gemm(h, L, kGateUp, wfmt_of(W.gate_up), gu, B);
      if (e != cudaSuccess) return e;
      GemmArgs d{};
      d.M = T; d.N = hid; d.K = I; d.a = B.m; d.lda = I; d.w = W.down.w; d.scale = W.down.scale;
      d.bias = W.down.bias; d.group = c.group_size; d.epilogue = EPI_STORE; d.out = B.pend; d.ldo = hid;
      e = linear_gemm(h, L, kDown, wfmt_of(W.down), d, B);
      if (e != cudaSuccess) return e;
    }
    have_pend = true;
    h_in = h_cur;
    h_cur = (h_cur == B.hA) ? B.hB : B.hA;
  }
  // final: out = RMSNorm(R(h + pend)) with the final gain
  NormArgs n{};
  n.h_in = h_in; n.pend = B.pend; n.h_out = h_cur; n.y = out; n.gain = h->final_norm; n.rows = T; n.hidden = hid;
  n.eps = c.rms_eps;
  return launch(L, "add_rmsnorm", [&] { return launch_add_rmsnorm(L.ctx, dt, n); });
}

cudaError_t enqueue_forward(qwen3_handle* h, Launcher& L, const Plan& P, const void* x, void* out, const Bufs& B) {
  return P.gemv ? enqueue_decode(h, L, P, x, out, B) : enqueue_prefill(h, L, P, x, out, B);
}

}  // namespace

extern "C" qwen3_status qwen3_forward(qwen3_handle* h, const void* x, int32_t T, const int32_t* seq_ids,
                                      const int32_t* positions, void* out, void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (!x || !out || !seq_ids || !positions) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (T < 1 || T > (1 << 20)) return fail(h, QWEN3_E_ARG, "row count out of range");
  if (!aligned16(x) || !aligned16(out)) return fail(h, QWEN3_E_ARG, "x and out must be 16-byte aligned");
  Plan P;
  qwen3_status st = build_plan(h, T, seq_ids, positions, P);
  if (st != QWEN3_OK) return st;
  if (h->cluster_attn) P.cluster = decode_cluster_size(h, P);
  st = ensure_workspace(h, P, T);
  if (st != QWEN3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Bufs B = bufs_of(h);
  Launcher L{h, {s, h->pdl && !h->profile, h->num_sms}};
  st = upload_plan(h, P, s);
  if (st != QWEN3_OK) return st;
  const bool graph = h->use_graphs && !h->profile && P.gemv;
  cudaError_t e;
  if (graph) {
    const int runs = P.attn == ATTN_DECODE && P.n_items > std::max(1, (h->num_sms + h->cfg.n_kv_heads - 1) / h->cfg.n_kv_heads);
    const GraphKey key{T, P.attn * 64 + P.max_nq + (runs ? 32 : 0) + (P.cluster > 1 ? 16 : 0), x, out};
    if (h->graphs.size() > 32) {  // callers cycling through buffers: start over
      for (auto& g : h->graphs) cudaGraphExecDestroy(g.second.first);
      h->graphs.clear();
    }
    auto it = h->graphs.find(key);
    if (it != h->graphs.end() && it->second.second != h->ws_generation) {
      cudaGraphExecDestroy(it->second.first);
      h->graphs.erase(it);
      it = h->graphs.end();
    }
    if (it == h->graphs.end()) {
      Launcher G{h, {h->gstream, h->pdl, h->num_sms}};
      cudaGraph_t g = nullptr;
      e = cudaStreamBeginCapture(h->gstream, cudaStreamCaptureModeThreadLocal);
      if (e != cudaSuccess) return cuda_fail(h, e, "graph capture begin");
      cudaError_t ee = enqueue_forward(h, G, P, x, out, B);
      e = cudaStreamEndCapture(h->gstream, &g);
      if (ee != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_fail(h, ee, "graph capture");
      }
      if (e != cudaSuccess) return cuda_fail(h, e, "graph capture end");
      cudaGraphExec_t ex = nullptr;
      e = cudaGraphInstantiate(&ex, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return cuda_fail(h, e, "graph instantiate");
      it = h->graphs.emplace(key, std::make_pair(ex, h->ws_generation)).first;
      h->launches = G.count;
    }
    // x and out are part of the key: a graph is replayed only with the buffers it was captured on.
    cudaGraphExec_t ex = it->second.first;
    e = cudaEventRecord(h->ev_in, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->gstream, h->ev_in, 0);
    if (e == cudaSuccess) e = cudaGraphLaunch(ex, h->gstream);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_out, h->gstream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_out, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "graph launch");
    h->last_launches = h->launches;
  } else {
    e = enqueue_forward(h, L, P, x, out, B);
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
    h->last_launches = L.count;
  }
  for (int t = 0; t < T; ++t) h->lengths[seq_ids[t]] = positions[t] + 1;
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_moe_layer(qwen3_handle* h, int32_t layer, const void* y, int32_t T, void* out,
                                        int32_t* topk_idx, float* topk_w, void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (!y || !out || !topk_idx || !topk_w) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (layer < 0 || layer >= h->cfg.num_layers || !is_moe_layer(h, layer))
    return fail(h, QWEN3_E_ARG, "layer is not a MoE layer");
  if (T < 1 || T > (1 << 20)) return fail(h, QWEN3_E_ARG, "row count out of range");
  Plan P;
  P.T = T;
  P.gemv = T <= 4;
  qwen3_status st = ensure_workspace(h, P, T);
  if (st != QWEN3_OK) return st;
  Bufs B = bufs_of(h);
  Launcher L{h, {static_cast<cudaStream_t>(stream), h->pdl && !h->profile, h->num_sms}};
  cudaError_t e = moe_block(h, L, layer, y, T, out, nullptr, nullptr, topk_idx, topk_w, B);
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  h->last_launches = L.count;
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_selftest_bounded_wait(qwen3_handle* h, void* stream) {
  if (!h) return QWEN3_E_ARG;
  cudaError_t e = launch_wait_probe(static_cast<cudaStream_t>(stream), static_cast<int*>(h->dev_err.p));
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_device_error(qwen3_handle* h, int32_t* code) {
  if (!h || !code) return QWEN3_E_ARG;
  *code = 0;
  if (!h->dev_err.p) return QWEN3_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "device error poll");
  int v = 0;
  cudaMemcpy(&v, h->dev_err.p, sizeof(int), cudaMemcpyDeviceToHost);
  if (v) {
    cudaMemset(h->dev_err.p, 0, sizeof(int));
    *code = v;
    return fail(h, QWEN3_E_DEVICE, "a kernel gave up waiting for its data (code " + std::to_string(v) + ")");
  }
  return QWEN3_OK;
}

// ======================================================================
// embedding rows, output head, pooled sentence vector
// ======================================================================
namespace {

// Host ints -> device buffer through the pinned staging ring.
qwen3_status upload_ints(qwen3_handle* h, const int32_t* v, int n, DevBuf& dst, cudaStream_t s) {
  qwen3_status st = ensure(h, dst, (size_t)n * 4 + 64, false);
  if (st != QWEN3_OK) return st;
  const int i = h->ring_pos;
  h->ring_pos = (h->ring_pos + 1) % qwen3_handle::kRing;
  cudaEventSynchronize(h->pinned_ev[i]);
  const size_t bytes = (size_t)n * 4;
  if (h->pinned_bytes[i] < bytes) {
    if (h->pinned[i]) cudaFreeHost(h->pinned[i]);
    h->pinned[i] = nullptr;
    const size_t nb = std::max(bytes, (size_t)4096) * 2;
    if (cudaHostAlloc(&h->pinned[i], nb, cudaHostAllocDefault) != cudaSuccess) {
      cudaGetLastError();
      h->pinned_bytes[i] = 0;
      return fail(h, QWEN3_E_OOM, "pinned host allocation failed");
    }
    h->pinned_bytes[i] = nb;
  }
  std::memcpy(h->pinned[i], v, bytes);
  cudaError_t e = cudaMemcpyAsync(dst.p, h->pinned[i], bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "id upload");
  cudaEventRecord(h->pinned_ev[i], s);
  return QWEN3_OK;
}

}  // namespace

extern "C" qwen3_status qwen3_embed(qwen3_handle* h, const void* table, int32_t vocab, const int32_t* ids, int32_t n,
                                    void* out, void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (!table || !ids || !out) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (vocab < 1 || n < 1 || n > (1 << 20)) return fail(h, QWEN3_E_ARG, "vocab or row count out of range");
  if (!aligned16(table) || !aligned16(out)) return fail(h, QWEN3_E_ARG, "table and out must be 16-byte aligned");
  for (int t = 0; t < n; ++t)
    if (ids[t] < 0 || ids[t] >= vocab)
      return fail(h, QWEN3_E_ARG, "token id " + std::to_string(ids[t]) + " at row " + std::to_string(t) +
                                      " is outside [0, " + std::to_string(vocab) + ")");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  qwen3_status st = upload_ints(h, ids, n, h->ids, s);
  if (st != QWEN3_OK) return st;
  Launcher L{h, {s, h->pdl && !h->profile, h->num_sms}};
  EmbedArgs a{table, static_cast<const int*>(h->ids.p), n, h->cfg.hidden, out};
  cudaError_t e = launch(L, "embed_gather", [&] { return launch_embed_gather(L.ctx, h->dt, a); });
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  h->last_launches = L.count;
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_head(qwen3_handle* h, const void* w, int32_t n_out, const void* x, int32_t T,
                                   float* logits, void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (!w || !x || !logits) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (n_out < 1 || T < 1 || T > (1 << 20)) return fail(h, QWEN3_E_ARG, "row or output count out of range");
  if (!aligned16(w) || !aligned16(x)) return fail(h, QWEN3_E_ARG, "w and x must be 16-byte aligned");
  const int hid = h->cfg.hidden;
  Launcher L{h, {static_cast<cudaStream_t>(stream), h->pdl && !h->profile, h->num_sms}};
  cudaError_t e;
  if (T <= 4) {
    GemvArgs g{};
    g.T = T; g.K = hid; g.N = n_out; g.w = w; g.x_rows = T; g.x = x; g.epilogue = EPI_STORE_RF32;
    g.out = logits; g.ldo = n_out;
    e = launch(L, "gemv_head", [&] { return launch_gemv(L.ctx, h->dt, W_DT, g); });
  } else {
    GemmArgs g{};
    g.M = T; g.N = n_out; g.K = hid; g.a = x; g.lda = hid; g.w = w; g.epilogue = EPI_STORE_RF32;
    g.out = logits; g.ldo = n_out;
    e = launch(L, "gemm_head", [&] { return launch_gemm_simt(L.ctx, h->dt, W_DT, g); });
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  h->last_launches = L.count;
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_embed_pooled(qwen3_handle* h, const void* x, int32_t T, int32_t seq, void* out,
                                           void* stream) {
  if (!h) return QWEN3_E_ARG;
  if (!x || !out) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (seq < 0 || seq >= h->cfg.max_seqs) return fail(h, QWEN3_E_SEQ, "sequence id out of range");
  if (T < 1 || T > h->cfg.capacity)
    return fail(h, QWEN3_E_CAPACITY, "row count must be in [1, capacity] (the sequence restarts at position 0)");
  if (!aligned16(x) || !aligned16(out)) return fail(h, QWEN3_E_ARG, "x and out must be 16-byte aligned");
  const size_t row_bytes = (size_t)h->cfg.hidden * h->esz;
  qwen3_status st = ensure(h, h->pool_rows, (size_t)T * row_bytes, false);
  if (st != QWEN3_OK) return st;
  std::vector<int32_t> sids(T, seq), pos(T);
  for (int t = 0; t < T; ++t) pos[t] = t;
  const int32_t saved = h->lengths[seq];
  h->lengths[seq] = 0;  // positions 0..T-1 of a fresh sequence (the cache is cleared below)
  Plan P;
  st = build_plan(h, T, sids.data(), pos.data(), P);
  h->lengths[seq] = saved;
  if (st != QWEN3_OK) return st;
  st = qwen3_reset(h, seq, stream);
  if (st != QWEN3_OK) return st;
  st = qwen3_forward(h, x, T, sids.data(), pos.data(), h->pool_rows.p, stream);
  if (st != QWEN3_OK) return st;
  const int64_t fwd_launches = h->last_launches;
  Launcher L{h, {static_cast<cudaStream_t>(stream), h->pdl && !h->profile, h->num_sms}};
  L2PoolArgs a{static_cast<const char*>(h->pool_rows.p) + (size_t)(T - 1) * row_bytes, h->cfg.hidden, out};
  cudaError_t e = launch(L, "l2_pool", [&] { return launch_l2_pool(L.ctx, h->dt, a); });
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  h->last_launches = fwd_launches + L.count;
  return QWEN3_OK;
}

extern "C" qwen3_status qwen3_workspace_bytes(const qwen3_handle* h, int64_t* bytes) {
  if (!h || !bytes) return QWEN3_E_ARG;
  const DevBuf* bufs[] = {&h->hA, &h->hB, &h->pend, &h->y, &h->qkv, &h->q, &h->attn, &h->mbuf, &h->logits, &h->idx,
                          &h->wts, &h->counts, &h->row_off, &h->row_cnt, &h->tile_start, &h->cursor, &h->sorted_tok,
                          &h->sorted_src, &h->mexp, &h->zexp, &h->part_o, &h->part_ml, &h->counters, &h->desc,
                          &h->sumsq, &h->dev_err, &h->skws, &h->skcnt, &h->ysort, &h->ids,
                          &h->pool_rows, &h->rlpart, &h->rlcnt, &h->tcpart};
  int64_t n = 0;
  for (const DevBuf* b : bufs) n += (int64_t)b->bytes;
  *bytes = n;
  return QWEN3_OK;
}

// ======================================================================
// MoE block on caller-provided scratch (used by qwen3_moe_layer_static)
// ======================================================================
namespace {

// Scratch of the MoE block for T rows, carved in 256-byte-aligned pieces.
// [0, zeroed) holds the expert histogram and the scatter cursors, which the
// router and the scatter expect at zero.
struct MoeScratch {
  size_t counts, cursor, zeroed, row_off, row_cnt, tile_start, logits, sorted_tok, sorted_src, mexp, zexp, total;
};

MoeScratch moe_scratch_layout(const qwen3_config& c, size_t esz, size_t T) {
  MoeScratch s{};
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t o = off;
    off += (n + 255) / 256 * 256;
    return o;
  };
  const size_t E = (size_t)c.num_experts, slots = T * (size_t)c.top_k;
  s.counts = take(E * 4);
  s.cursor = take(E * 4);
  s.zeroed = off;
  s.row_off = take(E * 4);
  s.row_cnt = take(E * 4);
  s.tile_start = take((E + 1) * 4);
  s.logits = take(T * E * 4);
  s.sorted_tok = take(slots * 4);
  s.sorted_src = take(slots * 4);
  s.mexp = take(slots * (size_t)c.moe_intermediate * esz);
  s.zexp = take(slots * (size_t)c.hidden * esz);
  s.total = off;
  return s;
}

}  // namespace

namespace q3 {

int handle_device(const qwen3_handle* h) { return h->device; }

qwen3_status report_error(qwen3_handle* h, qwen3_status s, const char* msg) { return fail(h, s, msg); }

// qwen3_moe_layer with every scratch buffer taken from the device region
// [scratch, scratch + scratch_bytes) instead of the handle's workspace: the
// call allocates nothing and leaves the workspace as it is.  The region's
// zero-initialised part is cleared on `stream` before the kernels.
qwen3_status moe_layer_on_scratch(qwen3_handle* h, int32_t layer, const void* y, int32_t T, void* out,
                                  int32_t* topk_idx, float* topk_w, void* stream, void* scratch,
                                  size_t scratch_bytes) {
  if (!y || !out || !topk_idx || !topk_w || !scratch) return fail(h, QWEN3_E_ARG, "null pointer argument");
  if (layer < 0 || layer >= h->cfg.num_layers || !is_moe_layer(h, layer))
    return fail(h, QWEN3_E_ARG, "layer is not a MoE layer");
  if (T < 1 || T > (1 << 20)) return fail(h, QWEN3_E_ARG, "row count out of range");
  if (h->profile) return fail(h, QWEN3_E_UNSUPPORTED, "turn QWEN3_OPT_PROFILE off for the static-scratch MoE layer");
  const MoeScratch S = moe_scratch_layout(h->cfg, h->esz, (size_t)T);
  if (S.total > scratch_bytes) {
    int lo = 0, hi = T;  // largest row count that fits
    while (lo < hi) {
      const int mid = lo + (hi - lo + 1) / 2;
      if (moe_scratch_layout(h->cfg, h->esz, (size_t)mid).total <= scratch_bytes) lo = mid; else hi = mid - 1;
    }
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "%d rows need %zu bytes of scratch, more than the %zu-byte static scratch; at most %d rows of "
                  "this model fit per call",
                  T, S.total, scratch_bytes, lo);
    return fail(h, QWEN3_E_ARG, msg);
  }
  char* base = static_cast<char*>(scratch);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(base, 0, S.zeroed, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "static scratch clear");
  Bufs B{};
  B.counts = reinterpret_cast<int*>(base + S.counts);
  B.cursor = reinterpret_cast<int*>(base + S.cursor);
  B.row_off = reinterpret_cast<int*>(base + S.row_off);
  B.row_cnt = reinterpret_cast<int*>(base + S.row_cnt);
  B.tile_start = reinterpret_cast<int*>(base + S.tile_start);
  B.logits = reinterpret_cast<float*>(base + S.logits);
  B.sorted_tok = reinterpret_cast<int*>(base + S.sorted_tok);
  B.sorted_src = reinterpret_cast<int*>(base + S.sorted_src);
  B.mexp = base + S.mexp;
  B.zexp = base + S.zexp;
  // The tensor-core path gathers the rows into expert order first (ysort,
  // slots x hidden, the size of zexp).  ysort is read only by the gate|up GEMM
  // and zexp is first written by the down GEMM, which starts after it (stream
  // order; its stores follow its wait on the gate|up kernel), so the two share
  // one region.
  if (h->dt == DT_BF16 && T > 4) B.ysort = B.zexp;
  B.err = static_cast<int*>(h->dev_err.p);
  Launcher L{h, {s, h->pdl, h->num_sms}};
  e = moe_block(h, L, layer, y, T, out, nullptr, nullptr, topk_idx, topk_w, B);
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  h->last_launches = L.count;
  return QWEN3_OK;
}

}  // namespace q3
