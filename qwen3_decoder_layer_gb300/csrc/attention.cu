// GQA causal attention over the static KV cache (maya2_mlx/backbone.py,
// Backbone.forward: `mx.fast.scaled_dot_product_attention(q, K[:p0+T],
// V[:p0+T], scale=D^-0.5, mask="causal" if T > 1)`, "attention over keys
// 0..pos (fp32 softmax, one rounding)"; q head h reads kv head h / (H/KV), the
// repeat_kv of rlx_flow/blocks/qwen3_decoder.rs).
//
// Split-K ("flash-decoding") structure: the keys of each query block are cut
// into fixed-size chunks; each (query block, chunk, kv head) item computes the
// chunk's fp32 scores, their max m, sum l = sum exp(s - m) and the
// unnormalised output sum exp(s - m) v, and stores them.  The last item of a
// (query block, kv head) to finish -- counted with an atomic, no waiting --
// merges the chunks: M = max m_c, out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
// rounded once to the model dtype.  A persistent grid (kv head on y) walks
// the item list, so one launch shape serves every context length.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int PRE_CK = 64, PRE_NQ = 32, PRE_THREADS = 128;

// Merge the partials of one (query block, kv head); called by the whole block.
template <typename Dt, int D>
__device__ void combine(const AttnArgs& a, const AttnQBlock& qb, int j) {
  const int G = a.H / a.KV;
  const int nq = qb.nrows * G;
  for (int idx = threadIdx.x; idx < nq * D; idx += blockDim.x) {
    const int i = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
    for (int c = 0; c < qb.n_chunks; ++c) {
      const size_t part = ((size_t)(qb.part_base + c) * a.KV + j) * a.nq_max + i;
      M = fmaxf(M, __ldcg(a.part_ml + part * 2));
    }
    float L = 0.f, o = 0.f;
    for (int c = 0; c < qb.n_chunks; ++c) {
      const size_t part = ((size_t)(qb.part_base + c) * a.KV + j) * a.nq_max + i;
      const float m = __ldcg(a.part_ml + part * 2);
      if (m == -CUDART_INF_F) continue;
      const float f = expf(m - M);
      L = fmaf(__ldcg(a.part_ml + part * 2 + 1), f, L);
      o = fmaf(__ldcg(a.part_o + part * D + d), f, o);
    }
    const int row = qb.row0 + i / G, head = j * G + i % G;
    static_cast<Dt*>(a.out)[((size_t)row * a.H + head) * D + d] = from_f<Dt>(o / L);
  }
}

// Publish this item's partial; if it is the last of its group, merge.
template <typename Dt, int D>
__device__ void finish_item(const AttnArgs& a, const AttnQBlock& qb, int qbi, int j, int* flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(a.counters + (size_t)qbi * a.KV + j, 1);
    *flag = (prev == qb.n_chunks - 1);
  }
  __syncthreads();
  if (*flag) {
    __threadfence();
    combine<Dt, D>(a, qb, j);
    if (threadIdx.x == 0) a.counters[(size_t)qbi * a.KV + j] = 0;
  }
  __syncthreads();
}

// Prefill: 32 query vectors per item, 64-key chunks staged in shared memory;
// each thread computes a 4 x 4 score tile and a 4 x 8 output tile.
template <typename Dt, int D>
__global__ void __launch_bounds__(PRE_THREADS) attn_prefill_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float* Qt = sm;                        // [D][PRE_NQ]
  float* Kt = Qt + D * PRE_NQ;           // [D][PRE_CK]
  float* Vs = Kt + D * PRE_CK;           // [PRE_CK][D]
  float* Pt = Vs + PRE_CK * D;           // [PRE_CK][PRE_NQ]
  float* mls = Pt + PRE_CK * PRE_NQ;     // [PRE_NQ][2]
  __shared__ int flag;
  pdl_wait();
  pdl_launch();
  const int tid = threadIdx.x;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int n_items = *a.n_items;
  const int qg = tid >> 4, kg = tid & 15;  // 8 query groups x 16 key / dim groups
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const int nq = qb.nrows * G;
    const int key0 = item.chunk * PRE_CK;
    const int key1 = min(key0 + PRE_CK, qb.pos0 + qb.nrows);
    const int nk = key1 - key0;
    const size_t slab = (size_t)qb.seq * a.seq_stride + (size_t)j * a.capacity * D;
    const Dt* Kb = static_cast<const Dt*>(a.kc) + slab;
    const Dt* Vb = static_cast<const Dt*>(a.vc) + slab;
    for (int idx = tid; idx < PRE_NQ * D; idx += PRE_THREADS) {
      const int i = idx / D, d = idx % D;
      Qt[d * PRE_NQ + i] = i < nq ? to_f(static_cast<const Dt*>(a.q)[((size_t)(qb.row0 + i / G) * a.H + j * G + i % G) * D + d]) : 0.f;
    }
    for (int idx = tid; idx < PRE_CK * D; idx += PRE_THREADS) {
      const int u = idx / D, d = idx % D;
      const bool ok = u < nk;
      Kt[d * PRE_CK + u] = ok ? to_f(Kb[(size_t)(key0 + u) * D + d]) : 0.f;
      Vs[u * D + d] = ok ? to_f(Vb[(size_t)(key0 + u) * D + d]) : 0.f;
    }
    __syncthreads();
    float s[4][4] = {};
    for (int d = 0; d < D; ++d) {
      const float4 qv = *reinterpret_cast<const float4*>(Qt + d * PRE_NQ + qg * 4);
      const float4 kv = *reinterpret_cast<const float4*>(Kt + d * PRE_CK + kg * 4);
      const float qr[4] = {qv.x, qv.y, qv.z, qv.w}, kr[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) s[x][y] = fmaf(qr[x], kr[y], s[x][y]);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int i = qg * 4 + x;
      const int pos = qb.pos0 + i / G;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int u = kg * 4 + y;
        const bool vis = i < nq && u < nk && key0 + u <= pos;
        Pt[u * PRE_NQ + i] = vis ? s[x][y] * a.scale : -CUDART_INF_F;
      }
    }
    __syncthreads();
    // row statistics: 4 threads per query
    {
      const int i = tid >> 2, sub = tid & 3;
      float m = -CUDART_INF_F;
      for (int u = sub; u < PRE_CK; u += 4) m = fmaxf(m, Pt[u * PRE_NQ + i]);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      float l = 0.f;
      for (int u = sub; u < PRE_CK; u += 4) {
        const float v = Pt[u * PRE_NQ + i];
        const float p = (v == -CUDART_INF_F) ? 0.f : expf(v - m);
        Pt[u * PRE_NQ + i] = p;
        l += p;
      }
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (sub == 0) { mls[i * 2] = m; mls[i * 2 + 1] = l; }
    }
    __syncthreads();
    float o[4][8] = {};
    for (int u = 0; u < nk; ++u) {
      const float4 pv = *reinterpret_cast<const float4*>(Pt + u * PRE_NQ + qg * 4);
      const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
      const float4 v0 = *reinterpret_cast<const float4*>(Vs + u * D + kg * 8);
      const float4 v1 = *reinterpret_cast<const float4*>(Vs + u * D + kg * 8 + 4);
      const float vr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) o[x][y] = fmaf(pr[x], vr[y], o[x][y]);
    }
    const size_t part0 = ((size_t)(qb.part_base + item.chunk) * a.KV + j) * a.nq_max;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int i = qg * 4 + x;
      if (i >= nq) continue;
      if (kg * 8 < D) {
        float4* dst = reinterpret_cast<float4*>(a.part_o + (part0 + i) * D + kg * 8);
        dst[0] = make_float4(o[x][0], o[x][1], o[x][2], o[x][3]);
        dst[1] = make_float4(o[x][4], o[x][5], o[x][6], o[x][7]);
      }
    }
    if (tid < nq) {
      a.part_ml[(part0 + tid) * 2] = mls[tid * 2];
      a.part_ml[(part0 + tid) * 2 + 1] = mls[tid * 2 + 1];
    }
    finish_item<Dt, D>(a, qb, item.qb, j, &flag);
  }
}

template <int D> size_t prefill_smem() {
  return sizeof(float) * (D * PRE_NQ + D * PRE_CK + PRE_CK * D + PRE_CK * PRE_NQ + PRE_NQ * 2);
}

}  // namespace

int attn_prefill_chunk() { return PRE_CK; }
int attn_prefill_nq_max() { return PRE_NQ; }

template <typename Dt, int D>
static cudaError_t launch_pre(const LaunchCtx& c, const AttnArgs& a) {
  auto kern = attn_prefill_kernel<Dt, D>;
  cudaError_t e = set_max_smem((const void*)kern, (int)prefill_smem<D>());
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(a.grid_x, a.KV), dim3(PRE_THREADS), prefill_smem<D>(), c, a);
}

cudaError_t launch_attention_prefill(const LaunchCtx& c, int dt, const AttnArgs& a) {
  if (a.D == 128) return dt == DT_BF16 ? launch_pre<bf16, 128>(c, a) : launch_pre<float, 128>(c, a);
  if (a.D == 64) return dt == DT_BF16 ? launch_pre<bf16, 64>(c, a) : launch_pre<float, 64>(c, a);
  return cudaErrorInvalidValue;
}

}  // namespace q3
