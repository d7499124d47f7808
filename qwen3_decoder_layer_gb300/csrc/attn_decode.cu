// Decode attention over the static KV cache with the per-head q/k RMSNorm,
// RoPE and cache append fused in (maya2_mlx/backbone.py, Backbone.forward:
// "q, k = per-head RMSNorm (two roundings), RoPE in fp32 on the cos/sin
// table, attention over keys 0..pos (fp32 softmax, one rounding)"; GQA as the
// repeat_kv of rlx_flow/blocks/qwen3_decoder.rs).
//
// Split-K ("flash-decoding"): the keys of each query block (rows of one
// sequence, x G query heads of kv head j) are cut into chunks of SUBS
// sub-chunks of CK keys.  A work item is one (query block, chunk, kv head);
// a persistent grid walks the item list.  Each block streams the sub-chunks
// of its items, in order, through a 3-stage shared-memory ring filled by TMA
// bulk copies (the first ones issued before griddepcontrol.wait, so the KV
// stream overlaps the qkv projection), and keeps an online softmax (running
// max m, sum l, output o) over an item's sub-chunks.  Keys appended in this
// call are computed from the qkv row (RMSNorm + RoPE) and written over their
// slots once the sub-chunk has landed; the item that owns the row also stores
// them to the cache.  Each item stores its partial (m, l, o); the last item
// of a (query block, kv head) -- found with an atomic counter, no waiting --
// merges them: M = max m_c, out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
// rounded once to the model dtype.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int AD_THREADS = 128;
constexpr int AD_WARPS = AD_THREADS / 32;
constexpr int AD_NQ = 16;
constexpr int AD_STAGES = 3;
constexpr int AD_SUBS = 4;  // sub-chunks per item

template <typename Dt> struct ADT {
  static constexpr int CK = sizeof(Dt) == 2 ? 64 : 32;  // 16 KB per K or V sub-chunk at head_dim 128
};

template <typename Dt, int D> struct ADLayout {
  static constexpr size_t TILE = (size_t)ADT<Dt>::CK * D * sizeof(Dt);
  static constexpr size_t STAGE = 2 * TILE;
  static constexpr size_t OFF_QS = AD_STAGES * STAGE;                  // [NQ][D] fp32 queries
  static constexpr size_t OFF_SC = OFF_QS + (size_t)AD_NQ * D * 4;     // [NQ][CK] scores / p
  static constexpr size_t OFF_RUN = OFF_SC + (size_t)AD_NQ * ADT<Dt>::CK * 4;  // [NQ] m, l, alpha
  static constexpr size_t OFF_RED = OFF_RUN + (size_t)AD_NQ * 4 * 4;  // merge: [WARPS][NQ][D] fp32
  static constexpr size_t OFF_BAR = OFF_RED + (size_t)AD_WARPS * AD_NQ * D * 4;
  static constexpr size_t TOTAL = OFF_BAR + AD_STAGES * 8 + 16;
};

// Per-head RMSNorm + RoPE of one raw q or k head (warp-wide: lane holds
// elements lane*DPL .. +DPL) at position pos, rounded to the model dtype.
template <typename Dt, int D>
__device__ __forceinline__ void norm_rope_head(float* x, const Dt* gain, const float* cos_t, const float* sin_t,
                                               int pos, float eps) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  double ss = 0.0;
#pragma unroll
  for (int e = 0; e < DPL; ++e) ss = fma((double)x[e], (double)x[e], ss);
  ss = warp_sum_d(ss);
  const double rs = rms_scale(ss, D, eps);
#pragma unroll
  for (int e = 0; e < DPL; ++e) x[e] = rms_apply<Dt>(x[e], rs, to_f(gain[lane * DPL + e]));
  const float* cs = cos_t + (size_t)pos * D + lane * DPL;
  const float* sn = sin_t + (size_t)pos * D + lane * DPL;
  const bool first = lane < 16;
  float o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
    const double xc = (double)x[e] * (double)cs[e], ps = (double)partner * (double)sn[e];
    o[e] = rd_d<Dt>(first ? xc - ps : xc + ps);
  }
#pragma unroll
  for (int e = 0; e < DPL; ++e) x[e] = o[e];
}

// Keys of item `it`: [key0, key0 + nkeys).
struct ItemKeys {
  int key0, nkeys, nsub;
};
template <typename Dt>
__device__ __forceinline__ ItemKeys item_keys(const AttnDecArgs& a, int it) {
  constexpr int CK = ADT<Dt>::CK;
  const AttnItem item = a.items[it];
  const AttnQBlock qb = a.qblocks[item.qb];
  ItemKeys r;
  r.key0 = item.chunk * CK * AD_SUBS;
  r.nkeys = min(CK * AD_SUBS, qb.pos0 + qb.nrows - r.key0);
  r.nsub = (r.nkeys + CK - 1) / CK;
  return r;
}

template <typename Dt, int D>
__global__ void __launch_bounds__(AD_THREADS) attn_decode_kernel(AttnDecArgs a) {
  extern __shared__ __align__(128) uint8_t ad_smem[];
  using LY = ADLayout<Dt, D>;
  constexpr int CK = ADT<Dt>::CK;
  constexpr int EPV = 16 / sizeof(Dt);  // elements per 16-byte vector
  constexpr int LPK = D / EPV;          // lanes per key in the score loop
  constexpr int KPW = 32 / LPK;         // keys per warp step
  constexpr int DPL = D / 32;           // head elements per lane
  float* qs = reinterpret_cast<float*>(ad_smem + LY::OFF_QS);
  float* sc = reinterpret_cast<float*>(ad_smem + LY::OFF_SC);
  float* run = reinterpret_cast<float*>(ad_smem + LY::OFF_RUN);  // [i*4]: m, l, alpha
  float* red = reinterpret_cast<float*>(ad_smem + LY::OFF_RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ad_smem + LY::OFF_BAR);
  __shared__ int s_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int qkv_ld = (a.H + 2 * a.KV) * D;
  const int n_items = *a.n_items;
  const Dt* qkv = static_cast<const Dt*>(a.qkv);
  const Dt* kc = static_cast<const Dt*>(a.kc);
  const Dt* vc = static_cast<const Dt*>(a.vc);
  auto tiles = [&](int s) { return ad_smem + (size_t)s * LY::STAGE; };

  // Producer cursor (thread 0 only): next (local item, sub-chunk) to load.
  int p_k = 0, p_sub = 0, p_g = 0;
  auto produce = [&]() {  // issue the next sub-chunk of this block's item sequence, if any
    while (true) {
      const int it = blockIdx.x + p_k * gridDim.x;
      if (it >= n_items) return;
      const ItemKeys ik = item_keys<Dt>(a, it);
      if (p_sub >= ik.nsub) { ++p_k; p_sub = 0; continue; }
      const AttnQBlock qb = a.qblocks[a.items[it].qb];
      const int k0 = ik.key0 + p_sub * CK;
      const int nk = min(CK, ik.key0 + ik.nkeys - k0);
      const size_t off = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + k0) * D;
      const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
      const int s = p_g % AD_STAGES;
      mbar_expect_tx(&bars[s], 2 * bytes);
      tma_load_1d(tiles(s), kc + off, bytes, &bars[s]);
      tma_load_1d(tiles(s) + LY::TILE, vc + off, bytes, &bars[s]);
      ++p_sub;
      ++p_g;
      return;
    }
  };

  // The cached keys do not depend on the previous kernel: start the copies.
  if (tid == 0) {
    for (int s = 0; s < AD_STAGES; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
    for (int s = 0; s < AD_STAGES; ++s) produce();
  }
  // ... and ask L2 for the next kernel's operand (its share of it).
  if (tid == 32 && a.pf && a.pf_bytes) {
    const int nb = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
    const size_t per = ((a.pf_bytes + nb - 1) / nb + 15) & ~size_t(15);
    for (size_t b0 = per * b, b1 = min(per * (b + 1), a.pf_bytes); b0 < b1; b0 += 65536)
      prefetch_l2(static_cast<const char*>(a.pf) + b0, (uint32_t)min(b1 - b0, (size_t)65536));
  }
  __syncthreads();
  pdl_wait();
  pdl_launch();

  int g = 0;  // consumer position in the block's sub-chunk sequence
  bool failed = false;
  for (int k = 0; !failed; ++k) {
    const int it = blockIdx.x + k * gridDim.x;
    if (it >= n_items) break;
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const ItemKeys ik = item_keys<Dt>(a, it);
    const int nq = qb.nrows * G;

    // queries: RMSNorm + RoPE of this block's q heads of kv group j
    for (int i = warp; i < nq; i += AD_WARPS) {
      const int row = qb.row0 + i / G, hh = j * G + i % G;
      float x[DPL];
      const Dt* src = qkv + (size_t)row * qkv_ld + (size_t)hh * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) x[e] = to_f(src[e]);
      norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.q_gain), a.cos_t, a.sin_t, qb.pos0 + i / G, a.eps);
#pragma unroll
      for (int e = 0; e < DPL; ++e) qs[i * D + lane * DPL + e] = x[e];
    }
    if (tid < nq) {
      run[tid * 4] = -CUDART_INF_F;
      run[tid * 4 + 1] = 0.f;
    }
    float o[AD_NQ];
#pragma unroll
    for (int i = 0; i < AD_NQ; ++i) o[i] = 0.f;

    for (int sub = 0; sub < ik.nsub; ++sub, ++g) {
      const int s = g % AD_STAGES;
      const int key0 = ik.key0 + sub * CK;
      const int nk = min(CK, ik.key0 + ik.nkeys - key0);
      Dt* Kt = reinterpret_cast<Dt*>(tiles(s));
      Dt* Vt = reinterpret_cast<Dt*>(tiles(s) + LY::TILE);
      const bool landed = mbar_wait(&bars[s], (uint32_t)((g / AD_STAGES) & 1), a.err, 2);
      if (__syncthreads_or(!landed)) { failed = true; break; }
      // keys appended by this call that fall in the sub-chunk: computed here
      const int n0 = max(key0, qb.seg_pos0), n1 = min(key0 + nk, qb.seg_pos0 + qb.seg_n);
      for (int u = n0 + warp; u < n1; u += AD_WARPS) {
        const int row = qb.seg_row0 + (u - qb.seg_pos0);
        float x[DPL], v[DPL];
        const Dt* ksrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + j) * D + lane * DPL;
        const Dt* vsrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + a.KV + j) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) { x[e] = to_f(ksrc[e]); v[e] = to_f(vsrc[e]); }
        norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.k_gain), a.cos_t, a.sin_t, u, a.eps);
        const bool owner = row >= qb.row0 && row < qb.row0 + qb.nrows;
        const size_t goff = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + u) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          Kt[(u - key0) * D + lane * DPL + e] = from_f<Dt>(x[e]);
          Vt[(u - key0) * D + lane * DPL + e] = from_f<Dt>(v[e]);
          if (owner) {
            static_cast<Dt*>(a.kc)[goff + e] = from_f<Dt>(x[e]);
            static_cast<Dt*>(a.vc)[goff + e] = from_f<Dt>(v[e]);
          }
        }
      }
      __syncthreads();
      // scores: LPK lanes per key, KPW keys per warp step
      {
        const int sub_l = lane % LPK;
        for (int ub = warp * KPW; ub < nk; ub += AD_WARPS * KPW) {
          const int u = ub + lane / LPK;
          float kv[EPV];
          if (u < nk) {
            Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(Kt + (size_t)u * D + sub_l * EPV), kv);
          } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) kv[e] = 0.f;
          }
          for (int i = 0; i < nq; ++i) {
            const float* qp = qs + i * D + sub_l * EPV;
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < EPV; ++e) d = fmaf(qp[e], kv[e], d);
#pragma unroll
            for (int off = LPK / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (sub_l == 0 && u < nk)
              sc[i * CK + u] = (key0 + u <= qb.pos0 + i / G) ? d * a.scale : -CUDART_INF_F;
          }
        }
      }
      __syncthreads();
      // online softmax update per query (warp per query)
      for (int i = warp; i < nq; i += AD_WARPS) {
        float mc = -CUDART_INF_F;
        for (int u = lane; u < nk; u += 32) mc = fmaxf(mc, sc[i * CK + u]);
        mc = warp_max(mc);
        const float m_old = run[i * 4];
        const float m_new = fmaxf(m_old, mc);
        float l = 0.f;
        for (int u = lane; u < nk; u += 32) {
          const float x = sc[i * CK + u];
          const float p = (x == -CUDART_INF_F) ? 0.f : expf(x - m_new);
          sc[i * CK + u] = p;
          l += p;
        }
        l = warp_sum(l);
        if (lane == 0) {
          const float alpha = (m_old == -CUDART_INF_F) ? 0.f : expf(m_old - m_new);
          run[i * 4] = m_new;
          run[i * 4 + 1] = run[i * 4 + 1] * alpha + l;
          run[i * 4 + 2] = alpha;
        }
      }
      __syncthreads();
      if (tid < D) {
#pragma unroll
        for (int i = 0; i < AD_NQ; ++i)
          if (i < nq) o[i] *= run[i * 4 + 2];
        int u = 0;
        for (; u + 4 <= nk; u += 4) {
          const float v0 = to_f(Vt[(size_t)u * D + tid]), v1 = to_f(Vt[(size_t)(u + 1) * D + tid]);
          const float v2 = to_f(Vt[(size_t)(u + 2) * D + tid]), v3 = to_f(Vt[(size_t)(u + 3) * D + tid]);
#pragma unroll
          for (int i = 0; i < AD_NQ; ++i)
            if (i < nq) {
              const float4 p = *reinterpret_cast<const float4*>(sc + i * CK + u);
              o[i] = fmaf(p.x, v0, fmaf(p.y, v1, fmaf(p.z, v2, fmaf(p.w, v3, o[i]))));
            }
        }
        for (; u < nk; ++u) {
          const float v = to_f(Vt[(size_t)u * D + tid]);
#pragma unroll
          for (int i = 0; i < AD_NQ; ++i)
            if (i < nq) o[i] = fmaf(sc[i * CK + u], v, o[i]);
        }
      }
      // release the stage; refill it with the next sub-chunk of the sequence
      fence_proxy_async();
      __syncthreads();
      if (tid == 0) produce();
    }
    if (failed) break;

    // partial of this item
    const size_t part0 = ((size_t)(qb.part_base + item.chunk) * a.KV + j) * a.nq_max;
    if (tid < D) {
#pragma unroll
      for (int i = 0; i < AD_NQ; ++i)
        if (i < nq) a.part_o[(part0 + i) * D + tid] = o[i];
    }
    if (tid < nq) {
      a.part_ml[(part0 + tid) * 2] = run[tid * 4];
      a.part_ml[(part0 + tid) * 2 + 1] = run[tid * 4 + 1];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int prev = atomicAdd(a.counters + (size_t)item.qb * a.KV + j, 1);
      s_flag = (prev == qb.n_chunks - 1);
    }
    __syncthreads();
    if (s_flag) {
      __threadfence();
      const int nc = qb.n_chunks;
      const size_t pbase = (size_t)qb.part_base * a.KV + j;  // partial of chunk c: (pbase + c * KV) * nq_max
      // per-query max and normaliser (warp per query, lanes over chunks)
      for (int i = warp; i < nq; i += AD_WARPS) {
        float M = -CUDART_INF_F;
        for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(a.part_ml + ((pbase + (size_t)c * a.KV) * a.nq_max + i) * 2));
        M = warp_max(M);
        float Lsum = 0.f;
        for (int c = lane; c < nc; c += 32) {
          const size_t p = ((pbase + (size_t)c * a.KV) * a.nq_max + i) * 2;
          const float m = __ldcg(a.part_ml + p);
          if (m != -CUDART_INF_F) Lsum = fmaf(__ldcg(a.part_ml + p + 1), expf(m - M), Lsum);
        }
        Lsum = warp_sum(Lsum);
        if (lane == 0) { run[i * 4] = M; run[i * 4 + 1] = Lsum; }
      }
      __syncthreads();
      // weighted chunk sums: warp w takes chunks w, w + 4, ...; fixed-order sum over warps
      for (int i = 0; i < nq; ++i) {
        float acc[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
        const float M = run[i * 4];
#pragma unroll 4
        for (int c = warp; c < nc; c += AD_WARPS) {
          const size_t p = (pbase + (size_t)c * a.KV) * a.nq_max + i;
          const float m = __ldcg(a.part_ml + p * 2);
          const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[e] = fmaf(__ldcg(a.part_o + p * D + lane * DPL + e), f, acc[e]);
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) red[(warp * AD_NQ + i) * D + lane * DPL + e] = acc[e];
      }
      __syncthreads();
      for (int idx = tid; idx < nq * D; idx += AD_THREADS) {
        const int i = idx / D, d = idx % D;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < AD_WARPS; ++w) v += red[(w * AD_NQ + i) * D + d];
        const int row = qb.row0 + i / G, head = j * G + i % G;
        static_cast<Dt*>(a.out)[((size_t)row * a.H + head) * D + d] = from_f<Dt>(v / run[i * 4 + 1]);
      }
      if (tid == 0) a.counters[(size_t)item.qb * a.KV + j] = 0;
      __syncthreads();
    }
  }
  if (failed && tid == 0) {
    // give the copies still in flight a bounded chance to land before exiting
    for (int q = g + 1; q < p_g; ++q) mbar_wait(&bars[q % AD_STAGES], (uint32_t)((q / AD_STAGES) & 1), a.err, 2);
  }
}

template <typename Dt, int D>
cudaError_t ad_launch(const LaunchCtx& c, const AttnDecArgs& a) {
  auto kern = attn_decode_kernel<Dt, D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ADLayout<Dt, D>::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_k(kern, dim3(a.grid_x, a.KV), dim3(AD_THREADS), ADLayout<Dt, D>::TOTAL, c, a);
}

}  // namespace

int attn_decode2_chunk(int dt) { return (dt == DT_BF16 ? ADT<bf16>::CK : ADT<float>::CK) * AD_SUBS; }
int attn_decode2_nq_max() { return AD_NQ; }

cudaError_t launch_attn_decode2(const LaunchCtx& c, int dt, const AttnDecArgs& a) {
  if (a.D == 128) return dt == DT_BF16 ? ad_launch<bf16, 128>(c, a) : ad_launch<float, 128>(c, a);
  if (a.D == 64) return dt == DT_BF16 ? ad_launch<bf16, 64>(c, a) : ad_launch<float, 64>(c, a);
  return cudaErrorInvalidValue;
}

}  // namespace q3
