// Decode-path kernels (T <= 4 rows per call) of the Qwen3 stack forward
// (maya2_mlx/backbone.py, Backbone.forward), built so that each step's HBM
// stream starts before the step it depends on has finished:
//
//  * gemv2: the linears.  Every warp owns a strided set of weight rows (gate
//    and up rows together for SiLU * up) and streams them through its own
//    ring of shared-memory slots filled by TMA bulk copies.  The first copies
//    are issued before griddepcontrol.wait, i.e. while the previous kernel is
//    still running under programmatic dependent launch.  The residual
//    epilogue (o_proj, down_proj) updates h in place and accumulates the sum
//    of squares of the new rows, so the following RMSNorm needs no reduction.
//  * attn_decode2: split-K attention over the static KV cache with the
//    per-head q/k RMSNorm, RoPE and the cache append fused in.  K/V chunks of
//    each work item stream into a shared-memory ring by TMA (again issued
//    before the wait); keys appended in this call are computed from the qkv
//    projection and written over their slots once the chunk has landed.
//  * norm_apply: the final RMSNorm from the precomputed sum of squares.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ============================================================ gemv2
constexpr int G2_WARPS = 8;
constexpr int G2_THREADS = G2_WARPS * 32;
constexpr int G2_UNROLL = 4;
constexpr size_t G2_SMEM_LIMIT = 220 * 1024;

struct G2Layout {
  size_t x_bytes, row_bytes, unit_bytes, ring_bytes, total;
};

__host__ __device__ inline G2Layout g2_layout(int wbytes, int T, int K, bool pair, int stages) {
  G2Layout L;
  L.x_bytes = align_up((size_t)T * K * 4, 128);
  L.row_bytes = (size_t)K * wbytes;
  L.unit_bytes = align_up((pair ? 2 : 1) * L.row_bytes, 128);
  L.ring_bytes = (size_t)G2_WARPS * stages * L.unit_bytes;
  L.total = L.x_bytes + L.ring_bytes + (size_t)G2_WARPS * stages * 8 + G2_WARPS * 4 * 8;
  return L;
}

template <typename Dt, int WF> struct G2W;
template <typename Dt> struct G2W<Dt, W_DT> {
  static constexpr int EPV = Vec16<Dt>::N;
  static constexpr int BYTES = sizeof(Dt);
  __device__ static __forceinline__ void get(const uint4& r, float* w, const Gemv2Args&, size_t, int) {
    Vec16<Dt>::unpack(r, w);
  }
};
template <typename Dt> struct G2W<Dt, W_U8> {
  static constexpr int EPV = 16;
  static constexpr int BYTES = 1;
  __device__ static __forceinline__ void get(const uint4& r, float* w, const Gemv2Args& a, size_t row, int k0) {
    const size_t gi = row * (size_t)(a.K / a.group) + k0 / a.group;
    const float s = __bfloat162float(static_cast<const bf16*>(a.scale)[gi]);
    const float b = __bfloat162float(static_cast<const bf16*>(a.bias)[gi]);
    const uint32_t v[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[4 * i + j] = fmaf(s, (float)((v[i] >> (8 * j)) & 0xffu), b);
  }
};

template <typename Dt>
__device__ void g2_stage_x(const Gemv2Args& a, float* xs, double* red) {
  const int K = a.K;
  for (int t = 0; t < a.T; ++t) {
    float* xt = xs + (size_t)t * K;
    if (a.prologue == PRO_X) {
      const Dt* x = static_cast<const Dt*>(a.x) + (size_t)t * K;
      for (int k = threadIdx.x; k < K; k += blockDim.x) xt[k] = to_f(x[k]);
    } else if (a.prologue == PRO_SUMSQ) {
      const double rs = rms_scale(a.sumsq_in[t], K, a.eps);
      const Dt* h = static_cast<const Dt*>(a.h) + (size_t)t * K;
      const Dt* g = static_cast<const Dt*>(a.gain);
      for (int k = threadIdx.x; k < K; k += blockDim.x) xt[k] = rms_apply<Dt>(to_f(h[k]), rs, to_f(g[k]));
    } else {  // PRO_FULL
      const Dt* x = static_cast<const Dt*>(a.x) + (size_t)t * K;
      const Dt* pe = a.pend ? static_cast<const Dt*>(a.pend) + (size_t)t * K : nullptr;
      Dt* ho = blockIdx.x == 0 ? static_cast<Dt*>(a.h) + (size_t)t * K : nullptr;
      double ss = 0.0;
      for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float v = to_f(x[k]);
        if (pe) v = rd<Dt>(v + to_f(pe[k]));
        if (ho) ho[k] = from_f<Dt>(v);
        xt[k] = v;
        ss = fma((double)v, (double)v, ss);
      }
      ss = block_sum_d(ss, red);
      const double rs = rms_scale(ss, K, a.eps);
      const Dt* g = static_cast<const Dt*>(a.gain);
      for (int k = threadIdx.x; k < K; k += blockDim.x) xt[k] = rms_apply<Dt>(xt[k], rs, to_f(g[k]));
    }
  }
  if (a.prologue == PRO_FULL && blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.sumsq_zero_n; i += blockDim.x) a.sumsq_zero[i] = 0.0;
}

template <typename Dt, int WF, int NT, int EPI>
__global__ void __launch_bounds__(G2_THREADS, 1) gemv2_kernel(Gemv2Args a) {
  extern __shared__ __align__(128) uint8_t g2_smem[];
  using W = G2W<Dt, WF>;
  constexpr bool PAIR = (EPI == EPI_SWIGLU);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  const G2Layout L = g2_layout(W::BYTES, NT, a.K, PAIR, S);
  float* xs = reinterpret_cast<float*>(g2_smem);
  uint8_t* ring = g2_smem + L.x_bytes + (size_t)warp * S * L.unit_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(g2_smem + L.x_bytes + L.ring_bytes) + warp * S;
  double* red = reinterpret_cast<double*>(g2_smem + L.x_bytes + L.ring_bytes + (size_t)G2_WARPS * S * 8);
  __shared__ double red_norm[32];

  const int gw = blockIdx.x * G2_WARPS + warp, nw = gridDim.x * G2_WARPS;
  const char* wb = static_cast<const char*>(a.w);
  const uint32_t unit_tx = (uint32_t)((PAIR ? 2 : 1) * L.row_bytes);

  auto issue = [&](int u, int s) {
    uint8_t* dst = ring + (size_t)s * L.unit_bytes;
    mbar_expect_tx(&bars[s], unit_tx);
    tma_load_1d(dst, wb + (size_t)u * L.row_bytes, (uint32_t)L.row_bytes, &bars[s]);
    if (PAIR) tma_load_1d(dst + L.row_bytes, wb + (size_t)(u + a.N) * L.row_bytes, (uint32_t)L.row_bytes, &bars[s]);
  };

  // Weights do not depend on the previous kernel: start streaming them now.
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
    for (int s = 0; s < S; ++s) {
      const int u = gw + s * nw;
      if (u < a.N) issue(u, s);
    }
  }
  __syncwarp();
  pdl_wait();
  pdl_launch();
  g2_stage_x<Dt>(a, xs, red_norm);
  __syncthreads();

  const int nvec = a.K / W::EPV;
  double ssq = 0.0;  // lane t: squares of updated rows of x-row t (residual epilogue)
  bool ok = true;
  int k = 0;
  for (;; ++k) {
    const int u = gw + k * nw;
    if (u >= a.N) break;
    const int s = k % S;
    if (!mbar_wait(&bars[s], (uint32_t)((k / S) & 1), a.err, 1)) { ok = false; break; }
    const uint8_t* slot = ring + (size_t)s * L.unit_bytes;
    float acc[NT], acc2[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = acc2[t] = 0.f;
    for (int v0 = lane; v0 < nvec; v0 += 32 * G2_UNROLL) {
      uint4 q0[G2_UNROLL], q1[G2_UNROLL];
#pragma unroll
      for (int i = 0; i < G2_UNROLL; ++i) {
        const int v = v0 + 32 * i;
        if (v < nvec) {
          q0[i] = *reinterpret_cast<const uint4*>(slot + (size_t)v * 16);
          if (PAIR) q1[i] = *reinterpret_cast<const uint4*>(slot + L.row_bytes + (size_t)v * 16);
        }
      }
#pragma unroll
      for (int i = 0; i < G2_UNROLL; ++i) {
        const int v = v0 + 32 * i;
        if (v >= nvec) break;
        const int k0 = v * W::EPV;
        float w0[W::EPV];
        W::get(q0[i], w0, a, (size_t)u, k0);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float* xp = xs + (size_t)t * a.K + k0;
#pragma unroll
          for (int e = 0; e < W::EPV; ++e) acc[t] = fmaf(w0[e], xp[e], acc[t]);
        }
        if (PAIR) {
          float w1[W::EPV];
          W::get(q1[i], w1, a, (size_t)u + a.N, k0);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float* xp = xs + (size_t)t * a.K + k0;
#pragma unroll
            for (int e = 0; e < W::EPV; ++e) acc2[t] = fmaf(w1[e], xp[e], acc2[t]);
          }
        }
      }
    }
    // the slot is free once every lane has read it: refill it
    __syncwarp();
    if (lane == 0) {
      const int un = u + S * nw;
      if (un < a.N) {
        fence_proxy_async();
        issue(un, s);
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[t] = warp_sum(acc[t]);
      if (PAIR) acc2[t] = warp_sum(acc2[t]);
    }
    if (lane < NT) {
      float v = acc[0], v2 = acc2[0];
#pragma unroll
      for (int t = 1; t < NT; ++t)
        if (lane == t) { v = acc[t]; v2 = acc2[t]; }
      const size_t o = (size_t)lane * a.ldo + u;
      if (EPI == EPI_STORE) {
        static_cast<Dt*>(a.out)[o] = from_f<Dt>(v);
      } else if (EPI == EPI_STORE_F32) {
        static_cast<float*>(a.out)[o] = v;
      } else if (EPI == EPI_RESIDUAL) {
        Dt* p = static_cast<Dt*>(a.out) + o;
        const float hn = rd<Dt>(to_f(*p) + rd<Dt>(v));
        *p = from_f<Dt>(hn);
        ssq = fma((double)hn, (double)hn, ssq);
      } else {  // SwiGLU: act = R(silu(R(g))) in fp32, out = R(act * R(u))
        const float g = rd<Dt>(v), up = rd<Dt>(v2);
        static_cast<Dt*>(a.out)[o] = from_f<Dt>(rd<Dt>(silu_f(g)) * up);
      }
    }
  }
  if (!ok && lane == 0) {
    // give the copies still in flight for this warp a bounded chance to land
    for (int j = k + 1; j < k + S; ++j)
      if (gw + j * nw < a.N) mbar_wait(&bars[j % S], (uint32_t)((j / S) & 1), a.err, 1);
  }
  if (EPI == EPI_RESIDUAL) {
    if (lane < NT) red[warp * 4 + lane] = ssq;
    __syncthreads();
    if (threadIdx.x < NT) {
      double s = 0.0;
      for (int w = 0; w < G2_WARPS; ++w) s += red[w * 4 + threadIdx.x];
      atomicAdd(a.sumsq_out + threadIdx.x, s);
    }
  }
}

template <typename Dt, int WF, int NT, int EPI>
cudaError_t g2_launch(const LaunchCtx& c, const Gemv2Args& a) {
  auto kern = gemv2_kernel<Dt, WF, NT, EPI>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G2_SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const G2Layout L = g2_layout(WF == W_U8 ? 1 : (int)sizeof(Dt), NT, a.K, EPI == EPI_SWIGLU, a.stages);
  int grid = (a.N + G2_WARPS - 1) / G2_WARPS;
  if (grid > c.num_sms) grid = c.num_sms;
  return launch_k(kern, dim3(grid), dim3(G2_THREADS), L.total, c, a);
}

template <typename Dt, int WF, int EPI>
cudaError_t g2_nt(const LaunchCtx& c, const Gemv2Args& a) {
  switch (a.T) {
    case 1: return g2_launch<Dt, WF, 1, EPI>(c, a);
    case 2: return g2_launch<Dt, WF, 2, EPI>(c, a);
    case 3: return g2_launch<Dt, WF, 3, EPI>(c, a);
    case 4: return g2_launch<Dt, WF, 4, EPI>(c, a);
  }
  return cudaErrorInvalidValue;
}

template <typename Dt, int WF>
cudaError_t g2_epi(const LaunchCtx& c, const Gemv2Args& a) {
  switch (a.epilogue) {
    case EPI_STORE: return g2_nt<Dt, WF, EPI_STORE>(c, a);
    case EPI_STORE_F32: return g2_nt<Dt, WF, EPI_STORE_F32>(c, a);
    case EPI_RESIDUAL: return g2_nt<Dt, WF, EPI_RESIDUAL>(c, a);
    case EPI_SWIGLU: return g2_nt<Dt, WF, EPI_SWIGLU>(c, a);
  }
  return cudaErrorInvalidValue;
}

// ============================================================ attn_decode2
constexpr int AD_THREADS = 128;
constexpr int AD_WARPS = AD_THREADS / 32;
constexpr int AD_NQ = 16;
constexpr int AD_STAGES = 3;

template <typename Dt> struct ADT {
  static constexpr int CK = sizeof(Dt) == 2 ? 64 : 32;  // keys per chunk: 16 KB per K or V tile at D = 128
};

template <typename Dt, int D> struct ADLayout {
  static constexpr size_t TILE = (size_t)ADT<Dt>::CK * D * sizeof(Dt);
  static constexpr size_t STAGE = 2 * TILE;
  static constexpr size_t QS = (size_t)AD_NQ * D * 4;
  static constexpr size_t SC = (size_t)AD_NQ * ADT<Dt>::CK * 4;
  static constexpr size_t OFF_QS = AD_STAGES * STAGE;
  static constexpr size_t OFF_SC = OFF_QS + QS;
  static constexpr size_t OFF_ML = OFF_SC + SC;
  static constexpr size_t OFF_CM = OFF_ML + AD_NQ * 2 * 4;  // combine: per-query max and sum
  static constexpr size_t OFF_BAR = OFF_CM + AD_NQ * 2 * 4;
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

template <typename Dt, int D>
__global__ void __launch_bounds__(AD_THREADS) attn_decode2_kernel(AttnDecArgs a) {
  extern __shared__ __align__(128) uint8_t ad_smem[];
  using LY = ADLayout<Dt, D>;
  constexpr int CK = ADT<Dt>::CK;
  constexpr int EPV = 16 / sizeof(Dt);  // elements per 16-byte vector
  constexpr int LPK = D / EPV;          // lanes per key in the score loop
  constexpr int KPW = 32 / LPK;         // keys per warp step
  constexpr int DPL = D / 32;           // head elements per lane
  float* qs = reinterpret_cast<float*>(ad_smem + LY::OFF_QS);
  float* sc = reinterpret_cast<float*>(ad_smem + LY::OFF_SC);
  float* ml = reinterpret_cast<float*>(ad_smem + LY::OFF_ML);
  float* cm = reinterpret_cast<float*>(ad_smem + LY::OFF_CM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ad_smem + LY::OFF_BAR);
  __shared__ int s_flag, s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int qkv_ld = (a.H + 2 * a.KV) * D;
  const int n_items = *a.n_items;
  const Dt* qkv = static_cast<const Dt*>(a.qkv);
  const Dt* kc = static_cast<const Dt*>(a.kc);
  const Dt* vc = static_cast<const Dt*>(a.vc);

  auto tiles = [&](int s) { return ad_smem + (size_t)s * LY::STAGE; };
  auto issue = [&](int it, int s) {
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const int key0 = item.chunk * CK;
    const int nk = min(CK, qb.pos0 + qb.nrows - key0);
    const size_t off = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + key0) * D;
    const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
    mbar_expect_tx(&bars[s], 2 * bytes);
    tma_load_1d(tiles(s), kc + off, bytes, &bars[s]);
    tma_load_1d(tiles(s) + LY::TILE, vc + off, bytes, &bars[s]);
  };

  // The cached keys do not depend on the previous kernel: start the copies.
  if (tid == 0) {
    for (int s = 0; s < AD_STAGES; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
    for (int s = 0; s < AD_STAGES; ++s) {
      const int it = blockIdx.x + s * gridDim.x;
      if (it < n_items) issue(it, s);
    }
    s_fail = 0;
  }
  __syncthreads();
  pdl_wait();
  pdl_launch();

  for (int k = 0;; ++k) {
    const int it = blockIdx.x + k * gridDim.x;
    if (it >= n_items) break;
    const int s = k % AD_STAGES;
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const int nq = qb.nrows * G;
    const int key0 = item.chunk * CK;
    const int key1 = min(key0 + CK, qb.pos0 + qb.nrows);
    const int nk = key1 - key0;
    Dt* Kt = reinterpret_cast<Dt*>(tiles(s));
    Dt* Vt = reinterpret_cast<Dt*>(tiles(s) + LY::TILE);

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
    const bool landed = mbar_wait(&bars[s], (uint32_t)((k / AD_STAGES) & 1), a.err, 2);
    if (__syncthreads_or(!landed)) break;
    // keys appended by this call that fall in the chunk: computed here
    const int n0 = max(key0, qb.seg_pos0), n1 = min(key1, qb.seg_pos0 + qb.seg_n);
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
      const int sub = lane % LPK;
      for (int ub = warp * KPW; ub < nk; ub += AD_WARPS * KPW) {
        const int u = ub + lane / LPK;
        float kv[EPV];
        if (u < nk) Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(Kt + (size_t)u * D + sub * EPV), kv);
        else
#pragma unroll
          for (int e = 0; e < EPV; ++e) kv[e] = 0.f;
        for (int i = 0; i < nq; ++i) {
          const float* qp = qs + i * D + sub * EPV;
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) d = fmaf(qp[e], kv[e], d);
#pragma unroll
          for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          if (sub == 0 && u < nk)
            sc[i * CK + u] = (key0 + u <= qb.pos0 + i / G) ? d * a.scale : -CUDART_INF_F;
        }
      }
    }
    __syncthreads();
    for (int i = warp; i < nq; i += AD_WARPS) {
      float m = -CUDART_INF_F;
      for (int u = lane; u < nk; u += 32) m = fmaxf(m, sc[i * CK + u]);
      m = warp_max(m);
      float l = 0.f;
      for (int u = lane; u < nk; u += 32) {
        const float x = sc[i * CK + u];
        const float p = (x == -CUDART_INF_F) ? 0.f : expf(x - m);
        sc[i * CK + u] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) { ml[i * 2] = m; ml[i * 2 + 1] = l; }
    }
    __syncthreads();
    const size_t part0 = ((size_t)(qb.part_base + item.chunk) * a.KV + j) * a.nq_max;
    if (tid < D) {
      float o[AD_NQ];
#pragma unroll
      for (int i = 0; i < AD_NQ; ++i) o[i] = 0.f;
      for (int u = 0; u < nk; ++u) {
        const float v = to_f(Vt[(size_t)u * D + tid]);
#pragma unroll
        for (int i = 0; i < AD_NQ; ++i)
          if (i < nq) o[i] = fmaf(sc[i * CK + u], v, o[i]);
      }
#pragma unroll
      for (int i = 0; i < AD_NQ; ++i)
        if (i < nq) a.part_o[(part0 + i) * D + tid] = o[i];
    }
    if (tid < nq) {
      a.part_ml[(part0 + tid) * 2] = ml[tid * 2];
      a.part_ml[(part0 + tid) * 2 + 1] = ml[tid * 2 + 1];
    }
    // publish; the last item of (query block, kv head) merges all chunks
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
      const size_t pbase = (size_t)qb.part_base * a.KV + j;  // part of chunk c: (pbase + c * KV) * nq_max
      // per-query max and normaliser
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
        if (lane == 0) { cm[i * 2] = M; cm[i * 2 + 1] = Lsum; }
      }
      __syncthreads();
      // chunk sums: warp w takes chunks w, w+4, ...; per-warp results in the
      // finished stage's tiles, then a fixed-order sum over warps
      float* red = reinterpret_cast<float*>(tiles(s));
      for (int i = 0; i < nq; ++i) {
        float o[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] = 0.f;
        const float M = cm[i * 2];
        for (int c = warp; c < nc; c += AD_WARPS) {
          const size_t p = (pbase + (size_t)c * a.KV) * a.nq_max + i;
          const float m = __ldcg(a.part_ml + p * 2);
          const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[e] = fmaf(__ldcg(a.part_o + p * D + lane * DPL + e), f, o[e]);
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) red[(warp * AD_NQ + i) * D + lane * DPL + e] = o[e];
      }
      __syncthreads();
      for (int idx = tid; idx < nq * D; idx += AD_THREADS) {
        const int i = idx / D, d = idx % D;
        float o = 0.f;
        for (int w = 0; w < AD_WARPS; ++w) o += red[(w * AD_NQ + i) * D + d];
        const int row = qb.row0 + i / G, head = j * G + i % G;
        static_cast<Dt*>(a.out)[((size_t)row * a.H + head) * D + d] = from_f<Dt>(o / cm[i * 2 + 1]);
      }
      if (tid == 0) a.counters[(size_t)item.qb * a.KV + j] = 0;
    }
    // release the stage and refill it with this block's item k + STAGES
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      const int nit = blockIdx.x + (k + AD_STAGES) * gridDim.x;
      if (nit < n_items) issue(nit, s);
    }
  }
}

template <typename Dt, int D>
cudaError_t ad_launch(const LaunchCtx& c, const AttnDecArgs& a) {
  auto kern = attn_decode2_kernel<Dt, D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ADLayout<Dt, D>::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_k(kern, dim3(a.grid_x, a.KV), dim3(AD_THREADS), ADLayout<Dt, D>::TOTAL, c, a);
}

// ============================================================ norm_apply
template <typename Dt>
__global__ void __launch_bounds__(256) norm_apply_kernel(NormApplyArgs a) {
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  const double rs = rms_scale(a.sumsq[t], a.hidden, a.eps);
  const Dt* h = static_cast<const Dt*>(a.h) + (size_t)t * a.hidden;
  const Dt* g = static_cast<const Dt*>(a.gain);
  Dt* out = static_cast<Dt*>(a.out) + (size_t)t * a.hidden;
  for (int k = threadIdx.x; k < a.hidden; k += blockDim.x) out[k] = from_f<Dt>(rms_apply<Dt>(to_f(h[k]), rs, to_f(g[k])));
}

}  // namespace

int gemv2_plan(int dt, int wfmt, int T, int K, int group, bool pair, size_t* smem) {
  (void)group;
  const int wbytes = wfmt == W_U8 ? 1 : (dt == DT_BF16 ? 2 : 4);
  for (int s = 4; s >= 1; --s) {
    const G2Layout L = g2_layout(wbytes, T, K, pair, s);
    if (L.total <= G2_SMEM_LIMIT) {
      if (smem) *smem = L.total;
      return s;
    }
  }
  return 0;
}

cudaError_t launch_gemv2(const LaunchCtx& c, int dt, int wfmt, const Gemv2Args& a) {
  if (a.T < 1 || a.T > 4 || a.stages < 1) return cudaErrorInvalidValue;
  if (dt == DT_BF16) return wfmt == W_U8 ? g2_epi<bf16, W_U8>(c, a) : g2_epi<bf16, W_DT>(c, a);
  return wfmt == W_U8 ? g2_epi<float, W_U8>(c, a) : g2_epi<float, W_DT>(c, a);
}

int attn_decode2_chunk(int dt) { return dt == DT_BF16 ? ADT<bf16>::CK : ADT<float>::CK; }
int attn_decode2_nq_max() { return AD_NQ; }

cudaError_t launch_attn_decode2(const LaunchCtx& c, int dt, const AttnDecArgs& a) {
  if (a.D == 128) return dt == DT_BF16 ? ad_launch<bf16, 128>(c, a) : ad_launch<float, 128>(c, a);
  if (a.D == 64) return dt == DT_BF16 ? ad_launch<bf16, 64>(c, a) : ad_launch<float, 64>(c, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_norm_apply(const LaunchCtx& c, int dt, const NormApplyArgs& a) {
  if (dt == DT_BF16) return launch_k(norm_apply_kernel<bf16>, dim3(a.T), dim3(256), 0, c, a);
  return launch_k(norm_apply_kernel<float>, dim3(a.T), dim3(256), 0, c, a);
}

}  // namespace q3
