// Decode-path linears (T <= 4 rows per call) of the Qwen3 stack forward
// (maya2_mlx/backbone.py, Backbone.forward: `Q.mm(y, L["qkv"])`,
// `Q.mm(a, L["o"])` with the residual add, `Q.mm(y2, L["gu"])` with the fp32
// SiLU * up, `Q.mm(act * u, L["down"])` with the residual add), and the final
// RMSNorm.
//
//  * gemv2: every warp owns a strided set of weight rows (gate and up rows
//    together for SiLU * up) and streams them through its own ring of
//    shared-memory slots filled by TMA bulk copies.  The first copies are
//    issued before griddepcontrol.wait, i.e. while the previous kernel is
//    still running under programmatic dependent launch, and one thread also
//    asks L2 for the next linear's weights.  The normalised input rows sit in
//    shared memory in the model dtype, so each lane reads its x vector as
//    contiguous 16-byte loads free of bank conflicts; each row's dot product
//    runs as independent accumulator chains (one per unrolled 16-byte vector).  The residual
//    epilogue (o_proj, down_proj) updates h in place and accumulates the sum
//    of squares of the new rows, so the following RMSNorm needs no reduction.
//  * norm_apply: the final RMSNorm from the precomputed sum of squares.
#include <math_constants.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int G2_MAX_WARPS = 16;
constexpr size_t G2_SMEM_LIMIT = 220 * 1024;
constexpr size_t G2_SMEM_CORES = 110 * 1024;  // two CTAs per SM

struct G2Layout {
  size_t x_bytes, row_bytes, unit_bytes, ring_bytes, total;
};

__host__ __device__ inline G2Layout g2_layout(int wbytes, int xbytes, int T, int K, bool pair, int stages,
                                              int nwarps) {
  G2Layout L;
  L.x_bytes = align_up((size_t)T * K * xbytes, 128);
  L.row_bytes = (size_t)K * wbytes;
  L.unit_bytes = align_up((pair ? 2 : 1) * L.row_bytes, 128);
  L.ring_bytes = (size_t)nwarps * stages * L.unit_bytes;
  L.total = L.x_bytes + L.ring_bytes + (size_t)nwarps * stages * 8 + G2_MAX_WARPS * 4 * 8;
  return L;
}

// Stage the T input rows in shared memory in the model dtype (16-byte vector
// loads), applying the prologue.  Every staged value is already a model-dtype
// value (x, R(x + pend), or the RMSNorm output), so nothing is lost.
template <typename Dt>
__device__ void g2_stage_x(const Gemv2Args& a, Dt* xs, float* red) {
  constexpr int V = Vec16<Dt>::N;
  constexpr int MAXC = 4;  // 16-byte chunks per thread kept in registers
  const int K = a.K;
  const int nch = a.T * K / V;
  __shared__ F2 s_rs[4];
  if (a.prologue == PRO_X) {
    const Dt* x = static_cast<const Dt*>(a.x);
    for (int c = threadIdx.x; c < nch; c += blockDim.x)
      *reinterpret_cast<uint4*>(xs + (size_t)c * V) = ld16(x + (size_t)c * V);
  } else if (a.prologue == PRO_SUMSQ && nch <= MAXC * (int)blockDim.x) {
    // h and the gain are fetched while one thread per row turns its double
    // sum of squares into the scale
    uint4 hv[MAXC], gv[MAXC];
    const Dt* h = static_cast<const Dt*>(a.h);
    const Dt* g = static_cast<const Dt*>(a.gain);
#pragma unroll
    for (int q = 0; q < MAXC; ++q) {
      const int c = threadIdx.x + q * blockDim.x;
      if (c < nch) {
        hv[q] = ld16(h + (size_t)c * V);
        gv[q] = ld16(g + (size_t)((c * V) % K));
      }
    }
    if (threadIdx.x < a.T) s_rs[threadIdx.x] = rms_scale2(f2_from_double(a.sumsq_in[threadIdx.x]), K, a.eps);
    __syncthreads();
#pragma unroll
    for (int q = 0; q < MAXC; ++q) {
      const int c = threadIdx.x + q * blockDim.x;
      if (c < nch) {
        const F2 rs = s_rs[c * V / K];
        float hf[V], gf[V], o[V];
        Vec16<Dt>::unpack(hv[q], hf);
        Vec16<Dt>::unpack(gv[q], gf);
        rms_apply2_v<Dt, V>(hf, rs, gf, o);
        const uint4 ov = Vec16<Dt>::pack(o);
        *reinterpret_cast<uint4*>(xs + (size_t)c * V) = ov;
        if (blockIdx.x == 0 && a.x_out) *reinterpret_cast<uint4*>(static_cast<Dt*>(a.x_out) + (size_t)c * V) = ov;
      }
    }
  } else if (a.prologue == PRO_SUMSQ) {
    if (threadIdx.x < a.T) s_rs[threadIdx.x] = rms_scale2(f2_from_double(a.sumsq_in[threadIdx.x]), K, a.eps);
    __syncthreads();
    const Dt* h = static_cast<const Dt*>(a.h);
    const Dt* g = static_cast<const Dt*>(a.gain);
    for (int c = threadIdx.x; c < nch; c += blockDim.x) {
      const F2 rs = s_rs[c * V / K];
      float hf[V], gf[V], o[V];
      Vec16<Dt>::unpack(ld16(h + (size_t)c * V), hf);
      Vec16<Dt>::unpack(ld16(g + (size_t)((c * V) % K)), gf);
      rms_apply2_v<Dt, V>(hf, rs, gf, o);
      const uint4 ov = Vec16<Dt>::pack(o);
      *reinterpret_cast<uint4*>(xs + (size_t)c * V) = ov;
      if (blockIdx.x == 0 && a.x_out) *reinterpret_cast<uint4*>(static_cast<Dt*>(a.x_out) + (size_t)c * V) = ov;
    }
  } else {  // PRO_FULL
    for (int t = 0; t < a.T; ++t) {
      Dt* xt = xs + (size_t)t * K;
      const Dt* x = static_cast<const Dt*>(a.x) + (size_t)t * K;
      const Dt* pe = a.pend ? static_cast<const Dt*>(a.pend) + (size_t)t * K : nullptr;
      Dt* ho = blockIdx.x == 0 ? static_cast<Dt*>(a.h) + (size_t)t * K : nullptr;
      F2 ss = {0.f, 0.f};
      for (int k = threadIdx.x * V; k < K; k += blockDim.x * V) {
        float v[V];
        Vec16<Dt>::unpack(ld16(x + k), v);
        if (pe) {
          float p[V];
          Vec16<Dt>::unpack(ld16(pe + k), p);
#pragma unroll
          for (int e = 0; e < V; ++e) v[e] = rd<Dt>(v[e] + p[e]);
        }
        const uint4 pv = Vec16<Dt>::pack(v);
        if (ho) *reinterpret_cast<uint4*>(ho + k) = pv;
        *reinterpret_cast<uint4*>(xt + k) = pv;
#pragma unroll
        for (int e = 0; e < V; ++e) f2_add_sq(ss, v[e]);
      }
      ss = f2_block_sum(ss, red);
      const F2 rs = rms_scale2(ss, K, a.eps);
      const Dt* g = static_cast<const Dt*>(a.gain);
      for (int k = threadIdx.x * V; k < K; k += blockDim.x * V) {
        float gv[V], hv[V], o[V];
        Vec16<Dt>::unpack(ld16(g + k), gv);
        Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(xt + k), hv);  // this thread's own stores
        rms_apply2_v<Dt, V>(hv, rs, gv, o);
        *reinterpret_cast<uint4*>(xt + k) = Vec16<Dt>::pack(o);
      }
    }
  }
  if (a.prologue == PRO_FULL && blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.sumsq_zero_n; i += blockDim.x) a.sumsq_zero[i] = 0.0;
}

// L2 prefetch of this block's share of [p, p + bytes) (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_share(const void* p, size_t bytes) {
  if (!p || !bytes) return;
  const size_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~size_t(15);
  size_t b0 = per * blockIdx.x;
  const size_t b1 = b0 + per < bytes ? b0 + per : bytes;
  for (; b0 < b1; b0 += 65536) {
    const size_t n = b1 - b0 < 65536 ? b1 - b0 : 65536;
    prefetch_l2(static_cast<const char*>(p) + b0, (uint32_t)n);
  }
}

template <typename Dt, int WF, int NT, int EPI>
__global__ void __launch_bounds__(G2_MAX_WARPS * 32, 1) gemv2_kernel(Gemv2Args a) {
  extern __shared__ __align__(128) uint8_t g2_smem[];
  using W = dec::WRow<Dt, WF>;
  constexpr bool PAIR = (EPI == EPI_SWIGLU);
  constexpr int U = (NT * (PAIR ? 2 : 1) * W::EPV > 32) ? 2 : 4;  // 16-byte vectors in flight per lane
  constexpr int XV = Vec16<Dt>::N;                                 // x elements per 16-byte vector
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int S = a.stages;
  const G2Layout L = g2_layout(W::BYTES, sizeof(Dt), NT, a.K, PAIR, S, nwarps);
  Dt* xs = reinterpret_cast<Dt*>(g2_smem);
  uint8_t* ring = g2_smem + L.x_bytes + (size_t)warp * S * L.unit_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(g2_smem + L.x_bytes + L.ring_bytes) + warp * S;
  float* red = reinterpret_cast<float*>(g2_smem + L.x_bytes + L.ring_bytes + (size_t)nwarps * S * 8);
  __shared__ float red_norm[64];

  const int gw = blockIdx.x * nwarps + warp, nw = gridDim.x * nwarps;
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
  // ... and ask L2 for the next kernel's operand, so HBM keeps streaming
  // across the kernel boundary.
  if (threadIdx.x == 32) prefetch_share(a.pf, a.pf_bytes);
  __syncwarp();
  pdl_wait();
  pdl_launch();
  g2_stage_x<Dt>(a, xs, red_norm);
  __syncthreads();

  const int nvec = a.K / W::EPV;
  F2 ssq = {0.f, 0.f};  // lane t: squares of updated elements of row t (residual epilogue)
  bool ok = true;
  int k = 0;
  for (;; ++k) {
    const int u = gw + k * nw;
    if (u >= a.N) break;
    const int s = k % S;
    // lane 0 waits for the row; the other lanes wait at the warp barrier
    int landed = 1;
    if (lane == 0) landed = mbar_wait(&bars[s], (uint32_t)((k / S) & 1), a.err, 1);
    __syncwarp();  // orders lane 0's acquire of the copy before the other lanes' reads
    if (!__shfl_sync(0xffffffffu, landed, 0)) { ok = false; break; }
    const uint8_t* slot = ring + (size_t)s * L.unit_bytes;
    float acc[NT][U], acc2[NT][U];  // independent chains, one per unrolled vector
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < U; ++i) acc[t][i] = acc2[t][i] = 0.f;
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
      uint4 q0[U], q1[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int v = v0 + 32 * i;
        if (v < nvec) {
          q0[i] = *reinterpret_cast<const uint4*>(slot + (size_t)v * 16);
          if (PAIR) q1[i] = *reinterpret_cast<const uint4*>(slot + L.row_bytes + (size_t)v * 16);
        }
      }
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const int v = v0 + 32 * i;
        if (v >= nvec) break;
        const int k0 = v * W::EPV;
        float w0[W::EPV], w1[W::EPV];
        W::get(q0[i], w0, a.scale, a.bias, a.K, a.group, (size_t)u, k0);
        if (PAIR) W::get(q1[i], w1, a.scale, a.bias, a.K, a.group, (size_t)u + a.N, k0);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          // this lane's x elements k0 .. k0 + EPV: contiguous 16-byte vectors
          float xv[W::EPV];
#pragma unroll
          for (int q = 0; q < W::EPV / XV; ++q)
            Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)t * a.K + k0 + q * XV), xv + q * XV);
#pragma unroll
          for (int e = 0; e < W::EPV; ++e) acc[t][i] = fmaf(w0[e], xv[e], acc[t][i]);
          if (PAIR) {
#pragma unroll
            for (int e = 0; e < W::EPV; ++e) acc2[t][i] = fmaf(w1[e], xv[e], acc2[t][i]);
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
    float r[NT], r2[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int i = 0; i < U; ++i) { s1 += acc[t][i]; s2 += acc2[t][i]; }
      r[t] = warp_sum(s1);
      r2[t] = PAIR ? warp_sum(s2) : 0.f;
    }
    if (lane < NT) {
      float v = r[0], v2 = r2[0];
#pragma unroll
      for (int t = 1; t < NT; ++t)
        if (lane == t) { v = r[t]; v2 = r2[t]; }
      const size_t o = (size_t)lane * a.ldo + u;
      if (EPI == EPI_STORE) {
        static_cast<Dt*>(a.out)[o] = from_f<Dt>(v);
      } else if (EPI == EPI_STORE_F32) {
        static_cast<float*>(a.out)[o] = v;
      } else if (EPI == EPI_RESIDUAL) {
        Dt* p = static_cast<Dt*>(a.out) + o;
        const float hn = rd<Dt>(to_f(*p) + rd<Dt>(v));
        *p = from_f<Dt>(hn);
        f2_add_sq(ssq, hn);
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
    if (lane < NT) { red[(warp * 4 + lane) * 2] = ssq.hi; red[(warp * 4 + lane) * 2 + 1] = ssq.lo; }
    __syncthreads();
    if (threadIdx.x < NT) {
      F2 s = {0.f, 0.f};
      for (int w = 0; w < nwarps; ++w) s = f2_add(s, F2{red[(w * 4 + threadIdx.x) * 2], red[(w * 4 + threadIdx.x) * 2 + 1]});
      atomicAdd(a.sumsq_out + threadIdx.x, (double)s.hi + (double)s.lo);
    }
  }
}

template <typename Dt, int WF, int NT, int EPI>
cudaError_t g2_launch(const LaunchCtx& c, const Gemv2Args& a) {
  auto kern = gemv2_kernel<Dt, WF, NT, EPI>;
  cudaError_t e = set_max_smem((const void*)kern, (int)G2_SMEM_LIMIT);
  if (e != cudaSuccess) return e;
  const G2Layout L = g2_layout(WF == W_U8 ? 1 : (int)sizeof(Dt), (int)sizeof(Dt), NT, a.K, EPI == EPI_SWIGLU,
                               a.stages, a.nwarps);
  int grid = (a.N + a.nwarps - 1) / a.nwarps;
  if (grid > c.num_sms) grid = c.num_sms;
  return launch_k(kern, dim3(grid), dim3(a.nwarps * 32), L.total, c, a);
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

// ============================================================ norm_apply
template <typename Dt>
__global__ void __launch_bounds__(256) norm_apply_kernel(NormApplyArgs a) {
  constexpr int V = Vec16<Dt>::N;
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  __shared__ F2 s_rs;
  if (threadIdx.x == 0) s_rs = rms_scale2(f2_from_double(a.sumsq[t]), a.hidden, a.eps);
  __syncthreads();
  const F2 rs = s_rs;
  const Dt* h = static_cast<const Dt*>(a.h) + (size_t)t * a.hidden;
  const Dt* g = static_cast<const Dt*>(a.gain);
  Dt* out = static_cast<Dt*>(a.out) + (size_t)t * a.hidden;
  for (int k = threadIdx.x * V; k < a.hidden; k += blockDim.x * V) {
    float hv[V], gv[V], o[V];
    Vec16<Dt>::unpack(ld16(h + k), hv);
    Vec16<Dt>::unpack(ld16(g + k), gv);
    rms_apply2_v<Dt, V>(hv, rs, gv, o);
    *reinterpret_cast<uint4*>(out + k) = Vec16<Dt>::pack(o);
  }
}

}  // namespace

int gemv2_plan(int dt, int wfmt, int T, int K, int group, bool pair, int* nwarps, bool coresident) {
  (void)group;
  const int wbytes = wfmt == W_U8 ? 1 : (dt == DT_BF16 ? 2 : 4);
  const int xbytes = dt == DT_BF16 ? 2 : 4;
  // co-resident: at most half of an SM (shared memory, threads), so the next
  // kernel's CTAs, launched early, start streaming their weights beside these
  const size_t limit = coresident ? G2_SMEM_CORES : G2_SMEM_LIMIT;
  const int max_warps = coresident ? G2_MAX_WARPS / 2 : G2_MAX_WARPS;
  for (int nw = max_warps; nw >= 4; nw /= 2)
    for (int s = 4; s >= (nw == 4 ? 1 : 2); --s) {
      const G2Layout L = g2_layout(wbytes, xbytes, T, K, pair, s, nw);
      if (L.total <= limit) {
        if (nwarps) *nwarps = nw;
        return s;
      }
    }
  if (nwarps) *nwarps = 4;
  if (g2_layout(wbytes, xbytes, T, K, pair, 1, 4).total <= limit) return 1;
  return coresident ? gemv2_plan(dt, wfmt, T, K, group, pair, nwarps, false) : 0;
}

cudaError_t launch_gemv2(const LaunchCtx& c, int dt, int wfmt, const Gemv2Args& a) {
  if (a.T < 1 || a.T > 4 || a.stages < 1 || a.nwarps < 1 || a.nwarps > G2_MAX_WARPS) return cudaErrorInvalidValue;
  if (dt == DT_BF16) return wfmt == W_U8 ? g2_epi<bf16, W_U8>(c, a) : g2_epi<bf16, W_DT>(c, a);
  return wfmt == W_U8 ? g2_epi<float, W_U8>(c, a) : g2_epi<float, W_DT>(c, a);
}

cudaError_t launch_norm_apply(const LaunchCtx& c, int dt, const NormApplyArgs& a) {
  if (dt == DT_BF16) return launch_k(norm_apply_kernel<bf16>, dim3(a.T), dim3(256), 0, c, a);
  return launch_k(norm_apply_kernel<float>, dim3(a.T), dim3(256), 0, c, a);
}

}  // namespace q3
