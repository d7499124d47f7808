// Weight-streaming GEMV for decode-sized row counts (maya2_mlx/backbone.py,
// Backbone.forward: `Q.mm(y, L["qkv"])`, `Q.mm(..., L["o"])`,
// `Q.mm(y2, L["gu"])` with the fp32 SiLU * up, `Q.mm(act * u, L["down"])`;
// @mlx-bun/inference qwen3-moe.ts Qwen3UnsortedExperts for the gathered
// expert projections).
//
// Used for the MoE router logits and the gathered (unsorted) expert
// projections of few rows: each warp streams whole weight rows with 16-byte
// non-allocating loads while the input rows sit in shared memory in the model
// dtype (each lane reads its x elements as contiguous 16-byte vectors, free of
// bank conflicts).
// Before waiting on the producer kernel, every block asks L2 to prefetch its
// weight rows (shared-weight mode).  Epilogues fuse rounding, fp32 output,
// the residual add and SiLU * up.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per lane per row

template <typename Dt, int WF> struct WTraits;
template <typename Dt> struct WTraits<Dt, W_DT> {
  static constexpr int EPV = Vec16<Dt>::N;
  static constexpr int BYTES = sizeof(Dt);
  __device__ static __forceinline__ void get(const uint4& r, float* w, const GemvArgs&, size_t, int) {
    Vec16<Dt>::unpack(r, w);
  }
};
template <typename Dt> struct WTraits<Dt, W_U8> {
  static constexpr int EPV = 16;
  static constexpr int BYTES = 1;
  // 16 codes of row `row` starting at element k0 (inside one group).
  __device__ static __forceinline__ void get(const uint4& r, float* w, const GemvArgs& a, size_t row,
                                             int k0) {
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

// Stage the input rows in shared memory in the model dtype (16-byte copies).
template <typename Dt>
__device__ void stage_x(const GemvArgs& a, Dt* xs) {
  constexpr int V = Vec16<Dt>::N;
  const Dt* x = static_cast<const Dt*>(a.x);
  for (int c = threadIdx.x; c < a.x_rows * a.K / V; c += blockDim.x)
    *reinterpret_cast<uint4*>(xs + (size_t)c * V) = ld16(x + (size_t)c * V);
}

template <typename Dt, int WF, int NT, int EPI>
__global__ void __launch_bounds__(kThreads) gemv_kernel(GemvArgs a) {
  extern __shared__ __align__(16) uint8_t gv_smem[];
  Dt* xs = reinterpret_cast<Dt*>(gv_smem);
  using W = WTraits<Dt, WF>;
  constexpr int XV = Vec16<Dt>::N;  // x elements per 16-byte vector
  constexpr bool PAIR = (EPI == EPI_SWIGLU);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool gather = a.slot_expert != nullptr;
  const long long units = gather ? (long long)a.T * a.N : (long long)a.N;
  const long long u0 = units * blockIdx.x / gridDim.x;
  const long long u1 = units * (blockIdx.x + 1) / gridDim.x;
  const size_t row_bytes = (size_t)a.K * W::BYTES;
  const char* wb = static_cast<const char*>(a.w);

  // Weights do not depend on the previous kernel: prefetch this block's rows.
  if (!gather && threadIdx.x == 0 && u1 > u0) {
    const size_t bytes = (size_t)(u1 - u0) * row_bytes;
    prefetch_l2(wb + (size_t)u0 * row_bytes, (uint32_t)bytes);
    if (PAIR) prefetch_l2(wb + (size_t)(u0 + a.N) * row_bytes, (uint32_t)bytes);
  }
  pdl_wait();
  pdl_launch();
  stage_x<Dt>(a, xs);
  __syncthreads();

  const int nvec = a.K / W::EPV;
  for (long long u = u0 + warp; u < u1; u += kWarps) {
    int b = 0, n = (int)u;
    size_t row = (size_t)n;  // row of the weight (stacked experts: counted across all experts)
    if (gather) {
      b = (int)(u / a.N);
      n = (int)(u % a.N);
      row = (size_t)a.slot_expert[b] * (size_t)(a.w_stride / a.K) + (size_t)n;
    }
    const char* r0 = wb + row * row_bytes;
    const char* r1 = wb + (row + a.N) * row_bytes;
    const Dt* xrow = xs + (size_t)(gather ? b / a.slot_div : 0) * a.K;
    float acc[NT], acc2[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = acc2[t] = 0.f;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
      uint4 q0[kUnroll], q1[kUnroll];
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int v = v0 + 32 * i;
        if (v < nvec) {
          q0[i] = ld_stream(r0 + (size_t)v * 16);
          if (PAIR) q1[i] = ld_stream(r1 + (size_t)v * 16);
        }
      }
#pragma unroll
      for (int i = 0; i < kUnroll; ++i) {
        const int v = v0 + 32 * i;
        if (v >= nvec) break;
        const int k0 = v * W::EPV;
        float w0[W::EPV], w1[W::EPV];
        W::get(q0[i], w0, a, row, k0);
        if (PAIR) W::get(q1[i], w1, a, row + a.N, k0);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          float xv[W::EPV];
#pragma unroll
          for (int q = 0; q < W::EPV / XV; ++q)
            Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(xrow + (size_t)t * a.K + k0 + q * XV), xv + q * XV);
#pragma unroll
          for (int e = 0; e < W::EPV; ++e) acc[t] = fmaf(w0[e], xv[e], acc[t]);
          if (PAIR) {
#pragma unroll
            for (int e = 0; e < W::EPV; ++e) acc2[t] = fmaf(w1[e], xv[e], acc2[t]);
          }
        }
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
      const size_t orow = gather ? (size_t)b : (size_t)lane;
      const size_t o = orow * (size_t)a.ldo + n;
      if (EPI == EPI_STORE) {
        static_cast<Dt*>(a.out)[o] = from_f<Dt>(v);
      } else if (EPI == EPI_STORE_F32) {
        static_cast<float*>(a.out)[o] = v;
      } else if (EPI == EPI_STORE_RF32) {
        static_cast<float*>(a.out)[o] = rd<Dt>(v);
      } else if (EPI == EPI_RESIDUAL) {
        Dt* p = static_cast<Dt*>(a.out) + o;
        *p = from_f<Dt>(to_f(*p) + rd<Dt>(v));
      } else {  // SwiGLU: act = R(silu(R(g))) in fp32, out = R(act * R(u))
        const float g = rd<Dt>(v), up = rd<Dt>(v2);
        static_cast<Dt*>(a.out)[o] = from_f<Dt>(rd<Dt>(silu_f(g)) * up);
      }
    }
  }
}

template <typename Dt, int WF, int NT, int EPI>
cudaError_t launch_one(const LaunchCtx& c, const GemvArgs& a) {
  auto kern = gemv_kernel<Dt, WF, NT, EPI>;
  const size_t smem = gemv_smem_bytes(a);
  cudaError_t e = set_max_smem((const void*)kern, 200 * 1024);
  if (e != cudaSuccess) return e;
  const long long units = a.slot_expert ? (long long)a.T * a.N : (long long)a.N;
  long long grid = (units + kWarps - 1) / kWarps;
  const long long cap = (long long)c.num_sms * 4;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_k(kern, dim3((unsigned)grid), dim3(kThreads), smem, c, a);
}

template <typename Dt, int WF, int EPI>
cudaError_t launch_nt(const LaunchCtx& c, const GemvArgs& a) {
  const int nt = a.slot_expert ? 1 : a.T;
  switch (nt) {
    case 1: return launch_one<Dt, WF, 1, EPI>(c, a);
    case 2: return launch_one<Dt, WF, 2, EPI>(c, a);
    case 3: return launch_one<Dt, WF, 3, EPI>(c, a);
    case 4: return launch_one<Dt, WF, 4, EPI>(c, a);
    default: return cudaErrorInvalidValue;
  }
}

template <typename Dt, int WF>
cudaError_t launch_epi(const LaunchCtx& c, const GemvArgs& a) {
  switch (a.epilogue) {
    case EPI_STORE: return launch_nt<Dt, WF, EPI_STORE>(c, a);
    case EPI_STORE_F32: return launch_nt<Dt, WF, EPI_STORE_F32>(c, a);
    case EPI_STORE_RF32: return launch_nt<Dt, WF, EPI_STORE_RF32>(c, a);
    case EPI_RESIDUAL: return launch_nt<Dt, WF, EPI_RESIDUAL>(c, a);
    case EPI_SWIGLU: return launch_nt<Dt, WF, EPI_SWIGLU>(c, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t gemv_smem_bytes(const GemvArgs& a) { return (size_t)a.x_rows * a.K * sizeof(float); }

cudaError_t launch_gemv(const LaunchCtx& c, int dt, int wfmt, const GemvArgs& a) {
  if (gemv_smem_bytes(a) > 200 * 1024) return cudaErrorInvalidValue;
  if (dt == DT_BF16) {
    if (wfmt == W_U8) return launch_epi<bf16, W_U8>(c, a);
    return launch_epi<bf16, W_DT>(c, a);
  }
  if (wfmt == W_U8) return launch_epi<float, W_U8>(c, a);
  return launch_epi<float, W_DT>(c, a);
}

}  // namespace q3
