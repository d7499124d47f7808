// Fused residual add + RMSNorm, and per-head q/k RMSNorm + RoPE + KV-cache
// append (maya2_mlx/backbone.py, Backbone.forward and Backbone._rope).
#include "common.cuh"
#include "kernels.h"

namespace q3 {

// h = R(h_in + pend); y = R(R(h * rsqrt(mean(h^2) + eps)) * gain) -- the
// Backbone's "one rounding" add and Qwen3's "two roundings" RMSNorm.
template <typename Dt>
__global__ void __launch_bounds__(256, 8) add_rmsnorm_kernel(NormArgs a) {  // 8 blocks per SM
  __shared__ float red[64];
  pdl_wait();
  pdl_launch();
  const int row = blockIdx.x;
  const Dt* hi = static_cast<const Dt*>(a.h_in) + (size_t)row * a.hidden;
  const Dt* pe = a.pend ? static_cast<const Dt*>(a.pend) + (size_t)row * a.hidden : nullptr;
  Dt* ho = static_cast<Dt*>(a.h_out) + (size_t)row * a.hidden;
  constexpr int V = Vec16<Dt>::N;
  F2 ss = {0.f, 0.f};
  for (int i = threadIdx.x * V; i < a.hidden; i += blockDim.x * V) {
    float h[V];
    Vec16<Dt>::unpack(ld16(hi + i), h);
    if (pe) {
      float p[V];
      Vec16<Dt>::unpack(ld16(pe + i), p);
#pragma unroll
      for (int e = 0; e < V; ++e) h[e] = rd<Dt>(h[e] + p[e]);
    }
    if (pe || ho != hi) *reinterpret_cast<uint4*>(ho + i) = Vec16<Dt>::pack(h);
#pragma unroll
    for (int e = 0; e < V; ++e) {
      if constexpr (sizeof(Dt) == 2) f2_add_sq_exact(ss, h[e]);  // bf16: the square is exact
      else f2_add_sq(ss, h[e]);
    }
  }
  ss = f2_block_sum(ss, red);
  if (!a.y) return;
  const F2 rs = rms_scale2(ss, a.hidden, a.eps);
  const Dt* g = static_cast<const Dt*>(a.gain);
  Dt* y = static_cast<Dt*>(a.y) + (size_t)row * a.hidden;
  for (int i = threadIdx.x * V; i < a.hidden; i += blockDim.x * V) {
    float h[V], gg[V], o[V];
    Vec16<Dt>::unpack(ld16(ho + i), h);  // own writes of this thread: visible
    Vec16<Dt>::unpack(ld16(g + i), gg);
    rms_apply2_v<Dt, V>(h, rs, gg, o);
    *reinterpret_cast<uint4*>(y + i) = Vec16<Dt>::pack(o);
  }
}

cudaError_t launch_add_rmsnorm(const LaunchCtx& c, int dt, const NormArgs& a) {
  if (dt == DT_BF16) return launch_k(add_rmsnorm_kernel<bf16>, dim3(a.rows), dim3(256), 0, c, a);
  return launch_k(add_rmsnorm_kernel<float>, dim3(a.rows), dim3(256), 0, c, a);
}

// EPL consecutive elements of the model dtype <-> fp32, one vector access.
template <typename Dt, int EPL>
__device__ __forceinline__ void ld_vec(const Dt* p, float* x) {
  if constexpr (sizeof(Dt) == 2 && EPL == 4) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xffff0000u);
  } else if constexpr (sizeof(Dt) == 2 && EPL == 2) {
    const uint32_t r = *reinterpret_cast<const uint32_t*>(p);
    x[0] = __uint_as_float(r << 16); x[1] = __uint_as_float(r & 0xffff0000u);
  } else if constexpr (EPL == 4) {
    const float4 r = *reinterpret_cast<const float4*>(p);
    x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
  } else {
    const float2 r = *reinterpret_cast<const float2*>(p);
    x[0] = r.x; x[1] = r.y;
  }
}
template <typename Dt, int EPL>
__device__ __forceinline__ void st_vec(Dt* p, const float* x) {
  if constexpr (sizeof(Dt) == 2 && EPL == 4) {
    uint2 r;
    r.x = __bfloat16_as_ushort(__float2bfloat16_rn(x[0])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[1])) << 16);
    r.y = __bfloat16_as_ushort(__float2bfloat16_rn(x[2])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[3])) << 16);
    *reinterpret_cast<uint2*>(p) = r;
  } else if constexpr (sizeof(Dt) == 2 && EPL == 2) {
    *reinterpret_cast<uint32_t*>(p) =
        __bfloat16_as_ushort(__float2bfloat16_rn(x[0])) | ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[1])) << 16);
  } else if constexpr (EPL == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  }
}
template <int EPL>
__device__ __forceinline__ void ld_f32(const float* p, float* x) {
  if constexpr (EPL == 4) {
    const float4 r = *reinterpret_cast<const float4*>(p);
    x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
  } else {
    const float2 r = *reinterpret_cast<const float2*>(p);
    x[0] = r.x; x[1] = r.y;
  }
}

// One warp per (row, group of up to RH heads of one kind): groups of q
// heads, then of k heads, then of v heads.  Lane l holds elements
// [l*EPL, (l+1)*EPL) of every head of its group (one vector access each, all
// in flight at once); the gain, cos and sin are loaded once per warp.  The
// RoPE partner of element d (d < D/2) is d + D/2, held by lane l ^ 16.
constexpr int RH = 4;
template <typename Dt, int D>
__global__ void __launch_bounds__(256) qk_rope_cache_kernel(QkRopeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int gq = (a.H + RH - 1) / RH, gk = (a.KV + RH - 1) / RH, ng = gq + 2 * gk;
  if (gw >= a.T * ng) return;
  const int t = gw / ng, g = gw % ng;
  const int kind = g < gq ? 0 : g < gq + gk ? 1 : 2;  // q, k, v
  const int first = kind == 0 ? g * RH : (g - gq - (kind == 2 ? gk : 0)) * RH;
  const int nheads = min(RH, (kind == 0 ? a.H : a.KV) - first);
  const int col0 = kind == 0 ? first : kind == 1 ? a.H + first : a.H + a.KV + first;  // head index in the qkv row
  const int nh = a.H + 2 * a.KV;
  const Dt* src = static_cast<const Dt*>(a.qkv) + (size_t)t * nh * D + (size_t)col0 * D + lane * EPL;
  float x[RH][EPL];
#pragma unroll
  for (int r = 0; r < RH; ++r)
    if (r < nheads) ld_vec<Dt, EPL>(src + (size_t)r * D, x[r]);
  const int seq = a.row_seq[t], pos = a.row_pos[t];
  if (kind == 2) {  // v: appended as produced
#pragma unroll
    for (int r = 0; r < RH; ++r)
      if (r < nheads)
        st_vec<Dt, EPL>(static_cast<Dt*>(a.vcache) + (size_t)seq * a.seq_stride +
                            ((size_t)(first + r) * a.capacity + pos) * D + lane * EPL,
                        x[r]);
    return;
  }
  float gain[EPL], cs[EPL], sn[EPL];
  ld_vec<Dt, EPL>(static_cast<const Dt*>(kind == 0 ? a.q_gain : a.k_gain) + lane * EPL, gain);
  ld_f32<EPL>(a.cos_t + (size_t)pos * D + lane * EPL, cs);
  ld_f32<EPL>(a.sin_t + (size_t)pos * D + lane * EPL, sn);
  F2 ss[RH];
#pragma unroll
  for (int r = 0; r < RH; ++r) {
    ss[r] = F2{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < EPL; ++e) f2_add_sq(ss[r], x[r][e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < RH; ++r) {
      F2 b;
      b.hi = __shfl_xor_sync(0xffffffffu, ss[r].hi, o);
      b.lo = __shfl_xor_sync(0xffffffffu, ss[r].lo, o);
      ss[r] = f2_add(ss[r], b);
    }
  const bool lo_half = lane < 16;
#pragma unroll
  for (int r = 0; r < RH; ++r) {
    if (r >= nheads) break;
    const F2 rs = rms_scale2(ss[r], D, a.eps);
    rms_apply2_v<Dt, EPL>(x[r], rs, gain, x[r]);
    // RoPE: o1 = y1*c - y2*s (first half), o2 = y2*c + y1*s (second half), one
    // rounding.  bf16: both products are exact in fp32 and fmaf rounds their
    // difference once; fp32: formed and differenced in double.
    float o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float partner = __shfl_xor_sync(0xffffffffu, x[r][e], 16);
      if (sizeof(Dt) == 2) {
        const float ps = partner * sn[e];  // exact: 8-bit x 8-bit significands
        o[e] = rd<Dt>(lo_half ? fmaf(x[r][e], cs[e], -ps) : fmaf(x[r][e], cs[e], ps));
      } else {
        const double xc = (double)x[r][e] * (double)cs[e], ps = (double)partner * (double)sn[e];
        o[e] = rd_d<Dt>(lo_half ? xc - ps : xc + ps);
      }
    }
    Dt* dst = kind == 0 ? static_cast<Dt*>(a.q_out) + ((size_t)t * a.H + first + r) * D + lane * EPL
                        : static_cast<Dt*>(a.kcache) + (size_t)seq * a.seq_stride +
                              ((size_t)(first + r) * a.capacity + pos) * D + lane * EPL;
    st_vec<Dt, EPL>(dst, o);
  }
}

cudaError_t launch_qk_rope_cache(const LaunchCtx& c, int dt, const QkRopeArgs& a) {
  const int warps = a.T * ((a.H + RH - 1) / RH + 2 * ((a.KV + RH - 1) / RH));
  const dim3 grid((warps + 7) / 8), block(256);
  if (a.D == 128) {
    if (dt == DT_BF16) return launch_k(qk_rope_cache_kernel<bf16, 128>, grid, block, 0, c, a);
    return launch_k(qk_rope_cache_kernel<float, 128>, grid, block, 0, c, a);
  }
  if (a.D == 64) {
    if (dt == DT_BF16) return launch_k(qk_rope_cache_kernel<bf16, 64>, grid, block, 0, c, a);
    return launch_k(qk_rope_cache_kernel<float, 64>, grid, block, 0, c, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace q3
