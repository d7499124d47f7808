// Fused residual add + RMSNorm, and per-head q/k RMSNorm + RoPE + KV-cache
// append (maya2_mlx/backbone.py, Backbone.forward and Backbone._rope).
#include "common.cuh"
#include "kernels.h"

namespace q3 {

// h = R(h_in + pend); y = R(R(h * rsqrt(mean(h^2) + eps)) * gain) -- the
// Backbone's "one rounding" add and Qwen3's "two roundings" RMSNorm.
template <typename Dt>
__global__ void __launch_bounds__(256) add_rmsnorm_kernel(NormArgs a) {
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
    for (int e = 0; e < V; ++e) f2_add_sq(ss, h[e]);
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
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] = rms_apply2<Dt>(h[e], rs, gg[e]);
    *reinterpret_cast<uint4*>(y + i) = Vec16<Dt>::pack(o);
  }
}

cudaError_t launch_add_rmsnorm(const LaunchCtx& c, int dt, const NormArgs& a) {
  if (dt == DT_BF16) return launch_k(add_rmsnorm_kernel<bf16>, dim3(a.rows), dim3(256), 0, c, a);
  return launch_k(add_rmsnorm_kernel<float>, dim3(a.rows), dim3(256), 0, c, a);
}

// One warp per (row, head) with heads 0..H-1 = q, H..H+KV-1 = k, then v.
// Lane l holds elements [l*EPL, (l+1)*EPL) of the head; the RoPE partner of
// element d (d < D/2) is d + D/2, held by lane l ^ 16.
template <typename Dt, int D>
__global__ void __launch_bounds__(256) qk_rope_cache_kernel(QkRopeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nh = a.H + 2 * a.KV;
  if (gw >= a.T * nh) return;
  const int t = gw / nh, hh = gw % nh;
  const Dt* src = static_cast<const Dt*>(a.qkv) + (size_t)t * nh * D + (size_t)hh * D + lane * EPL;
  float x[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = to_f(src[e]);
  const int seq = a.row_seq[t], pos = a.row_pos[t];
  if (hh >= a.H + a.KV) {  // v: appended as produced
    Dt* dst = static_cast<Dt*>(a.vcache) + (size_t)seq * a.seq_stride +
              ((size_t)(hh - a.H - a.KV) * a.capacity + pos) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = from_f<Dt>(x[e]);
    return;
  }
  const bool is_q = hh < a.H;
  const Dt* gain = static_cast<const Dt*>(is_q ? a.q_gain : a.k_gain) + lane * EPL;
  F2 ss = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < EPL; ++e) f2_add_sq(ss, x[e]);
  ss = f2_warp_sum(ss);
  const F2 rs = rms_scale2(ss, D, a.eps);
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = rms_apply2<Dt>(x[e], rs, to_f(gain[e]));
  // RoPE: o1 = y1*c - y2*s (first half), o2 = y2*c + y1*s (second half), one
  // rounding.  bf16: both products are exact in fp32 and fmaf rounds their
  // difference once; fp32: formed and differenced in double.
  const float* cs = a.cos_t + (size_t)pos * D + lane * EPL;
  const float* sn = a.sin_t + (size_t)pos * D + lane * EPL;
  const bool first = lane < 16;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
    if (sizeof(Dt) == 2) {
      const float ps = partner * sn[e];  // exact: 8-bit x 8-bit significands
      o[e] = rd<Dt>(first ? fmaf(x[e], cs[e], -ps) : fmaf(x[e], cs[e], ps));
    } else {
      const double xc = (double)x[e] * (double)cs[e], ps = (double)partner * (double)sn[e];
      o[e] = rd_d<Dt>(first ? xc - ps : xc + ps);
    }
  }
  Dt* dst;
  if (is_q) {
    dst = static_cast<Dt*>(a.q_out) + ((size_t)t * a.H + hh) * D + lane * EPL;
  } else {
    dst = static_cast<Dt*>(a.kcache) + (size_t)seq * a.seq_stride +
          ((size_t)(hh - a.H) * a.capacity + pos) * D + lane * EPL;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) dst[e] = from_f<Dt>(o[e]);
}

cudaError_t launch_qk_rope_cache(const LaunchCtx& c, int dt, const QkRopeArgs& a) {
  const int warps = a.T * (a.H + 2 * a.KV);
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
