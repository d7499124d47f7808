// Device helpers shared by the decode-path kernels (weight-row decoding for
// the streaming GEMVs; per-head RMSNorm + RoPE; lane vectors of a head row).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace q3 {
namespace dec {

// One 16-byte weight vector as floats: model-dtype weights, or affine int8
// codes dequantised as scale * q + bias with the row's group scale and bias.
template <typename Dt, int WF> struct WRow;
template <typename Dt> struct WRow<Dt, W_DT> {
  static constexpr int EPV = Vec16<Dt>::N;
  static constexpr int BYTES = sizeof(Dt);
  __device__ static __forceinline__ void get(const uint4& r, float* w, const void*, const void*, int, int, size_t,
                                             int) {
    Vec16<Dt>::unpack(r, w);
  }
};
template <typename Dt> struct WRow<Dt, W_U8> {
  static constexpr int EPV = 16;
  static constexpr int BYTES = 1;
  // row `row` of a [rows, K] code matrix, elements k0 .. k0 + 15 (one group)
  __device__ static __forceinline__ void get(const uint4& r, float* w, const void* scale, const void* bias, int K,
                                             int group, size_t row, int k0) {
    const size_t gi = row * (size_t)(K / group) + k0 / group;
    const float s = __bfloat162float(static_cast<const bf16*>(scale)[gi]);
    const float b = __bfloat162float(static_cast<const bf16*>(bias)[gi]);
    const uint32_t v[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[4 * i + j] = fmaf(s, (float)((v[i] >> (8 * j)) & 0xffu), b);
  }
};

// Per-head RMSNorm + RoPE of one raw q or k head (warp-wide: lane holds
// elements lane*DPL .. +DPL) at position pos, rounded to the model dtype.
// RMS statistics in compensated fp32 pairs.  RoPE: for bf16 both products
// are exact in fp32 and fmaf rounds their difference once; for fp32 they are
// formed in double.
template <typename Dt, int D>
__device__ __forceinline__ void norm_rope_head(float* x, const Dt* gain, const float* cos_t, const float* sin_t,
                                               int pos, float eps) {
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  float cs[DPL], sn[DPL], gg[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) {
    cs[e] = cos_t[(size_t)pos * D + lane * DPL + e];
    sn[e] = sin_t[(size_t)pos * D + lane * DPL + e];
    gg[e] = to_f(gain[lane * DPL + e]);
  }
  F2 ss = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < DPL; ++e) f2_add_sq(ss, x[e]);
  ss = f2_warp_sum(ss);
  const F2 rs = rms_scale2(ss, D, eps);
#pragma unroll
  for (int e = 0; e < DPL; ++e) x[e] = rms_apply2<Dt>(x[e], rs, gg[e]);
  const bool first = lane < 16;
  float o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) {
    const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
    if (sizeof(Dt) == 2) {
      const float ps = partner * sn[e];  // exact: 8-bit x 8-bit significands
      o[e] = rd<Dt>(first ? fmaf(x[e], cs[e], -ps) : fmaf(x[e], cs[e], ps));
    } else {
      const double xc = (double)x[e] * (double)cs[e], pd = (double)partner * (double)sn[e];
      o[e] = rd_d<Dt>(first ? xc - pd : xc + pd);
    }
  }
#pragma unroll
  for (int e = 0; e < DPL; ++e) x[e] = o[e];
}

// DPL consecutive elements at p (one aligned vector load) as floats.
template <typename Dt, int DPL>
__device__ __forceinline__ void load_lane_vec(const Dt* p, float* v) {
  constexpr int BYTES = DPL * (int)sizeof(Dt);
  static_assert(BYTES == 4 || BYTES == 8 || BYTES == 16, "lane vector");
  constexpr int NW = BYTES / 4;
  uint32_t w[NW];
  if (NW == 4) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    w[0] = r.x; w[NW > 1 ? 1 : 0] = r.y; w[NW > 2 ? 2 : 0] = r.z; w[NW > 3 ? 3 : 0] = r.w;
  } else if (NW == 2) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    w[0] = r.x; w[NW > 1 ? 1 : 0] = r.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
#pragma unroll
  for (int e = 0; e < DPL; ++e)
    v[e] = sizeof(Dt) == 2 ? __uint_as_float((e & 1) ? (w[e / 2] & 0xffff0000u) : (w[e / 2] << 16))
                           : __uint_as_float(w[e]);
}
template <int DPL>
__device__ __forceinline__ void store_lane_vec(float* p, const float* v) {
  if (DPL == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[DPL > 1 ? 1 : 0], v[DPL > 2 ? 2 : 0], v[DPL > 3 ? 3 : 0]);
  } else if (DPL == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[DPL > 1 ? 1 : 0]);
  } else {
#pragma unroll
    for (int e = 0; e < DPL; ++e) p[e] = v[e];
  }
}

}  // namespace dec
}  // namespace q3
