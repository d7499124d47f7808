// Shared device helpers: dtype conversion and rounding, warp/block
// reductions, streaming loads, programmatic-dependent-launch controls.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

namespace q3 {

// Raise a kernel's dynamic shared-memory limit on the current device.  The
// attribute belongs to a (kernel, device) pair, so it is set once for each
// pair seen (under a lock; launches from several threads are safe): the first
// call fixes the limit, so `bytes` must be the most the kernel is ever
// launched with.
inline cudaError_t set_max_smem(const void* kern, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kern, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kern, dev});
  return e;
}

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename Dt> __device__ __forceinline__ Dt from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// Round an fp32 value to the model dtype and back (round to nearest even).
template <typename Dt> __device__ __forceinline__ float rd(float x) { return to_f(from_f<Dt>(x)); }

// Round a double straight to the model dtype (one rounding, ties to even) and
// return it as fp32 (exact: the result has at most 24 significant bits).
// bf16: keep 8 significant bits of the double's 53 by adding half of the
// dropped 45-bit field (minus one unless the kept lsb is odd) and truncating.
// Normal-range values only, which is every value rounded here.
template <typename Dt> __device__ __forceinline__ float rd_d(double x);
template <> __device__ __forceinline__ float rd_d<float>(double x) { return __double2float_rn(x); }
template <> __device__ __forceinline__ float rd_d<__nv_bfloat16>(double x) {
  unsigned long long b = (unsigned long long)__double_as_longlong(x);
  const unsigned long long lsb = (b >> 45) & 1ull;
  b += (1ull << 44) - 1ull + lsb;
  b &= ~((1ull << 45) - 1ull);
  return (float)__longlong_as_double((long long)b);
}

// Unpack 16 bytes of a dtype into fp32 (8 bf16 or 4 fp32).
template <typename Dt> struct Vec16;
template <> struct Vec16<bf16> {
  static constexpr int N = 8;
  __device__ static __forceinline__ void unpack(const uint4& r, float* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i + 1]));
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static __forceinline__ void unpack(const uint4& r, float* f) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// 16-byte load of data read once (weights, KV): bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld16(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// Programmatic dependent launch.  wait: block until the preceding kernel in
// the stream has completed and its memory is visible (a no-op when the launch
// did not use the attribute).  launch: allow the next kernel to start its
// prologue.  Every kernel here calls wait before touching data another kernel
// writes, and launch only after wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bulk prefetch of a global range into L2 (no completion tracking needed).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- TMA / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Order this thread's earlier generic-proxy shared-memory accesses before its
// following async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`: gives up after ~2^31 SM cycles
// (about a second), records `code` in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 31)) {
      if (err) atomicExch(err, code);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block; `red` must hold 32 floats.  All threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  return warp_sum(t);
}

// ---------------------------------------------------------------- double-float
// fp32 pairs (hi + lo) with error-free transformations: FP64 throughput on this
// part is a small fraction of FP32, so the RMSNorm statistics, scale and
// normalised product are carried in pairs of floats instead of doubles, with
// the same effect (no rounding decision differs from exact arithmetic except
// where the exact value is within ~2^-40 relative of a tie).
struct F2 {
  float hi, lo;
};
// s + e == a + b exactly (Knuth's two-sum; additions only, so no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e += a.lo + b.lo;
  F2 r;
  r.hi = s + e;
  r.lo = e - (r.hi - s);
  return r;
}
// Add v*v (formed exactly with an fma for the low part) to an accumulator.
__device__ __forceinline__ void f2_add_sq(F2& acc, float v) {
  const float p = v * v;
  const float pe = fmaf(v, v, -p);
  float s, e;
  two_sum(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo += e + pe;
}
// The same when v * v is exact in fp32 (v a bf16 value: 8-bit significand).
__device__ __forceinline__ void f2_add_sq_exact(F2& acc, float v) {
  const float p = v * v;
  float s, e;
  two_sum(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo += e;
}
__device__ __forceinline__ F2 f2_warp_sum(F2 a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    F2 b;
    b.hi = __shfl_xor_sync(0xffffffffu, a.hi, o);
    b.lo = __shfl_xor_sync(0xffffffffu, a.lo, o);
    a = f2_add(a, b);
  }
  return a;
}
// Sum over the block; `red` must hold 64 floats.  All threads get the result.
__device__ __forceinline__ F2 f2_block_sum(F2 v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = f2_warp_sum(v);
  __syncthreads();
  if (lane == 0) { red[2 * warp] = v.hi; red[2 * warp + 1] = v.lo; }
  __syncthreads();
  F2 t;
  t.hi = lane < nw ? red[2 * lane] : 0.f;
  t.lo = lane < nw ? red[2 * lane + 1] : 0.f;
  return f2_warp_sum(t);
}
__device__ __forceinline__ F2 f2_from_double(double d) {
  F2 r;
  r.hi = (float)d;
  r.lo = (float)(d - (double)r.hi);
  return r;
}

// RMSNorm scale 1/sqrt(sumsq/n + eps) as a float pair: rsqrtf, then one Newton
// step evaluated with error-free products (relative error ~1e-13).
__device__ __forceinline__ F2 rms_scale2(F2 ss, int n, float eps) {
  const float fn = (float)n;
  F2 m;
  m.hi = ss.hi / fn;
  m.lo = (fmaf(-m.hi, fn, ss.hi) + ss.lo) / fn;  // residual of the division
  {
    float s, e;
    two_sum(m.hi, eps, s, e);
    e += m.lo;
    m.hi = s + e;
    m.lo = e - (m.hi - s);
  }
  const float y = rsqrtf(m.hi);
  const float t = y * y, te = fmaf(y, y, -t);           // y^2 = t + te exactly
  const float u = m.hi * t, ue = fmaf(m.hi, t, -u);    // m.hi * t = u + ue exactly
  // 1 - m y^2, with u within a few ulps of 1 so 1 - u is exact
  const float r = ((1.0f - u) - ue) - (m.hi * te + m.lo * t);
  F2 out;
  const float c = 0.5f * y * r;
  out.hi = y + c;
  out.lo = c - (out.hi - y);
  return out;
}

// R(h * rs) to the model dtype from the float pair rs: the fp32 product p
// with its exact residual decides, only when p lands exactly on a rounding
// tie of the model dtype, which way the exact product lies.
template <typename Dt> __device__ __forceinline__ float mul_round(float h, F2 rs);
template <> __device__ __forceinline__ float mul_round<float>(float h, F2 rs) { return fmaf(h, rs.hi, h * rs.lo); }
// Branch-free (selects only), so that independent elements interleave.
template <> __device__ __forceinline__ float mul_round<__nv_bfloat16>(float h, F2 rs) {
  const float p = h * rs.hi;
  const uint32_t b = __float_as_uint(p);
  const float res = fmaf(h, rs.hi, -p) + h * rs.lo;  // exact product - p (to fp32 accuracy)
  // p halfway between two bf16 values: the residual's sign picks the side
  const uint32_t lo = b & 0xffff0000u;  // toward zero
  const float down = __uint_as_float(lo), up = __uint_as_float(lo + 0x10000u);  // up = away from zero
  const float side = ((res > 0.f) == (p > 0.f)) ? up : down;
  return ((b & 0xffffu) != 0x8000u || res == 0.f) ? rd<__nv_bfloat16>(p) : side;
}
// Qwen3 RMSNorm element with its two roundings: R(R(h * rs) * g).
template <typename Dt>
__device__ __forceinline__ float rms_apply2(float h, F2 rs, float g) {
  return rd<Dt>(mul_round<Dt>(h, rs) * g);
}

// N elements of the RMSNorm with its two roundings, o = R(R(h * rs) * g).
// bf16: the rounding of h * rs.hi decides unless that product sits exactly on
// a rounding tie (rare); only a group holding such a tie takes mul_round's
// exact path, so the common case is one product and one rounding per element
// (the same results as rms_apply2 element by element).
template <typename Dt, int N>
__device__ __forceinline__ void rms_apply2_v(const float* h, F2 rs, const float* g, float* o) {
  if constexpr (sizeof(Dt) == 2) {
    float p[N];
    bool tie = false;
#pragma unroll
    for (int e = 0; e < N; ++e) {
      p[e] = h[e] * rs.hi;
      tie |= (__float_as_uint(p[e]) & 0xffffu) == 0x8000u;
    }
    if (!tie) {
#pragma unroll
      for (int e = 0; e < N; ++e) o[e] = rd<Dt>(rd<Dt>(p[e]) * g[e]);
      return;
    }
  }
#pragma unroll
  for (int e = 0; e < N; ++e) o[e] = rms_apply2<Dt>(h[e], rs, g[e]);
}

// g * sigmoid(g) with the fast division (the result is rounded to the model
// dtype by every caller; the IEEE division's slow path is avoided for 0).
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + expf(-g)); }

}  // namespace q3
