// Skinny GEMM for 5..64 activation rows: the linears of a batched decode step
// (maya2_mlx/backbone.py, Backbone.forward run on one new row per sequence)
// when the weights are affine int8 (dequantised in fp32 inside the kernel, as
// the scale * q + bias form of the int8 export prescribes) or the stack runs
// in fp32.
//
// C[M, N] = A[M, K] . W[N, K]^T.  A tile covers all M rows (32 or 64) and 64
// output columns (for SiLU * up: 64 gate rows and the 64 matching up rows);
// the K range is split over several CTAs so that the grid fills the GPU even
// for N = 2048.  Each CTA streams its weight slice once, dequantises it into
// shared memory as fp32, and accumulates a 2x4 or 4x4 (x2 for gate|up)
// register tile per thread in fp32.  With one K split the epilogue runs from
// registers; otherwise each split stores its partial tile to its own slice of
// an fp32 workspace and the last CTA of a tile (an atomic counter) adds the
// slices in split order -- the result does not depend on which CTA finishes
// when -- and applies the epilogue (rounding, residual add or SiLU * up),
// leaving the counter at zero for the next call.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int SK_BN = 64, SK_BK = 32, SK_THREADS = 256, SK_MAX_SPLIT = 8;

template <typename Dt, int WF, int MT, int EPI>
__global__ void __launch_bounds__(SK_THREADS) gemm_skinny_kernel(SkinnyArgs a) {
  constexpr bool PAIR = EPI == EPI_SWIGLU;
  constexpr int TM = MT / 16;  // rows per thread
  __shared__ float As[SK_BK][MT + 4];
  __shared__ float Ws[SK_BK][2 * SK_BN + 4];
  __shared__ int s_last;
  pdl_wait();
  pdl_launch();
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int n0 = blockIdx.x * SK_BN;
  const int ks = blockIdx.y;
  const int kt0 = ks * a.ktiles_per_split, kt1 = min(a.K / SK_BK, kt0 + a.ktiles_per_split);
  const Dt* A = static_cast<const Dt*>(a.a);
  float acc[TM][4], acc2[PAIR ? TM : 1][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[i][j] = 0.f;
      if (PAIR) acc2[PAIR ? i : 0][j] = 0.f;
    }
  // Global -> registers for one k-tile (issued a tile ahead), registers ->
  // shared memory (dequantised, fp32, transposed) for the current one.
  constexpr int AV = Vec16<Dt>::N;
  constexpr int EPV = WF == W_U8 ? 16 : (int)(16 / sizeof(Dt));
  constexpr int VPR = SK_BK / EPV;                                  // 16-byte weight vectors per tile row
  constexpr int NW = ((PAIR ? 2 : 1) * SK_BN * VPR + SK_THREADS - 1) / SK_THREADS;  // per thread
  constexpr int NA = (MT * SK_BK / AV + SK_THREADS - 1) / SK_THREADS;
  const size_t wb = WF == W_U8 ? 1 : sizeof(Dt);
  uint4 wq[NW], aq[NA];
  float wsc[NW], wbi[NW];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int idx = tid + q * SK_THREADS;
      const int r = idx / VPR, v = idx % VPR;
      const int n = PAIR ? (r < SK_BN ? n0 + r : n0 + r - SK_BN) : n0 + r;
      wq[q] = make_uint4(0, 0, 0, 0);
      wsc[q] = wbi[q] = 0.f;
      if (r < (PAIR ? 2 : 1) * SK_BN && n < a.N) {
        const size_t row = PAIR && r >= SK_BN ? (size_t)a.N + n : (size_t)n;
        const int k = k0 + v * EPV;
        wq[q] = ld_stream(static_cast<const char*>(a.w) + (row * a.K + k) * wb);
        if (WF == W_U8) {
          const size_t gi = row * (size_t)(a.K / a.group) + k / a.group;
          wsc[q] = __bfloat162float(static_cast<const bf16*>(a.scale)[gi]);
          wbi[q] = __bfloat162float(static_cast<const bf16*>(a.bias)[gi]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NA; ++q) {
      const int idx = tid + q * SK_THREADS;
      const int m = idx / (SK_BK / AV), v = idx % (SK_BK / AV);
      aq[q] = make_uint4(0, 0, 0, 0);
      if (idx < MT * SK_BK / AV && m < a.M) aq[q] = ld16(A + (size_t)m * a.lda + k0 + v * AV);
    }
  };
  auto commit = [&]() {
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int idx = tid + q * SK_THREADS;
      const int r = idx / VPR, v = idx % VPR;
      if (r < (PAIR ? 2 : 1) * SK_BN) {
        float w[EPV];
        if (WF == W_U8) {
          const uint32_t u[4] = {wq[q].x, wq[q].y, wq[q].z, wq[q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) w[4 * i + j] = fmaf(wsc[q], (float)((u[i] >> (8 * j)) & 0xffu), wbi[q]);
        } else {
          Vec16<Dt>::unpack(wq[q], w);
        }
#pragma unroll
        for (int e = 0; e < EPV; ++e) Ws[v * EPV + e][r] = w[e];
      }
    }
#pragma unroll
    for (int q = 0; q < NA; ++q) {
      const int idx = tid + q * SK_THREADS;
      if (idx < MT * SK_BK / AV) {
        const int m = idx / (SK_BK / AV), v = idx % (SK_BK / AV);
        float x[AV];
        Vec16<Dt>::unpack(aq[q], x);
#pragma unroll
        for (int e = 0; e < AV; ++e) As[v * AV + e][m] = x[e];
      }
    }
  };
  if (kt0 < kt1) fetch(kt0 * SK_BK);
  for (int kt = kt0; kt < kt1; ++kt) {
    commit();
    __syncthreads();
    if (kt + 1 < kt1) fetch((kt + 1) * SK_BK);  // in flight during this tile's FMAs
#pragma unroll 8
    for (int kk = 0; kk < SK_BK; ++kk) {
      float ar[TM];
      if (TM == 4) {
        const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
        ar[0] = av.x; ar[TM > 1 ? 1 : 0] = av.y; ar[TM > 2 ? 2 : 0] = av.z; ar[TM > 3 ? 3 : 0] = av.w;
      } else {
        const float2 av = *reinterpret_cast<const float2*>(&As[kk][ty * 2]);
        ar[0] = av.x; ar[TM > 1 ? 1 : 0] = av.y;
      }
      const float4 bv = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
      if (PAIR) {
        const float4 uv = *reinterpret_cast<const float4*>(&Ws[kk][SK_BN + tx * 4]);
        const float ur[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc2[PAIR ? i : 0][j] = fmaf(ar[i], ur[j], acc2[PAIR ? i : 0][j]);
      }
    }
    __syncthreads();
  }

  // epilogue on (m, n) with the full sums g (and u for SiLU * up)
  auto finish = [&](int m, int n, float g, float u) {
    const size_t o = (size_t)m * a.ldo + n;
    if (EPI == EPI_STORE) static_cast<Dt*>(a.out)[o] = from_f<Dt>(g);
    else if (EPI == EPI_STORE_F32) static_cast<float*>(a.out)[o] = g;
    else if (EPI == EPI_RESIDUAL) {
      Dt* p = static_cast<Dt*>(a.out) + o;
      *p = from_f<Dt>(to_f(*p) + rd<Dt>(g));
    } else {
      const float gg = rd<Dt>(g), uu = rd<Dt>(u);
      static_cast<Dt*>(a.out)[o] = from_f<Dt>(rd<Dt>(silu_f(gg)) * uu);
    }
  };
  const int ldw = PAIR ? 2 * a.N : a.N;  // workspace row pitch (gate sums, then up sums)
  const size_t slice = (size_t)a.M * ldw;  // floats per split
  if (gridDim.y == 1) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int m = ty * TM + i, n = n0 + tx * 4 + j;
        if (m < a.M && n < a.N) finish(m, n, acc[i][j], PAIR ? acc2[PAIR ? i : 0][j] : 0.f);
      }
    return;
  }
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = ty * TM + i, n = n0 + tx * 4 + j;
      if (m < a.M && n < a.N) {
        float* w = a.ws + ks * slice + (size_t)m * ldw + n;
        __stcg(w, acc[i][j]);
        if (PAIR) __stcg(w + a.N, acc2[PAIR ? i : 0][j]);
      }
    }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counters + blockIdx.x, 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < a.M * SK_BN; idx += SK_THREADS) {
    const int m = idx / SK_BN, n = n0 + idx % SK_BN;
    if (n >= a.N) continue;
    const float* pg = a.ws + (size_t)m * ldw + n;
    float g = 0.f, u = 0.f;
    for (int k = 0; k < (int)gridDim.y; ++k) {
      g += __ldcg(pg + k * slice);
      if (PAIR) u += __ldcg(pg + k * slice + a.N);
    }
    finish(m, n, g, u);
  }
  if (tid == 0) a.counters[blockIdx.x] = 0;
}

template <typename Dt, int WF, int MT>
cudaError_t sk_epi(const LaunchCtx& c, const SkinnyArgs& a, dim3 grid) {
  switch (a.epilogue) {
    case EPI_STORE: return launch_k(gemm_skinny_kernel<Dt, WF, MT, EPI_STORE>, grid, dim3(SK_THREADS), 0, c, a);
    case EPI_STORE_F32: return launch_k(gemm_skinny_kernel<Dt, WF, MT, EPI_STORE_F32>, grid, dim3(SK_THREADS), 0, c, a);
    case EPI_RESIDUAL: return launch_k(gemm_skinny_kernel<Dt, WF, MT, EPI_RESIDUAL>, grid, dim3(SK_THREADS), 0, c, a);
    case EPI_SWIGLU: return launch_k(gemm_skinny_kernel<Dt, WF, MT, EPI_SWIGLU>, grid, dim3(SK_THREADS), 0, c, a);
  }
  return cudaErrorInvalidValue;
}

template <typename Dt, int WF>
cudaError_t sk_mt(const LaunchCtx& c, const SkinnyArgs& a, dim3 grid) {
  return a.M <= 32 ? sk_epi<Dt, WF, 32>(c, a, grid) : sk_epi<Dt, WF, 64>(c, a, grid);
}

}  // namespace

bool gemm_skinny_supported(int M, int N, int K) { return M >= 1 && M <= 64 && N >= 1 && K % SK_BK == 0; }

size_t gemm_skinny_ws_floats(int M, int N, int epilogue) {
  return (size_t)SK_MAX_SPLIT * M * (epilogue == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N);
}
int gemm_skinny_tiles(int N) { return (N + SK_BN - 1) / SK_BN; }

cudaError_t launch_gemm_skinny(const LaunchCtx& c, int dt, int wfmt, SkinnyArgs a) {
  if (!gemm_skinny_supported(a.M, a.N, a.K)) return cudaErrorInvalidValue;
  const int tiles = gemm_skinny_tiles(a.N), ktiles = a.K / SK_BK;
  // split K so that the grid holds about two CTAs per SM
  int split = std::max(1, std::min({ktiles, (2 * c.num_sms + tiles - 1) / tiles, SK_MAX_SPLIT}));
  a.ktiles_per_split = (ktiles + split - 1) / split;
  split = (ktiles + a.ktiles_per_split - 1) / a.ktiles_per_split;
  if (split > 1 && (!a.ws || !a.counters)) return cudaErrorInvalidValue;
  const dim3 grid(tiles, split);
  if (dt == DT_BF16) return wfmt == W_U8 ? sk_mt<bf16, W_U8>(c, a, grid) : sk_mt<bf16, W_DT>(c, a, grid);
  return wfmt == W_U8 ? sk_mt<float, W_U8>(c, a, grid) : sk_mt<float, W_DT>(c, a, grid);
}

}  // namespace q3
