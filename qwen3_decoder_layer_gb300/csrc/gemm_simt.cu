// CUDA-core tiled GEMM with fp32 accumulation: the strict fp32 path (the
// Backbone's fp32 mode needs true fp32 products, not TF32) and the general
// path for row counts and weight formats the tensor-core GEMM does not take.
// Grouped mode runs the sorted expert GEMMs of @mlx-bun/inference
// qwen3-moe.ts Qwen3SortedExperts: rows sorted by expert, one weight matrix
// per expert, output rows scattered back to (token, slot) order.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, THREADS = 256;

template <typename Dt, int WF>
__device__ __forceinline__ float load_w(const GemmArgs& a, const char* wbase, size_t row, int k) {
  if (WF == W_U8) {
    const uint8_t q = reinterpret_cast<const uint8_t*>(wbase)[row * a.K + k];
    const size_t gi = row * (size_t)(a.K / a.group) + k / a.group;
    const float s = __bfloat162float(static_cast<const bf16*>(a.scale)[gi]);
    const float b = __bfloat162float(static_cast<const bf16*>(a.bias)[gi]);
    return fmaf(s, (float)q, b);
  }
  return to_f(reinterpret_cast<const Dt*>(wbase)[row * a.K + k]);
}

template <typename Dt, int WF, int EPI>
__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(GemmArgs a) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float Cs[EPI == EPI_SWIGLU ? BM : 1][BN + 1];
  constexpr bool PAIR = (EPI == EPI_SWIGLU);
  constexpr int BNO = PAIR ? BN / 2 : BN;  // output columns per tile
  pdl_wait();
  pdl_launch();
  const int tid = threadIdx.x;
  int r_begin, r_end, grp = 0;
  if (a.tile_start) {
    const int mt = blockIdx.y;
    if (mt >= a.tile_start[a.n_groups]) return;
    int lo = 0, hi = a.n_groups - 1;  // last group with tile_start <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_start[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    grp = lo;
    r_begin = a.row_off[grp] + (mt - a.tile_start[grp]) * BM;
    r_end = min(r_begin + BM, a.row_off[grp] + a.row_cnt[grp]);
  } else {
    r_begin = blockIdx.y * BM;
    r_end = min(r_begin + BM, a.M);
  }
  const int n0 = blockIdx.x * BNO;
  const char* wbase = static_cast<const char*>(a.w);
  // group grp's matrix starts at weight row grp * (w_stride / K): rows (and the
  // int8 scale / bias rows) are counted across the stacked matrices
  const size_t grow0 = a.tile_start ? (size_t)grp * (size_t)(a.w_stride / a.K) : 0;
  const Dt* A = static_cast<const Dt*>(a.a);

  // loaders: A tile 64 x 16 and B tile 64 x 16, 4 elements per thread each
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  const int am = r_begin + lr;
  const bool a_ok = am < r_end;
  const size_t arow = a_ok ? (size_t)(a.a_rows ? a.a_rows[am] : am) : 0;
  int bn;  // weight row loaded by this thread
  bool b_ok;
  if (PAIR) {
    const int j = lr < BN / 2 ? n0 + lr : n0 + (lr - BN / 2);
    b_ok = j < a.N;
    bn = lr < BN / 2 ? j : a.N + j;
  } else {
    bn = n0 + lr;
    b_ok = bn < a.N;
  }

  const int ty = tid >> 4, tx = tid & 15;  // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += BK) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      As[lk + e][lr] = a_ok ? to_f(A[arow * a.lda + k0 + lk + e]) : 0.f;
      Bs[lk + e][lr] = b_ok ? load_w<Dt, WF>(a, wbase, grow0 + (size_t)bn, k0 + lk + e) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
    __syncthreads();
  }

  if (PAIR) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
    __syncthreads();
    for (int idx = tid; idx < BM * BNO; idx += THREADS) {
      const int i = idx / BNO, j = idx % BNO;
      const int m = r_begin + i, n = n0 + j;
      if (m >= r_end || n >= a.N) continue;
      const float g = rd<Dt>(Cs[i][j]), up = rd<Dt>(Cs[i][j + BN / 2]);
      const size_t orow = a.c_rows ? (size_t)a.c_rows[m] : (size_t)m;
      static_cast<Dt*>(a.out)[orow * a.ldo + n] = from_f<Dt>(rd<Dt>(silu_f(g)) * up);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = r_begin + ty * 4 + i;
    if (m >= r_end) continue;
    const size_t orow = a.c_rows ? (size_t)a.c_rows[m] : (size_t)m;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      const size_t o = orow * a.ldo + n;
      if (EPI == EPI_STORE) static_cast<Dt*>(a.out)[o] = from_f<Dt>(acc[i][j]);
      else if (EPI == EPI_STORE_F32) static_cast<float*>(a.out)[o] = acc[i][j];
      else if (EPI == EPI_STORE_RF32) static_cast<float*>(a.out)[o] = rd<Dt>(acc[i][j]);
      else {  // residual
        Dt* p = static_cast<Dt*>(a.out) + o;
        *p = from_f<Dt>(to_f(*p) + rd<Dt>(acc[i][j]));
      }
    }
  }
}

template <typename Dt, int WF>
cudaError_t launch_epi(const LaunchCtx& c, const GemmArgs& a) {
  const int bno = a.epilogue == EPI_SWIGLU ? BN / 2 : BN;
  const int gy = a.tile_start ? a.max_tiles : (a.M + BM - 1) / BM;
  const dim3 grid((a.N + bno - 1) / bno, gy), block(THREADS);
  if (gy == 0) return cudaSuccess;
  switch (a.epilogue) {
    case EPI_STORE: return launch_k(gemm_simt_kernel<Dt, WF, EPI_STORE>, grid, block, 0, c, a);
    case EPI_STORE_F32: return launch_k(gemm_simt_kernel<Dt, WF, EPI_STORE_F32>, grid, block, 0, c, a);
    case EPI_STORE_RF32: return launch_k(gemm_simt_kernel<Dt, WF, EPI_STORE_RF32>, grid, block, 0, c, a);
    case EPI_RESIDUAL: return launch_k(gemm_simt_kernel<Dt, WF, EPI_RESIDUAL>, grid, block, 0, c, a);
    case EPI_SWIGLU: return launch_k(gemm_simt_kernel<Dt, WF, EPI_SWIGLU>, grid, block, 0, c, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_simt_tile_m() { return BM; }

cudaError_t launch_gemm_simt(const LaunchCtx& c, int dt, int wfmt, const GemmArgs& a) {
  if (a.K % BK) return cudaErrorInvalidValue;
  if (dt == DT_BF16) {
    if (wfmt == W_U8) return launch_epi<bf16, W_U8>(c, a);
    return launch_epi<bf16, W_DT>(c, a);
  }
  if (wfmt == W_U8) return launch_epi<float, W_U8>(c, a);
  return launch_epi<float, W_DT>(c, a);
}

}  // namespace q3
