// Skinny GEMMs for 5..64 activation rows: the linears of a batched decode step
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

// ---------------------------------------------------------------- int8 weights, up to 32 rows
// Weight-streaming variant for affine int8 weights, bf16 activations and at
// most MT (16 or 32) activation rows -- the batched decode step of an int8
// stack when tensor cores are switched off (the tensor-core form is
// gemm_w8_tc.cu).  Each lane owns four weight rows (SiLU * up: gate rows n, n + 32 and
// the matching up rows; otherwise rows n + 32 r of a 128-row tile) and
// dequantises them in registers straight from global memory (scale * q + bias
// in fp32, the same single-rounding form as above).  The activation rows are
// staged once per CTA in shared memory as fp32 [k][m] and read as warp-wide
// broadcasts; a warp takes 16 of them, so each 16-byte shared-memory load
// feeds 16 FMAs per lane -- four wavefronts per 16 FMA instructions, which
// keeps the shared-memory pipe level with the FMA pipe -- and no cross-lane
// reduction is needed.  The CTA's warps split the K range (and the two token
// halves) and add their partials in a fixed order through shared memory; K
// splits over CTAs go through the workspace and the last CTA of a tile adds
// them in split order, as above.
constexpr int W8_WARPS = 8, W8_THREADS = W8_WARPS * 32;
constexpr int W8_KC = 768;         // K per CTA at most (the staged activation slice)
constexpr int W8_MAX_SPLIT = 16;   // the workspace holds SK_MAX_SPLIT x 64 rows = 16 x 32
constexpr int W8_R = 4;            // weight rows per lane
constexpr int W8_MW = 16;          // activation rows per warp

__device__ __forceinline__ float u8_to_f(uint32_t word, int byte) {
  // 2^23 + q as a float, minus 2^23: exact for q in [0, 255]
  return __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7540u | (unsigned)byte)) - 8388608.f;
}

template <int MT>
__host__ __device__ constexpr size_t w8_smem_bytes() {
  return (size_t)(W8_KC * MT > W8_WARPS * W8_R * W8_MW * 32 ? W8_KC * MT : W8_WARPS * W8_R * W8_MW * 32) *
         sizeof(float);
}

template <int MT, int EPI>
__global__ void __launch_bounds__(W8_THREADS, 2) gemm_w8_kernel(SkinnyArgs a) {
  constexpr bool PAIR = EPI == EPI_SWIGLU;
  constexpr int TN = PAIR ? 64 : 128;      // output columns per tile
  constexpr int TH = MT / W8_MW;           // token halves
  constexpr int KP = W8_WARPS / TH;        // K parts per token half
  extern __shared__ __align__(16) float w8s[];  // As[k][MT] for the CTA's K range; then warp partials
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int th = warp % TH, kp = warp / TH;
  const int c0 = blockIdx.x * TN;  // first output column of the tile
  // this lane's weight rows; row r of the lane is output column col(r) (+ N for up rows)
  size_t wrow[W8_R];
  bool live[W8_R];
#pragma unroll
  for (int r = 0; r < W8_R; ++r) {
    const int col = PAIR ? c0 + (r & 1) * 32 + lane : c0 + r * 32 + lane;
    live[r] = col < a.N;
    wrow[r] = (size_t)col + (PAIR && r >= 2 ? (size_t)a.N : 0);
  }
  const int nsteps = a.K / 32, spc = a.ktiles_per_split;
  const int s0 = blockIdx.y * spc, s1 = min(nsteps, s0 + spc);
  const int kbase = s0 * 32;
  // this warp's half-steps (16 k each) of the CTA's range
  const int nh = 2 * (s1 - s0);
  const int h0 = 2 * s0 + (nh * kp) / KP, h1 = 2 * s0 + (nh * (kp + 1)) / KP;
  const uint8_t* W = static_cast<const uint8_t*>(a.w);
  const unsigned short* SC = static_cast<const unsigned short*>(a.scale);
  const unsigned short* BI = static_cast<const unsigned short*>(a.bias);
  const int gpr = a.K / a.group;  // groups per row
  uint4 q[W8_R];
  uint32_t sb[W8_R] = {};  // bf16 scale (low half) and bias (high half) of the half-step's group
  // weights of half-step h; the group's scale and bias only where a group
  // starts (or at the warp's first half-step) -- fsb keeps them otherwise
  auto fetch = [&](int h, uint4 (&f)[W8_R], uint32_t (&fsb)[W8_R]) {
    const int k = h * 16, g = k / a.group;
    const bool new_group = h == h0 || k % a.group == 0;
#pragma unroll
    for (int r = 0; r < W8_R; ++r) {
      if (live[r]) {
        f[r] = ld_stream(W + wrow[r] * a.K + k);
        if (new_group) fsb[r] = (uint32_t)SC[wrow[r] * gpr + g] | ((uint32_t)BI[wrow[r] * gpr + g] << 16);
      } else {
        f[r] = make_uint4(0, 0, 0, 0);
        fsb[r] = 0;
      }
    }
  };
  if (h0 < h1) fetch(h0, q, sb);  // weights do not depend on the previous kernel
  pdl_wait();
  pdl_launch();
  // stage the activation slice: As[k - kbase][m] = A[m][k] (rows >= M are zero); batches of
  // independent loads so that a thread waits for L2 once per batch
  {
    constexpr int SB = 8;
    const bf16* A = static_cast<const bf16*>(a.a);
    const int total = (s1 - s0) * 4 * MT;  // 8-element chunks of k, times MT rows
    for (int base = tid; base < total; base += W8_THREADS * SB) {
      uint4 v[SB];
#pragma unroll
      for (int u = 0; u < SB; ++u) {
        const int idx = base + u * W8_THREADS, m = idx % MT, c = idx / MT;
        v[u] = make_uint4(0, 0, 0, 0);
        if (idx < total && m < a.M) v[u] = ld16(A + (size_t)m * a.lda + kbase + c * 8);
      }
#pragma unroll
      for (int u = 0; u < SB; ++u) {
        const int idx = base + u * W8_THREADS, m = idx % MT, c = idx / MT;
        if (idx < total) {
          float x[8];
          Vec16<bf16>::unpack(v[u], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) w8s[(c * 8 + e) * MT + m] = x[e];
        }
      }
    }
  }
  __syncthreads();
  float acc[W8_R][W8_MW];
#pragma unroll
  for (int r = 0; r < W8_R; ++r)
#pragma unroll
    for (int m = 0; m < W8_MW; ++m) acc[r][m] = 0.f;
  for (int h = h0; h < h1; ++h) {
    uint4 c[W8_R];
    uint32_t csb[W8_R];
#pragma unroll
    for (int r = 0; r < W8_R; ++r) { c[r] = q[r]; csb[r] = sb[r]; }
    if (h + 1 < h1) fetch(h + 1, q, sb);  // in flight during this half-step
    float scl[W8_R], bia[W8_R];
#pragma unroll
    for (int r = 0; r < W8_R; ++r) {
      scl[r] = __uint_as_float(csb[r] << 16);
      bia[r] = __uint_as_float(csb[r] & 0xffff0000u);
    }
    const float* As = w8s + (size_t)(h * 16 - kbase) * MT + th * W8_MW;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float w[W8_R];
#pragma unroll
      for (int r = 0; r < W8_R; ++r) {
        const uint32_t word = kk < 4 ? c[r].x : kk < 8 ? c[r].y : kk < 12 ? c[r].z : c[r].w;
        w[r] = fmaf(scl[r], u8_to_f(word, kk & 3), bia[r]);
      }
      const float4* ap = reinterpret_cast<const float4*>(As + kk * MT);
#pragma unroll
      for (int j = 0; j < W8_MW / 4; ++j) {
        const float4 av = ap[j];
#pragma unroll
        for (int r = 0; r < W8_R; ++r) {
          acc[r][4 * j] = fmaf(w[r], av.x, acc[r][4 * j]);
          acc[r][4 * j + 1] = fmaf(w[r], av.y, acc[r][4 * j + 1]);
          acc[r][4 * j + 2] = fmaf(w[r], av.z, acc[r][4 * j + 2]);
          acc[r][4 * j + 3] = fmaf(w[r], av.w, acc[r][4 * j + 3]);
        }
      }
    }
  }
  // warp partials: red[kp][th][r][m][lane], added over kp in order
  __syncthreads();
  float* red = w8s;
#pragma unroll
  for (int r = 0; r < W8_R; ++r)
#pragma unroll
    for (int m = 0; m < W8_MW; ++m) red[(((kp * TH + th) * W8_R + r) * W8_MW + m) * 32 + lane] = acc[r][m];
  __syncthreads();
  // full sum of lane row r of lane l for activation row m
  auto csum = [&](int r, int m, int l) {
    const int t = m / W8_MW, mm = m % W8_MW;
    float v = 0.f;
#pragma unroll
    for (int p = 0; p < KP; ++p) v += red[(((p * TH + t) * W8_R + r) * W8_MW + mm) * 32 + l];
    return v;
  };
  auto finish = [&](int m, int col, float g, float u) {
    const size_t o = (size_t)m * a.ldo + col;
    if (EPI == EPI_STORE) static_cast<bf16*>(a.out)[o] = from_f<bf16>(g);
    else if (EPI == EPI_STORE_F32) static_cast<float*>(a.out)[o] = g;
    else if (EPI == EPI_RESIDUAL) {
      bf16* p = static_cast<bf16*>(a.out) + o;
      *p = from_f<bf16>(to_f(*p) + rd<bf16>(g));
    } else {
      const float gg = rd<bf16>(g), uu = rd<bf16>(u);
      static_cast<bf16*>(a.out)[o] = from_f<bf16>(rd<bf16>(silu_f(gg)) * uu);
    }
  };
  const int ldw = PAIR ? 2 * a.N : a.N;
  const size_t slice = (size_t)a.M * ldw;
  // tile column j (0 .. TN) of activation row m: lane j % 32, lane row j / 32 (pair: + 2 for up)
  if (gridDim.y == 1) {
    for (int idx = tid; idx < a.M * TN; idx += W8_THREADS) {
      const int m = idx / TN, j = idx % TN;
      if (c0 + j < a.N) finish(m, c0 + j, csum(j / 32, m, j % 32), PAIR ? csum(j / 32 + 2, m, j % 32) : 0.f);
    }
    return;
  }
  // this split's partial tile into its workspace slice (gate sums, then up sums)
  for (int idx = tid; idx < a.M * TN; idx += W8_THREADS) {
    const int m = idx / TN, j = idx % TN;
    if (c0 + j < a.N) {
      float* wsp = a.ws + blockIdx.y * slice + (size_t)m * ldw + c0 + j;
      __stcg(wsp, csum(j / 32, m, j % 32));
      if (PAIR) __stcg(wsp + a.N, csum(j / 32 + 2, m, j % 32));
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counters + blockIdx.x, 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < a.M * TN; idx += W8_THREADS) {
    const int m = idx / TN, col = c0 + idx % TN;
    if (col >= a.N) continue;
    const float* pg = a.ws + (size_t)m * ldw + col;
    float g = 0.f, u = 0.f;
    for (int k = 0; k < (int)gridDim.y; ++k) {
      g += __ldcg(pg + k * slice);
      if (PAIR) u += __ldcg(pg + k * slice + a.N);
    }
    finish(m, col, g, u);
  }
  if (tid == 0) a.counters[blockIdx.x] = 0;
}

template <int MT, int EPI>
cudaError_t w8_go(const LaunchCtx& c, const SkinnyArgs& a, dim3 grid) {
  constexpr size_t smem = w8_smem_bytes<MT>();
  const cudaError_t e = set_max_smem((const void*)gemm_w8_kernel<MT, EPI>, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(gemm_w8_kernel<MT, EPI>, grid, dim3(W8_THREADS), smem, c, a);
}

template <int MT>
cudaError_t w8_epi(const LaunchCtx& c, const SkinnyArgs& a, dim3 grid) {
  switch (a.epilogue) {
    case EPI_STORE: return w8_go<MT, EPI_STORE>(c, a, grid);
    case EPI_STORE_F32: return w8_go<MT, EPI_STORE_F32>(c, a, grid);
    case EPI_RESIDUAL: return w8_go<MT, EPI_RESIDUAL>(c, a, grid);
    case EPI_SWIGLU: return w8_go<MT, EPI_SWIGLU>(c, a, grid);
  }
  return cudaErrorInvalidValue;
}

// The int8 variant takes bf16 activations, at most 32 rows, K a multiple of
// 32 within W8_MAX_SPLIT CTA slices, and groups that are whole 16-k halves.
bool w8_supported(int dt, int wfmt, const SkinnyArgs& a) {
  return dt == DT_BF16 && wfmt == W_U8 && a.M >= 1 && a.M <= 32 && a.K % 32 == 0 && a.group % 16 == 0 &&
         a.K % a.group == 0 && a.K <= W8_KC * W8_MAX_SPLIT;
}

cudaError_t launch_w8(const LaunchCtx& c, SkinnyArgs a) {
  const bool pair = a.epilogue == EPI_SWIGLU;
  const int tn = pair ? 64 : 128, tiles = (a.N + tn - 1) / tn, nsteps = a.K / 32;
  // the fewest K splits (each within the staged slice) that fill whole waves
  // of two resident CTAs per SM best
  const int smin = (nsteps + W8_KC / 32 - 1) / (W8_KC / 32), slots = 2 * c.num_sms;
  int split = 0;
  double best = -1.0;
  for (int sp = smin; sp <= std::min(W8_MAX_SPLIT, nsteps); ++sp) {
    const int ctas = tiles * sp, waves = (ctas + slots - 1) / slots;
    const double util = (double)ctas / ((double)waves * slots);
    if (util > best + 1e-9) { best = util; split = sp; }
  }
  if (split == 0) return cudaErrorInvalidValue;
  a.ktiles_per_split = (nsteps + split - 1) / split;
  split = (nsteps + a.ktiles_per_split - 1) / a.ktiles_per_split;
  if (a.ktiles_per_split * 32 > W8_KC) return cudaErrorInvalidValue;
  if (split > 1 && (!a.ws || !a.counters)) return cudaErrorInvalidValue;
  const dim3 grid(tiles, split);
  return a.M <= 16 ? w8_epi<16>(c, a, grid) : w8_epi<32>(c, a, grid);
}

}  // namespace

bool gemm_skinny_supported(int M, int N, int K) { return M >= 1 && M <= 64 && N >= 1 && K % SK_BK == 0; }

size_t gemm_skinny_ws_floats(int M, int N, int epilogue) {
  return (size_t)SK_MAX_SPLIT * M * (epilogue == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N);
}
int gemm_skinny_tiles(int N) { return (N + SK_BN - 1) / SK_BN; }

cudaError_t launch_gemm_skinny(const LaunchCtx& c, int dt, int wfmt, SkinnyArgs a) {
  if (!gemm_skinny_supported(a.M, a.N, a.K)) return cudaErrorInvalidValue;
  if (w8_supported(dt, wfmt, a)) return launch_w8(c, a);
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
