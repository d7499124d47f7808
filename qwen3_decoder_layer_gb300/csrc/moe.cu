// Qwen3-MoE router and token-by-expert permutation (@mlx-bun/inference
// qwen3-moe.ts: Qwen3MoeSparseMoeBlock.forward -- "precise" softmax over all
// experts, argpartition top-k, take_along_axis, renormalise when
// norm_topk_prob, weighted sum; Qwen3SortedExperts -- rows sorted by expert,
// gathered, projected, and put back with the inverse permutation).
#include <math_constants.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int kMaxEPerLane = 8;  // E <= 256

// One warp per token.  Expert e lives in lane e % 32, register e / 32.
// Top-k is taken on the fp32 logits (softmax is monotone), larger first,
// ties to the lower expert index; weights are the softmax probabilities of
// the chosen experts, divided by their sum when norm != 0.
__global__ void __launch_bounds__(256) router_topk_kernel(RouterArgs a) {
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const float* lg = a.logits + (size_t)t * a.E;
  float v[kMaxEPerLane];
  float m = -CUDART_INF_F;
#pragma unroll
  for (int r = 0; r < kMaxEPerLane; ++r) {
    const int e = r * 32 + lane;
    v[r] = e < a.E ? lg[e] : -CUDART_INF_F;
    m = fmaxf(m, v[r]);
  }
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < kMaxEPerLane; ++r)
    if (r * 32 + lane < a.E) s += expf(v[r] - m);
  s = warp_sum(s);
  uint32_t taken = 0;
  float wsum = 0.f, wmine = 0.f;
  int emine = 0;
  for (int sel = 0; sel < a.k; ++sel) {
    float bv = -CUDART_INF_F;
    int be = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < kMaxEPerLane; ++r) {
      const int e = r * 32 + lane;
      if (e < a.E && !(taken >> r & 1u) && (v[r] > bv || be == 0x7fffffff)) { bv = v[r]; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    const float p = expf(bv - m) / s;
    wsum += p;
    if (lane == sel) { wmine = p; emine = be; }
  }
  if (lane < a.k) {
    a.idx[(size_t)t * a.k + lane] = emine;
    a.w[(size_t)t * a.k + lane] = a.norm ? wmine / wsum : wmine;
    if (a.counts) atomicAdd(a.counts + emine, 1);
  }
}

// Single block, one thread per expert (E <= 256): exclusive prefix sums of
// the experts' row counts (sorted row offsets) and of their row tiles, by a
// warp-shuffle scan inside each warp and a scan of the warp totals.
__global__ void __launch_bounds__(256) moe_scan_kernel(MoeScanArgs a) {
  __shared__ int s_rows[8], s_tiles[8];
  pdl_wait();
  pdl_launch();
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int c = e < a.E ? a.counts[e] : 0;
  const int tl = (c + a.bm - 1) / a.bm;
  int rows = c, tiles = tl;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int r = __shfl_up_sync(0xffffffffu, rows, o), t = __shfl_up_sync(0xffffffffu, tiles, o);
    if (lane >= o) { rows += r; tiles += t; }
  }
  if (lane == 31) { s_rows[warp] = rows; s_tiles[warp] = tiles; }
  __syncthreads();
  int rbase = 0, tbase = 0;
  for (int w = 0; w < warp; ++w) { rbase += s_rows[w]; tbase += s_tiles[w]; }
  if (e < a.E) {
    a.row_off[e] = rbase + rows - c;
    a.row_cnt[e] = c;
    a.tile_start[e] = tbase + tiles - tl;
    a.cursor[e] = 0;
    a.counts[e] = 0;
    if (e == a.E - 1) a.tile_start[a.E] = tbase + tiles;
  }
}

__global__ void moe_scatter_kernel(MoeScatterArgs a) {
  pdl_wait();
  pdl_launch();
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= a.T * a.k) return;
  const int e = a.idx[f];
  const int pos = a.row_off[e] + atomicAdd(a.cursor + e, 1);
  a.sorted_tok[pos] = f / a.k;
  a.sorted_src[pos] = f;
}

// One thread per output element (blocks tile the row); with the residual add,
// each block adds its share of the row's sum of squares (fp64 atomic; the
// slot is zero at the start of the step).
template <typename Dt>
__global__ void __launch_bounds__(256) moe_combine_kernel(MoeCombineArgs a) {
  __shared__ float red[64];
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.y, n = blockIdx.x * blockDim.x + threadIdx.x;
  const Dt* z = static_cast<const Dt*>(a.z) + (size_t)t * a.k * a.hidden;
  const float* w = a.w + (size_t)t * a.k;
  F2 ss = {0.f, 0.f};
  if (n < a.hidden) {
    float acc = 0.f;
    for (int i = 0; i < a.k; ++i) acc = fmaf(w[i], to_f(z[(size_t)i * a.hidden + n]), acc);
    const float pend = rd<Dt>(acc);
    if (a.h) {
      Dt* h = static_cast<Dt*>(a.h) + (size_t)t * a.hidden;
      const float hn = rd<Dt>(to_f(h[n]) + pend);
      h[n] = from_f<Dt>(hn);
      f2_add_sq(ss, hn);
    } else {
      static_cast<Dt*>(a.out)[(size_t)t * a.hidden + n] = from_f<Dt>(pend);
    }
  }
  if (a.h) {
    ss = f2_block_sum(ss, red);
    if (threadIdx.x == 0) atomicAdd(a.sumsq_out + t, (double)ss.hi + (double)ss.lo);
  }
}

}  // namespace

// Router logits of many rows: logits[t, e] = sum_k y[t, k] W[e, k], one
// fp32 fused multiply-add chain per output in k order (the order of the
// CUDA-core GEMM), stored unrounded.  A block takes 8 rows, staged in shared
// memory, and every expert: warp w the experts 16w .. 16w + 15, lane (row
// pair, expert pair) four outputs, so each 16-byte weight load feeds 2 rows
// and each staged row load 2 experts.  (More than 256 experts: blocks along y.)
template <typename Dt>
__global__ void __launch_bounds__(512) router_logits_kernel(GemmArgs a) {
  extern __shared__ __align__(16) uint8_t rl_smem[];
  constexpr int V = Vec16<Dt>::N;
  Dt* ys = reinterpret_cast<Dt*>(rl_smem);  // [8][K + V]: rows padded by 16 bytes (no bank conflicts)
  pdl_wait();
  pdl_launch();
  const int K = a.K, E = a.N, r0 = blockIdx.x * 8;
  const int nv = K / V, pitch = K + V;
  for (int c = threadIdx.x; c < 8 * nv; c += blockDim.x) {
    const int r = c / nv, v = c % nv;
    const uint4 val = r0 + r < a.M ? ld16(static_cast<const Dt*>(a.a) + (size_t)(r0 + r) * a.lda + (size_t)v * V)
                                   : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(ys + (size_t)r * pitch + (size_t)v * V) = val;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rp = lane >> 3, e0 = blockIdx.y * 256 + warp * 16 + (lane & 7) * 2;  // 256 experts per block
  if (e0 >= E) return;
  const Dt* w0 = static_cast<const Dt*>(a.w) + (size_t)e0 * K;
  const Dt* w1 = e0 + 1 < E ? w0 + K : w0;
  const Dt* y0 = ys + (size_t)(2 * rp) * pitch;
  const Dt* y1 = y0 + pitch;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  // the weight vectors of the next PF steps are in flight while a step computes
  // (the chains stay in k order)
  constexpr int PF = 4;
  uint4 qa[PF], qb[PF];
#pragma unroll
  for (int p = 0; p < PF; ++p) {
    if (p * V < K) {
      qa[p] = ld16(w0 + p * V);
      qb[p] = ld16(w1 + p * V);
    }
  }
  for (int k = 0; k < K; k += PF * V) {
#pragma unroll
    for (int p = 0; p < PF; ++p) {
      const int kk = k + p * V;
      if (kk >= K) break;
      float wa[V], wb[V], ya[V], yb[V];
      Vec16<Dt>::unpack(qa[p], wa);
      Vec16<Dt>::unpack(qb[p], wb);
      if (kk + PF * V < K) {
        qa[p] = ld16(w0 + kk + PF * V);
        qb[p] = ld16(w1 + kk + PF * V);
      }
      Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(y0 + kk), ya);
      Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(y1 + kk), yb);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        acc[0][0] = fmaf(ya[e], wa[e], acc[0][0]);
        acc[0][1] = fmaf(ya[e], wb[e], acc[0][1]);
        acc[1][0] = fmaf(yb[e], wa[e], acc[1][0]);
        acc[1][1] = fmaf(yb[e], wb[e], acc[1][1]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = r0 + 2 * rp + i;
    if (row >= a.M) continue;
    float* o = static_cast<float*>(a.out) + (size_t)row * a.ldo + e0;
    o[0] = acc[i][0];
    if (e0 + 1 < E) o[1] = acc[i][1];
  }
}

bool router_logits_supported(int dt, int E, int K) {
  const int V = dt == DT_BF16 ? 8 : 4;
  const size_t smem = (size_t)8 * (K + V) * (dt == DT_BF16 ? 2 : 4);
  return E >= 2 && E % 2 == 0 && E <= 512 && K % V == 0 && smem <= 200 * 1024;
}

cudaError_t launch_router_logits(const LaunchCtx& c, int dt, const GemmArgs& a) {
  if (!router_logits_supported(dt, a.N, a.K) || (a.lda % (dt == DT_BF16 ? 8 : 4)) ||
      (reinterpret_cast<uintptr_t>(a.a) & 15) || (reinterpret_cast<uintptr_t>(a.w) & 15))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)8 * (a.K + (dt == DT_BF16 ? 8 : 4)) * (dt == DT_BF16 ? 2 : 4);
  const dim3 grid((a.M + 7) / 8, (a.N + 255) / 256), block(std::min((a.N + 15) / 16, 16) * 32);
  // (the attribute is set once per kernel: to the largest size this launcher takes)
  if (dt == DT_BF16) {
    cudaError_t e = set_max_smem((const void*)router_logits_kernel<bf16>, 200 * 1024);
    if (e != cudaSuccess) return e;
    return launch_k(router_logits_kernel<bf16>, grid, block, smem, c, a);
  }
  cudaError_t e = set_max_smem((const void*)router_logits_kernel<float>, 200 * 1024);
  if (e != cudaSuccess) return e;
  return launch_k(router_logits_kernel<float>, grid, block, smem, c, a);
}

cudaError_t launch_router_topk(const LaunchCtx& c, const RouterArgs& a) {
  if (a.E > 32 * kMaxEPerLane || a.k > 32 || a.k > a.E) return cudaErrorInvalidValue;
  return launch_k(router_topk_kernel, dim3((a.T + 7) / 8), dim3(256), 0, c, a);
}

// out[r] = x[rows[r]], 16-byte vectors.
template <typename Dt>
__global__ void __launch_bounds__(256) moe_gather_kernel(MoeGatherArgs a) {
  constexpr int V = Vec16<Dt>::N;
  pdl_wait();
  pdl_launch();
  const int vpr = a.K / V;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)a.n * vpr;
       i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / vpr), v = (int)(i % vpr);
    const Dt* src = static_cast<const Dt*>(a.x) + (size_t)a.rows[r] * a.K + (size_t)v * V;
    *reinterpret_cast<uint4*>(static_cast<Dt*>(a.out) + (size_t)r * a.K + (size_t)v * V) = ld16(src);
  }
}

cudaError_t launch_moe_gather(const LaunchCtx& c, int dt, const MoeGatherArgs& a) {
  const size_t vec = (size_t)a.n * a.K / (dt == DT_BF16 ? 8 : 4);
  const int grid = (int)std::min<size_t>((vec + 255) / 256, (size_t)c.num_sms * 8);
  if (grid < 1) return cudaSuccess;
  if (dt == DT_BF16) return launch_k(moe_gather_kernel<bf16>, dim3(grid), dim3(256), 0, c, a);
  return launch_k(moe_gather_kernel<float>, dim3(grid), dim3(256), 0, c, a);
}

cudaError_t launch_moe_scan(const LaunchCtx& c, const MoeScanArgs& a) {
  if (a.E > 256) return cudaErrorInvalidValue;
  return launch_k(moe_scan_kernel, dim3(1), dim3(256), 0, c, a);
}

cudaError_t launch_moe_scatter(const LaunchCtx& c, const MoeScatterArgs& a) {
  const int n = a.T * a.k;
  return launch_k(moe_scatter_kernel, dim3((n + 255) / 256), dim3(256), 0, c, a);
}

cudaError_t launch_moe_combine(const LaunchCtx& c, int dt, const MoeCombineArgs& a) {
  const dim3 grid((a.hidden + 255) / 256, a.T);
  if (dt == DT_BF16) return launch_k(moe_combine_kernel<bf16>, grid, dim3(256), 0, c, a);
  return launch_k(moe_combine_kernel<float>, grid, dim3(256), 0, c, a);
}

}  // namespace q3
