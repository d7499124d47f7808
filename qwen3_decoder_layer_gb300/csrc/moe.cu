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

namespace {

// Router logits of many rows: logits[t, e] = sum_k y[t, k] W[e, k] in fp32,
// stored unrounded (the products of two bf16 values are exact in fp32; only
// the additions round).  K is cut into at most 8 fixed ranges (by K alone);
// each output is one fused multiply-add chain per range in k order, and the
// range sums are added in range order, however many blocks share the work, so
// the result is the same bits with or without a split.  A block computes a
// 32-row x 128-expert tile over a run of ranges: chunks of 32 k staged in
// shared memory as fp32 (rows, resp. experts, contiguous for each k), each
// thread owns a 4 x 4 block of outputs.  Split tiles store one partial per
// range; the last block of the tile to finish adds them.
constexpr int RL_BM = 32, RL_BE = 128, RL_BK = 32, RL_THREADS = 256;

template <typename Dt>
__global__ void __launch_bounds__(RL_THREADS) router_logits_kernel(RouterLogitsArgs a, int splits, int cpr, int nranges,
                                                                  int rpb) {
  constexpr int V = Vec16<Dt>::N;  // elements per 16-byte vector
  __shared__ __align__(16) float ys[RL_BK][RL_BM];
  __shared__ __align__(16) float ws[RL_BK][RL_BE];
  __shared__ int s_last;
  pdl_wait();
  pdl_launch();
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int tiles_e = (a.E + RL_BE - 1) / RL_BE;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int r0 = (tile / tiles_e) * RL_BM, e0 = (tile % tiles_e) * RL_BE;
  const int nchunks = a.K / RL_BK;
  const int rb = split * rpb, re = min(nranges, rb + rpb);  // this block's ranges
  const int c0 = rb * cpr, c1 = min(nchunks, re * cpr);
  // staging roles: experts e0 + (tid & 127), 16 k from (tid >> 7) * 16; rows
  // r0 + (tid & 31), 8 k from (tid >> 5) * 8 (threads 0..127)
  const int we = e0 + (tid & 127), wk = (tid >> 7) * 16;
  const int yr = r0 + (tid & 31), yk = (tid >> 5) * 8;
  const Dt* wsrc = static_cast<const Dt*>(a.w) + (size_t)min(we, a.E - 1) * a.K + wk;
  const Dt* ysrc = static_cast<const Dt*>(a.y) + (size_t)min(yr, a.M - 1) * a.ldy + yk;
  const bool wlive = we < a.E, ylive = tid < 128 && yr < a.M;
  uint4 wq[16 / V], yq[8 / V];
  auto fetch = [&](int ch) {
#pragma unroll
    for (int i = 0; i < 16 / V; ++i) wq[i] = wlive ? ld16(wsrc + (size_t)ch * RL_BK + i * V) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < 8 / V; ++i) yq[i] = ylive ? ld16(ysrc + (size_t)ch * RL_BK + i * V) : make_uint4(0u, 0u, 0u, 0u);
  };
  auto stage = [&]() {
#pragma unroll
    for (int i = 0; i < 16 / V; ++i) {
      float f[V];
      Vec16<Dt>::unpack(wq[i], f);
#pragma unroll
      for (int j = 0; j < V; ++j) ws[wk + i * V + j][tid & 127] = f[j];
    }
    if (tid < 128) {
#pragma unroll
      for (int i = 0; i < 8 / V; ++i) {
        float f[V];
        Vec16<Dt>::unpack(yq[i], f);
#pragma unroll
        for (int j = 0; j < V; ++j) ys[yk + i * V + j][tid & 31] = f[j];
      }
    }
  };
  const int ebase = e0 + 4 * tx;
  auto store_rows = [&](float* dst, int ld, const float (&v)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = r0 + 4 * ty + i;
      if (row >= a.M) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ebase + j < a.E) dst[(size_t)row * ld + ebase + j] = v[i][j];
    }
  };
  float acc[4][4], tot[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = tot[i][j] = 0.f;
  if (c0 < c1) fetch(c0);
  for (int ch = c0; ch < c1; ++ch) {
    __syncthreads();  // the previous chunk is consumed
    stage();
    __syncthreads();
    if (ch + 1 < c1) fetch(ch + 1);  // in flight while this chunk computes
#pragma unroll 8
    for (int k = 0; k < RL_BK; ++k) {
      const float4 yv = *reinterpret_cast<const float4*>(&ys[k][4 * ty]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[k][4 * tx]);
      const float yy[4] = {yv.x, yv.y, yv.z, yv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(yy[i], ww[j], acc[i][j]);
    }
    if ((ch + 1) % cpr == 0 || ch + 1 == c1) {  // the end of range ch / cpr
      const int r = ch / cpr;
      if (splits == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) tot[i][j] = r == 0 ? acc[i][j] : tot[i][j] + acc[i][j];
      } else {
        store_rows(a.part + (size_t)r * a.M * a.E, a.E, acc);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    }
  }
  if (splits == 1) {
    store_rows(a.out, a.ldo, tot);
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.counters[tile], 1) == splits - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the tile's last block: the partials in range order
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = r0 + 4 * ty + i;
    if (row >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (ebase + j >= a.E) continue;
      float s = 0.f;
      for (int q = 0; q < nranges; ++q)
        s = q == 0 ? __ldcg(a.part + ((size_t)q * a.M + row) * a.E + ebase + j)
                   : s + __ldcg(a.part + ((size_t)q * a.M + row) * a.E + ebase + j);
      a.out[(size_t)row * a.ldo + ebase + j] = s;
    }
  }
  if (tid == 0) a.counters[tile] = 0;  // ready for the next call
}

}  // namespace

int router_logits_tiles(int M, int E) { return ((M + RL_BM - 1) / RL_BM) * ((E + RL_BE - 1) / RL_BE); }

bool router_logits_supported(int dt, int E, int K) {
  (void)dt;
  return E >= 1 && K % RL_BK == 0 && K >= RL_BK;
}

cudaError_t launch_router_logits(const LaunchCtx& c, int dt, const RouterLogitsArgs& a) {
  if (a.M < 1 || !router_logits_supported(dt, a.E, a.K) || (a.ldy % (dt == DT_BF16 ? 8 : 4)) ||
      (reinterpret_cast<uintptr_t>(a.y) & 15) || (reinterpret_cast<uintptr_t>(a.w) & 15))
    return cudaErrorInvalidValue;
  const int tiles = router_logits_tiles(a.M, a.E), nchunks = a.K / RL_BK;
  // the fixed k ranges (a function of K only), at most kRouterMaxSplits
  const int cpr = (nchunks + kRouterMaxSplits - 1) / kRouterMaxSplits;
  const int nranges = (nchunks + cpr - 1) / cpr;
  // blocks per tile: about two blocks per SM when partials have room
  int splits = 1;
  if (a.part && a.counters && a.max_splits >= nranges)
    splits = std::min(nranges, std::max(1, (2 * c.num_sms + tiles - 1) / tiles));
  const int rpb = (nranges + splits - 1) / splits;
  splits = (nranges + rpb - 1) / rpb;
  const dim3 grid(tiles, splits), block(RL_THREADS);
  if (dt == DT_BF16) return launch_k(router_logits_kernel<bf16>, grid, block, 0, c, a, splits, cpr, nranges, rpb);
  return launch_k(router_logits_kernel<float>, grid, block, 0, c, a, splits, cpr, nranges, rpb);
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
