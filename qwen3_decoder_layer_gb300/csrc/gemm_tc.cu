// Tensor-core GEMM for the prefill linears (maya2_mlx/backbone.py,
// Backbone.forward: the fused q|k|v, o_proj, fused gate|up with SiLU * up and
// down_proj products for T > 4 rows), bf16 in, fp32 accumulate, on sm_103a:
//
//   C[M, N] = A[M, K] . B[N, K]^T      (A: activations, B: nn.Linear weight; both K-major)
//
// A persistent grid (one CTA per SM) walks the 128 x 256 output tiles; each
// tile is computed with tcgen05.mma (cta_group::1, kind::f16, M = 128,
// N = 256, K = 16 per instruction) into one of two tensor-memory
// accumulators, so that the epilogue of a tile overlaps the MMAs of the next.  A 4-stage ring of 128 x 64 (A) and 256 x 64 (B) bf16 tiles
// is filled by 2-D TMA loads with 128-byte swizzle; mbarriers hand stages
// from the TMA warp to the MMA warp (full) and back (empty, signalled by
// tcgen05.commit).  Four epilogue warps read the accumulator with
// tcgen05.ld (warp q owns TMEM lanes 32q..32q+31, i.e. rows of the tile),
// apply the fused epilogue (rounding / residual add / SiLU * up) and store:
// each warp writes 64 output columns of its 32 rows into a swizzled
// shared-memory slab (lane = row) and reads it back transposed (8 lanes per
// row), so that every global load of the residual and every store covers
// whole 128-byte lines.
// For SiLU * up the B tile is two 128-row boxes: gate rows n0.. and up rows
// N + n0.., so TMEM columns 0..127 hold g and 128..255 hold u of the same
// output columns.
#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"

namespace q3 {

namespace {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_THREADS = 192;  // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr uint32_t TC_TMEM_COLS = 512;  // two 256-column accumulators
constexpr size_t TC_A_BYTES = (size_t)TC_BM * TC_BK * 2;   // 16 KB
constexpr size_t TC_B_BYTES = (size_t)TC_BN * TC_BK * 2;   // 32 KB
constexpr size_t TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
// epilogue staging: per epilogue warp 32 rows x 64 output columns (128 B per row)
constexpr size_t TC_STG_WARP = 32 * 128;
constexpr size_t TC_SMEM = TC_STAGES * TC_STAGE_BYTES + 256 /* barriers */ + 4 * TC_STG_WARP + 1024 /* align */;

using namespace tc;

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = idesc_bf16(TC_BM, TC_BN, false);

// Where tile t lives: A rows [m0, mlim) (the tile reads 128 rows from m0;
// rows from mlim on belong to the next group or lie outside and are not
// stored), output columns from n0, weight rows from brow (gate) / brow_up.
struct TileInfo {
  int m0, mlim, n0;
  int brow, brow_up;
};
template <bool GROUPED>
__device__ __forceinline__ TileInfo tile_of(const GemmTcArgs& a, int t, int tiles_m, int ncol) {
  TileInfo ti;
  const int mt = t % tiles_m, tn = t / tiles_m;
  ti.n0 = tn * ncol;
  if (!GROUPED) {
    ti.m0 = mt * TC_BM;
    ti.mlim = a.M;
    ti.brow = ti.n0;
    ti.brow_up = a.N + ti.n0;
  } else {
    int lo = 0, hi = a.n_groups - 1;  // last group with tile_start <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_start[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    ti.m0 = a.row_off[lo] + (mt - a.tile_start[lo]) * TC_BM;
    ti.mlim = a.row_off[lo] + a.row_cnt[lo];
    ti.brow = (int)(lo * a.w_group_rows) + ti.n0;
    ti.brow_up = (int)(lo * a.w_group_rows) + a.N + ti.n0;
  }
  return ti;
}

template <int EPI, bool GROUPED>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   GemmTcArgs a) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TC_STAGES * TC_STAGE_BYTES);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* acc_full = empty + TC_STAGES;  // [2] accumulator b holds a finished tile
  uint64_t* acc_empty = acc_full + 2;      // [2] the epilogue has read accumulator b
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncol = EPI == EPI_SWIGLU ? TC_BN / 2 : TC_BN;  // output columns of a tile
  const int nk = a.K / TC_BK;
  // tile t -> rows (t % tiles_m), columns (t / tiles_m): blocks running at the
  // same time share weight tiles in L2

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, TC_TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch();
  // grouped: the tile count comes from the routing scan of the previous kernel
  const int tiles_m = GROUPED ? a.tile_start[a.n_groups] : (a.M + TC_BM - 1) / TC_BM;
  const int tiles = tiles_m * (a.N / ncol);

  if (warp == 4) {
    if (lane == 0) {  // TMA producer: the k-blocks of this block's tiles, in order
      int q = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const TileInfo ti = tile_of<GROUPED>(a, t, tiles_m, ncol);
        for (int kt = 0; kt < nk; ++kt, ++q) {
          const int s = q % TC_STAGES;
          if (q >= TC_STAGES && !(ok = mbar_wait(&empty[s], (uint32_t)((q / TC_STAGES - 1) & 1), a.err, 3))) break;
          uint8_t* sa = smem + s * TC_STAGE_BYTES;
          uint8_t* sb = sa + TC_A_BYTES;
          mbar_expect_tx(&full[s], (uint32_t)TC_STAGE_BYTES);
          tma_load_2d(sa, &map_a, kt * TC_BK, ti.m0, &full[s]);
          if (EPI == EPI_SWIGLU) {
            tma_load_2d(sb, &map_b, kt * TC_BK, ti.brow, &full[s]);
            tma_load_2d(sb + TC_B_BYTES / 2, &map_b, kt * TC_BK, ti.brow_up, &full[s]);
          } else {
            tma_load_2d(sb, &map_b, kt * TC_BK, ti.brow, &full[s]);
          }
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {  // MMA issuer: tile i accumulates in TMEM columns (i & 1) * 256
      int q = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const int b = i & 1, use = i >> 1;
        if (use > 0 && !(ok = mbar_wait(&acc_empty[b], (uint32_t)((use - 1) & 1), a.err, 6))) break;
        fence_after();
        const uint32_t d = tmem + (uint32_t)(b * TC_BN);
        for (int kt = 0; kt < nk; ++kt, ++q) {
          const int s = q % TC_STAGES;
          if (!(ok = mbar_wait(&full[s], (uint32_t)((q / TC_STAGES) & 1), a.err, 4))) break;
          fence_after();
          const uint32_t sa = smem_u32(smem + s * TC_STAGE_BYTES);
          const uint32_t sb = sa + (uint32_t)TC_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            mma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), kIdesc, (kt | kk) != 0);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
    }
  } else {  // epilogue: warp q reads TMEM lanes 32q .. 32q + 31 = tile rows
    // staging slab of this warp: row r's 16-byte chunk j sits at chunk j ^ (r & 7)
    uint4* stg = reinterpret_cast<uint4*>(smem + TC_STAGES * TC_STAGE_BYTES + 256 + warp * TC_STG_WARP);
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int b = i & 1, use = i >> 1;
      const TileInfo ti = tile_of<GROUPED>(a, t, tiles_m, ncol);
      int okl = 1;  // lane 0 waits for the accumulator; the other lanes wait at the warp barrier
      if (lane == 0) okl = mbar_wait(&acc_full[b], (uint32_t)(use & 1), a.err, 5);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, okl, 0)) break;
      fence_after();
      const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * TC_BN);
      // the 8 rows this lane stores per 64-column slab: r = 4k + lane / 8, chunk lane % 8
      const int jr = lane & 7, r0 = lane >> 3;
      const int rbase = ti.m0 + warp * 32;
      for (int c = 0; c < ncol; c += 64) {
        // 1. this lane's row: 64 columns from tensor memory, rounded to bf16, into the slab
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float o[32];
          if (EPI == EPI_SWIGLU) {
            uint32_t g[32], u[32];
            tmem_ld32(tl + c + 32 * h, g);
            tmem_ld32(tl + TC_BN / 2 + c + 32 * h, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float gv = rd<bf16>(__uint_as_float(g[e])), uv = rd<bf16>(__uint_as_float(u[e]));
              o[e] = rd<bf16>(silu_f(gv)) * uv;
            }
          } else {
            uint32_t r[32];
            tmem_ld32(tl + c + 32 * h, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) stg[lane * 8 + ((4 * h + v) ^ (lane & 7))] = Vec16<bf16>::pack(o + 8 * v);
        }
        __syncwarp();
        // 2. transposed: 8 lanes per row, whole 128-byte lines to global memory
        uint4 x[8];
        size_t orow[8];
        bool live[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = 4 * k + r0, row = rbase + r;
          live[k] = row < ti.mlim;
          orow[k] = !live[k] ? 0 : (GROUPED && a.c_rows) ? (size_t)a.c_rows[row] : (size_t)row;
          x[k] = stg[r * 8 + (jr ^ (r & 7))];
        }
        bf16* base = static_cast<bf16*>(a.out) + ti.n0 + c + 8 * jr;
        if (EPI == EPI_RESIDUAL) {
          uint4 hres[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (live[k]) hres[k] = *reinterpret_cast<const uint4*>(base + orow[k] * a.ldo);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float hv[8], av[8];
            Vec16<bf16>::unpack(hres[k], hv);
            Vec16<bf16>::unpack(x[k], av);
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] += av[e];
            x[k] = Vec16<bf16>::pack(hv);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (live[k]) *reinterpret_cast<uint4*>(base + orow[k] * a.ldo) = x[k];
        __syncwarp();  // the slab is rewritten by the next 64 columns
      }
      // accumulator b may be overwritten by the tile after next
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acc_empty[b]);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 5) {
    fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host
// 2-D bf16 map over a row-major [rows, cols] matrix with row pitch `ld`
// elements, box {64 columns, box_rows rows}, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {ld * 2};
  return make_map_bf16(m, base, 2, dims, strides, box_rows);
}

template <int EPI, bool GROUPED>
cudaError_t tc_launch(const LaunchCtx& c, const CUtensorMap& ma, const CUtensorMap& mb, const GemmTcArgs& a) {
  auto kern = gemm_tc_kernel<EPI, GROUPED>;
  cudaError_t e = set_max_smem((const void*)kern, (int)TC_SMEM);
  if (e != cudaSuccess) return e;
  const int ncol = EPI == EPI_SWIGLU ? TC_BN / 2 : TC_BN;
  const int tiles = (a.N / ncol) * (GROUPED ? a.max_tiles_m : (a.M + TC_BM - 1) / TC_BM);
  const dim3 grid(std::min(tiles, c.num_sms));  // persistent: tiles t = blockIdx.x, + gridDim.x, ...
  return launch_k(kern, grid, dim3(TC_THREADS), TC_SMEM, c, ma, mb, a);
}

}  // namespace

bool gemm_tc_supported(int M, int N, int K, int epilogue) {
  if (!encode_fn()) return false;
  if (M < 1 || K % TC_BK) return false;
  if (epilogue == EPI_SWIGLU) return N % (TC_BN / 2) == 0;
  if (epilogue == EPI_STORE || epilogue == EPI_RESIDUAL) return N % TC_BN == 0;
  return false;
}

cudaError_t launch_gemm_tc(const LaunchCtx& c, const GemmTcArgs& a) {
  if (!gemm_tc_supported(a.M, a.N, a.K, a.epilogue)) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.a) & 15) || (reinterpret_cast<uintptr_t>(a.w) & 15) || (a.lda % 8) ||
      (a.ldo % 8))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  const uint64_t wrows = a.tile_start ? (uint64_t)a.w_rows_total : a.epilogue == EPI_SWIGLU ? 2ull * a.N : (uint64_t)a.N;
  if (!make_map(&ma, a.a, (uint64_t)a.M, (uint64_t)a.K, (uint64_t)a.lda, TC_BM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, a.w, wrows, (uint64_t)a.K, (uint64_t)a.K, a.epilogue == EPI_SWIGLU ? TC_BN / 2 : TC_BN))
    return cudaErrorInvalidValue;
  if (a.tile_start) {
    if (a.epilogue == EPI_STORE) return tc_launch<EPI_STORE, true>(c, ma, mb, a);
    if (a.epilogue == EPI_SWIGLU) return tc_launch<EPI_SWIGLU, true>(c, ma, mb, a);
    return cudaErrorInvalidValue;
  }
  switch (a.epilogue) {
    case EPI_STORE: return tc_launch<EPI_STORE, false>(c, ma, mb, a);
    case EPI_RESIDUAL: return tc_launch<EPI_RESIDUAL, false>(c, ma, mb, a);
    case EPI_SWIGLU: return tc_launch<EPI_SWIGLU, false>(c, ma, mb, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace q3
