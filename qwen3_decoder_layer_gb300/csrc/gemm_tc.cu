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
// For the q|k|v product (EPI_QKROPE, Backbone.forward's q_norm / k_norm, the
// rotary embedding of Backbone._rope and the cache append) the q|k|v rows
// never reach global memory: eight epilogue warps (two per TMEM lane
// quadrant, one 128-column half of the tile each) work one row per lane --
// the head's sum of squares, the RMSNorm, the rotation of the pairs
// (d, d + HD/2) -- and store queries to q_out [M][H][HD], keys and values to
// their cache rows.
// Split k (one row tile): the k-steps are cut into ranges, each (tile, range)
// item stores its fp32 accumulator, and a second kernel adds the ranges in
// order and applies the epilogue.
#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"

namespace q3 {

namespace {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
// Warps 0 .. E-1 epilogue, E TMA, E+1 MMA; E = 4, or 8 for the q|k|v
// epilogue (warps w and w + 4 share TMEM lanes 32 (w & 3) .. + 31 and take
// the two halves of the tile's columns).
__host__ __device__ constexpr int tc_epi_warps(int epi) { return epi == EPI_QKROPE ? 8 : 4; }
__host__ __device__ constexpr int tc_threads(int epi) { return (tc_epi_warps(epi) + 2) * 32; }
constexpr uint32_t TC_TMEM_COLS = 512;  // two 256-column accumulators
constexpr size_t TC_A_BYTES = (size_t)TC_BM * TC_BK * 2;   // 16 KB
constexpr size_t TC_B_BYTES = (size_t)TC_BN * TC_BK * 2;   // 32 KB
constexpr size_t TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
// epilogue staging: per epilogue warp 32 rows x 64 output columns (128 B per row)
constexpr size_t TC_STG_WARP = 32 * 128;
__host__ __device__ constexpr size_t tc_smem(int epi) {
  // the q|k|v epilogue stores each lane's own row and stages nothing
  return TC_STAGES * TC_STAGE_BYTES + 256 /* barriers */ + (epi == EPI_QKROPE ? 0 : 4 * TC_STG_WARP) +
         1024 /* align */;
}
static_assert(tc_smem(EPI_QKROPE) <= 227 * 1024, "q|k|v epilogue staging exceeds shared memory");

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

// The q|k|v epilogue of the heads in columns c0 .. c0 + 127 of one tile, by
// the lane owning tile row `row` (tl: the warp's TMEM lanes at the
// accumulator's first column; my_seq, my_pos: the row's sequence and position,
// 0 past the last row; csr: the row's RoPE table entries, (cos | sin << 16)
// bf16 pairs of the HD/2 frequencies).  The lane works on its row as tensor
// memory delivers it: the sum of squares of the head rounded to bf16, then
// (reading the row again) the RMSNorm with its two roundings and the one-rounding
// rotation of the pairs (d, d + HD/2): R(y1 c - y2 s), R(y2 c + y1 s) (both
// halves of a table row use the same frequencies); then 16-byte stores of
// its row: queries to q_out [M][H][HD], keys and values to their cache rows.
template <int HD>
__device__ __forceinline__ void qkrope_tile(const GemmTcArgs& a, const TileInfo& ti, uint32_t tl, int row,
                                            int my_seq, int my_pos, const uint4* csr, int c0) {
  constexpr int HALF = HD / 2;
  const QkRopeArgs& r = a.rope;
  const bool live = row < ti.mlim;
  for (int c = c0; c < c0 + TC_BN / 2; c += HD) {
    const int hd = (ti.n0 + c) / HD;  // head index in the q|k|v row (warp-uniform)
    const int kind = hd < r.H ? 0 : hd < r.H + r.KV ? 1 : 2;
    bf16* dst = kind == 0 ? static_cast<bf16*>(r.q_out) + ((size_t)row * r.H + hd) * HD
                          : static_cast<bf16*>(kind == 1 ? r.kcache : r.vcache) + (size_t)my_seq * r.seq_stride +
                                ((size_t)(hd - r.H - (kind == 2 ? r.KV : 0)) * r.capacity + my_pos) * HD;
    if (kind == 2) {  // values: rounded to bf16 and appended as they are
#pragma unroll
      for (int h = 0; h < HD / 32; ++h) {
        uint32_t v[32];
        tmem_ld32(tl + c + 32 * h, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(v[8 * q + e]);
          if (live) *reinterpret_cast<uint4*>(dst + 32 * h + 8 * q) = Vec16<bf16>::pack(o);
        }
      }
      continue;
    }
    // 1. the head's sum of squares of the bf16-rounded row: one chain per 32
    // columns, then added
    F2 ss = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < HD / 32; ++h) {
      uint32_t v[32];
      tmem_ld32(tl + c + 32 * h, v);
      F2 part = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 32; ++e) f2_add_sq_exact(part, rd<bf16>(__uint_as_float(v[e])));
      ss = h == 0 ? part : f2_add(ss, part);
    }
    const F2 rs = rms_scale2(ss, HD, r.eps);
    const bf16* g = static_cast<const bf16*>(kind == 0 ? r.q_gain : r.k_gain);
    // 2. the pairs (d, d + HALF), 16 values of d at a time, read again from
    // tensor memory
#pragma unroll
    for (int j = 0; j < HALF; j += 16) {
      uint32_t lo[16], hi[16];
      tmem_ld16(tl + c + j, lo);
      tmem_ld16(tl + c + HALF + j, hi);
#pragma unroll
      for (int q = 0; q < 2; ++q) {  // 8 values of d
        const int d0 = j + 8 * q;
        const uint4 gl = ld16(g + d0), gh = ld16(g + HALF + d0);
        const uint32_t glw[4] = {gl.x, gl.y, gl.z, gl.w}, ghw[4] = {gh.x, gh.y, gh.z, gh.w};
        const uint32_t cw[8] = {csr[d0 / 4].x, csr[d0 / 4].y, csr[d0 / 4].z, csr[d0 / 4].w,
                                csr[d0 / 4 + 1].x, csr[d0 / 4 + 1].y, csr[d0 / 4 + 1].z, csr[d0 / 4 + 1].w};
        // element e of a run of bf16 pairs: the low half of word e/2 when e is even
        auto half = [](uint32_t w, int e) { return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16)); };
        float y1[8], y2[8], gg[8];  // the rounded row values, normalised in place
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          y1[e] = rd<bf16>(__uint_as_float(lo[8 * q + e]));
          y2[e] = rd<bf16>(__uint_as_float(hi[8 * q + e]));
          gg[e] = half(glw[e / 2], e);
        }
        rms_apply2_v<bf16, 8>(y1, rs, gg, y1);
#pragma unroll
        for (int e = 0; e < 8; ++e) gg[e] = half(ghw[e / 2], e);
        rms_apply2_v<bf16, 8>(y2, rs, gg, y2);
        uint32_t o1[4], o2[4];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float cs = __uint_as_float(cw[e] << 16), sn = __uint_as_float(cw[e] & 0xffff0000u);
          // both products exact in fp32 (8-bit significands); one rounding of each result
          const float r1 = rd<bf16>(fmaf(y1[e], cs, -(y2[e] * sn))), r2 = rd<bf16>(fmaf(y2[e], cs, y1[e] * sn));
          if (e & 1) {
            o1[e / 2] |= __float_as_uint(r1) & 0xffff0000u;
            o2[e / 2] |= __float_as_uint(r2) & 0xffff0000u;
          } else {
            o1[e / 2] = __float_as_uint(r1) >> 16;
            o2[e / 2] = __float_as_uint(r2) >> 16;
          }
        }
        if (live) {
          *reinterpret_cast<uint4*>(dst + d0) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<uint4*>(dst + HALF + d0) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
      }
    }
  }
}

template <int EPI, bool GROUPED, int HD = 0>
__global__ void __launch_bounds__(tc_threads(EPI), 1)
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

  constexpr int NEPI = tc_epi_warps(EPI), TMA_WARP = NEPI, MMA_WARP = NEPI + 1;
  if (warp == TMA_WARP && lane == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], NEPI);  // one arrival per epilogue warp
    }
    mbar_fence_init();
  }
  if (warp == MMA_WARP) tmem_alloc(tmem_slot, TC_TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch();
  // grouped: the tile count comes from the routing scan of the previous kernel
  const int tiles_m = GROUPED ? a.tile_start[a.n_groups] : (a.M + TC_BM - 1) / TC_BM;
  const int tiles = tiles_m * (a.N / ncol);
  // split k (one row tile): item it = tile it % tiles over k-steps of range it / tiles
  const int splits = GROUPED ? 1 : max(1, a.splits);
  const int kps = (nk + splits - 1) / splits, items = tiles * splits;

  if (warp == TMA_WARP) {
    if (lane == 0) {  // TMA producer: the k-blocks of this block's tiles, in order
      int q = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const TileInfo ti = tile_of<GROUPED>(a, it % tiles, tiles_m, ncol);
        const int kb = (it / tiles) * kps, ke = min(nk, kb + kps);
        for (int kt = kb; kt < ke; ++kt, ++q) {
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
  } else if (warp == MMA_WARP) {
    if (lane == 0) {  // MMA issuer: tile i accumulates in TMEM columns (i & 1) * 256
      int q = 0, i = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x, ++i) {
        const int b = i & 1, use = i >> 1;
        if (use > 0 && !(ok = mbar_wait(&acc_empty[b], (uint32_t)((use - 1) & 1), a.err, 6))) break;
        fence_after();
        const uint32_t d = tmem + (uint32_t)(b * TC_BN);
        const int kb = (it / tiles) * kps, ke = min(nk, kb + kps);
        for (int kt = kb; kt < ke; ++kt, ++q) {
          const int s = q % TC_STAGES;
          if (!(ok = mbar_wait(&full[s], (uint32_t)((q / TC_STAGES) & 1), a.err, 4))) break;
          fence_after();
          const uint32_t sa = smem_u32(smem + s * TC_STAGE_BYTES);
          const uint32_t sb = sa + (uint32_t)TC_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            mma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), kIdesc, (kt != kb || kk != 0));
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
    }
  } else {  // epilogue: warp q reads TMEM lanes 32q .. 32q + 31 = tile rows
    // staging slab of this warp: row r's 16-byte chunk j sits at chunk j ^ (r & 7)
    uint4* stg = reinterpret_cast<uint4*>(smem + TC_STAGES * TC_STAGE_BYTES + 256 + warp * TC_STG_WARP);
    const int quad = warp & 3;  // TMEM lanes 32 quad .. + 31 = tile rows
    int i = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++i) {
      const int b = i & 1, use = i >> 1;
      const TileInfo ti = tile_of<GROUPED>(a, it % tiles, tiles_m, ncol);
      // q|k|v epilogue: the sequence and position of this lane's row, fetched
      // while the tile's MMAs run (rows past the last read 0)
      // and its RoPE table entries
      int my_seq = 0, my_pos = 0;
      uint4 csr[HD > 0 ? HD / 8 : 1];
      if constexpr (EPI == EPI_QKROPE) {
        const int myrow = ti.m0 + quad * 32 + lane;
        if (myrow < ti.mlim) { my_seq = a.rope.row_seq[myrow]; my_pos = a.rope.row_pos[myrow]; }
        const uint4* cp = reinterpret_cast<const uint4*>(a.rope.cs_bf16 + (size_t)my_pos * (HD / 2));
#pragma unroll
        for (int q = 0; q < HD / 8; ++q) csr[q] = __ldg(cp + q);
      }
      int okl = 1;  // lane 0 waits for the accumulator; the other lanes wait at the warp barrier
      if (lane == 0) okl = mbar_wait(&acc_full[b], (uint32_t)(use & 1), a.err, 5);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, okl, 0)) break;
      fence_after();
      const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * TC_BN);
      // the 8 rows this lane stores per 64-column slab: r = 4k + lane / 8, chunk lane % 8
      const int jr = lane & 7, r0 = lane >> 3;
      const int rbase = ti.m0 + quad * 32;
      if (splits > 1) {
        // split k: the raw fp32 accumulator of this range to the partial
        // tiles [split][M][N / ncol * 256] (the reduce kernel adds them in
        // range order and applies the epilogue)
        const int row = rbase + lane;
        float* dst = a.part + ((size_t)(it / tiles) * a.M + (row < ti.mlim ? row : 0)) * (size_t)(a.N / ncol * TC_BN) +
                     (size_t)(ti.n0 / ncol) * TC_BN;
        for (int c = 0; c < TC_BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(tl + c, v);
          if (row < ti.mlim) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(dst + c + 4 * q) =
                  make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                              __uint_as_float(v[4 * q + 3]));
          }
        }
      } else if constexpr (EPI == EPI_QKROPE)
        qkrope_tile<HD>(a, ti, tl, rbase + lane, my_seq, my_pos, csr, (warp >> 2) * (TC_BN / 2));
      else for (int c = 0; c < ncol; c += 64) {
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
  if (warp == MMA_WARP) {
    fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }
}

// Split-k reduction: out = epilogue(sum over the ranges, in range order, of
// the partial tiles), 8 output columns per thread; the epilogue arithmetic is
// the tile epilogue's (rounding, residual add, SiLU * up).
template <int EPI>
__global__ void __launch_bounds__(256) gemm_tc_reduce_kernel(GemmTcArgs a) {
  pdl_wait();
  pdl_launch();
  constexpr int NCOL = EPI == EPI_SWIGLU ? TC_BN / 2 : TC_BN;
  const size_t ntm = (size_t)(a.N / NCOL) * TC_BN;  // partial row pitch
  const int per_row = a.N / 8;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)a.M * per_row) return;
  const int row = (int)(idx / per_row), j0 = (int)(idx % per_row) * 8;
  // partial column of output column j0 (and of its up half for SiLU * up)
  const size_t c0 = EPI == EPI_SWIGLU ? (size_t)(j0 / NCOL) * TC_BN + j0 % NCOL : (size_t)j0;
  float g[8], u[8];
  for (int s = 0; s < a.splits; ++s) {
    const float* p = a.part + ((size_t)s * a.M + row) * ntm + c0;
    const float4 x0 = __ldcg(reinterpret_cast<const float4*>(p)), x1 = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = s == 0 ? xv[e] : g[e] + xv[e];
    if (EPI == EPI_SWIGLU) {
      const float4 y0 = __ldcg(reinterpret_cast<const float4*>(p + NCOL)),
                   y1 = __ldcg(reinterpret_cast<const float4*>(p + NCOL) + 1);
      const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) u[e] = s == 0 ? yv[e] : u[e] + yv[e];
    }
  }
  bf16* o = static_cast<bf16*>(a.out) + (size_t)row * a.ldo + j0;
  float r[8];
  if (EPI == EPI_SWIGLU) {
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = rd<bf16>(silu_f(rd<bf16>(g[e]))) * rd<bf16>(u[e]);
  } else if (EPI == EPI_RESIDUAL) {
    float hv[8];
    Vec16<bf16>::unpack(*reinterpret_cast<const uint4*>(o), hv);
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = hv[e] + rd<bf16>(g[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = g[e];
  }
  *reinterpret_cast<uint4*>(o) = Vec16<bf16>::pack(r);
}

// ---------------------------------------------------------------- host
// 2-D bf16 map over a row-major [rows, cols] matrix with row pitch `ld`
// elements, box {64 columns, box_rows rows}, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {ld * 2};
  return make_map_bf16(m, base, 2, dims, strides, box_rows);
}

template <int EPI, bool GROUPED, int HD = 0>
cudaError_t tc_launch(const LaunchCtx& c, const CUtensorMap& ma, const CUtensorMap& mb, const GemmTcArgs& a) {
  auto kern = gemm_tc_kernel<EPI, GROUPED, HD>;
  constexpr size_t smem = tc_smem(EPI);
  cudaError_t e = set_max_smem((const void*)kern, (int)smem);
  if (e != cudaSuccess) return e;
  const int ncol = EPI == EPI_SWIGLU ? TC_BN / 2 : TC_BN;
  const int tiles = (a.N / ncol) * (GROUPED ? a.max_tiles_m : (a.M + TC_BM - 1) / TC_BM) *
                    (GROUPED ? 1 : std::max(1, a.splits));
  const dim3 grid(std::min(tiles, c.num_sms));  // persistent: items it = blockIdx.x, + gridDim.x, ...
  return launch_k(kern, grid, dim3(tc_threads(EPI)), smem, c, ma, mb, a);
}

}  // namespace

bool gemm_tc_supported(int M, int N, int K, int epilogue) {
  if (!encode_fn()) return false;
  if (M < 1 || K % TC_BK) return false;
  if (epilogue == EPI_SWIGLU) return N % (TC_BN / 2) == 0;
  if (epilogue == EPI_STORE || epilogue == EPI_RESIDUAL || epilogue == EPI_QKROPE) return N % TC_BN == 0;
  return false;
}

int gemm_tc_splits(int M, int N, int K, int epilogue, int num_sms) {
  if (M > TC_BM || !(epilogue == EPI_STORE || epilogue == EPI_RESIDUAL || epilogue == EPI_SWIGLU) ||
      !gemm_tc_supported(M, N, K, epilogue))
    return 1;
  const int tiles = N / (epilogue == EPI_SWIGLU ? TC_BN / 2 : TC_BN), nk = K / TC_BK;
  if (2 * tiles > num_sms) return 1;
  const int s = std::min({16, nk / 2, num_sms / tiles});  // at least 2 k-steps per range
  if (s < 2) return 1;
  const int kps = (nk + s - 1) / s;
  return (nk + kps - 1) / kps;
}

size_t gemm_tc_part_floats(int M, int N, int epilogue, int splits) {
  const int ncol = epilogue == EPI_SWIGLU ? TC_BN / 2 : TC_BN;
  return (size_t)splits * M * (size_t)(N / ncol) * TC_BN;
}

cudaError_t launch_gemm_tc_reduce(const LaunchCtx& c, const GemmTcArgs& a) {
  if (a.splits < 2 || !a.part || a.N % 8 || (a.ldo % 8)) return cudaErrorInvalidValue;
  const long long n = (long long)a.M * (a.N / 8);
  const dim3 grid((unsigned)((n + 255) / 256)), block(256);
  switch (a.epilogue) {
    case EPI_STORE: return launch_k(gemm_tc_reduce_kernel<EPI_STORE>, grid, block, 0, c, a);
    case EPI_RESIDUAL: return launch_k(gemm_tc_reduce_kernel<EPI_RESIDUAL>, grid, block, 0, c, a);
    case EPI_SWIGLU: return launch_k(gemm_tc_reduce_kernel<EPI_SWIGLU>, grid, block, 0, c, a);
  }
  return cudaErrorInvalidValue;
}

bool gemm_tc_qkrope_supported(int M, int H, int KV, int D) {
  return (D == 64 || D == 128) && H > 0 && KV > 0 && gemm_tc_supported(M, (H + 2 * KV) * D, 64, EPI_QKROPE);
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
  if (a.epilogue == EPI_QKROPE) {
    const QkRopeArgs& r = a.rope;
    if (a.tile_start || !gemm_tc_qkrope_supported(a.M, r.H, r.KV, r.D) || a.N != (r.H + 2 * r.KV) * r.D ||
        !r.q_out || !r.kcache || !r.vcache || !r.q_gain || !r.k_gain || !r.cos_t || !r.sin_t || !r.row_seq ||
        !r.row_pos || (reinterpret_cast<uintptr_t>(r.q_out) & 15) || (reinterpret_cast<uintptr_t>(r.kcache) & 15) ||
        (reinterpret_cast<uintptr_t>(r.vcache) & 15) || (reinterpret_cast<uintptr_t>(r.q_gain) & 15) ||
        (reinterpret_cast<uintptr_t>(r.k_gain) & 15) || (reinterpret_cast<uintptr_t>(r.cos_t) & 15) ||
        (reinterpret_cast<uintptr_t>(r.sin_t) & 15) || !r.cs_bf16 || (reinterpret_cast<uintptr_t>(r.cs_bf16) & 15) ||
        (r.seq_stride % 8))
      return cudaErrorInvalidValue;
    return r.D == 128 ? tc_launch<EPI_QKROPE, false, 128>(c, ma, mb, a) : tc_launch<EPI_QKROPE, false, 64>(c, ma, mb, a);
  }
  if (a.splits > 1 && (a.tile_start || !a.part || a.M > TC_BM || a.splits > a.K / TC_BK ||
                       !(a.epilogue == EPI_STORE || a.epilogue == EPI_RESIDUAL || a.epilogue == EPI_SWIGLU)))
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
