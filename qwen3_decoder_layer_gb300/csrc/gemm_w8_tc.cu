// Tensor-core GEMM for affine int8 weights and up to 32 activation rows -- the
// linears of a batched decode step of an int8 stack (maya2_mlx/backbone.py,
// Backbone.forward run on one new row per sequence, with the weights in the
// group-wise affine int8 form w = scale * q + bias of the int8 export):
//
//   C[m, n] = sum_k A[m, k] (scale[n, g(k)] q[n, k] + bias[n, g(k)])
//           = sum_g scale[n, g] (sum_{k in g} q[n, k] A[m, k]) + bias[n, g] (sum_{k in g} A[m, k])
//
// The dequantised weight is never formed: the integer codes q (0..255, exact
// in bf16) go through tcgen05.mma as the 128-row A operand and the activation
// rows as the N = 32 B operand (no padded MMA work), one 64-k group per
// tensor-memory accumulator slot of 32 columns; the epilogue warps add
// scale * (sum q a) + bias * (sum a) group by group in fp32 registers.
//
// Warp roles (448 threads): warps 0-3 epilogue (warp q owns TMEM lanes
// 32q..32q+31 = weight rows of the tile), warp 4 TMA, warp 5 MMA, warps 6-13
// converters.  TMA fills a ring of load stages with the int8 tile (128 rows x
// 64 bytes; SiLU * up: 64 gate rows and the 64 matching up rows) and the
// activation tile (32 rows x 64 bf16, 128-byte swizzle).  The converters turn
// the codes into bf16 in the 128-byte-swizzled K-major layout the MMA reads,
// copy the activation tile beside them, and sum each activation row over the
// group; the MMA warp runs four K = 16 steps per group into slot i % 8.  K is
// split over CTAs when the tiles alone do not fill the GPU: each split stores
// its partial tile in its own fp32 workspace slice and the last CTA of a tile
// (an atomic counter) adds the slices in split order and applies the epilogue
// (rounding, residual add or SiLU * up), so the result does not depend on
// which CTA finishes when.
#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"

namespace q3 {

namespace {

using namespace tc;

constexpr int WT_ROWS = 128;        // weight rows per tile (MMA M)
constexpr int WT_MT = 32;           // activation rows (MMA N)
constexpr int WT_BK = 64;           // k per group step (one quantisation group at most)
constexpr int WT_LSTAGES = 10;      // load ring: int8 tile + activation tile
constexpr int WT_CSTAGES = 4;       // converted ring: bf16 codes + activation copy
constexpr int WT_SLOTS = 8;         // TMEM accumulator slots of 32 columns
constexpr int WT_SRING = 16;        // activation-sum ring (see the converter)
constexpr int WT_THREADS = 448;  // 4 epilogue, TMA, MMA, 8 converter warps
constexpr uint32_t WT_TMEM_COLS = WT_SLOTS * WT_MT;  // 256

constexpr size_t WT_I8_BYTES = (size_t)WT_ROWS * WT_BK;        // 8 KB
constexpr size_t WT_ACT_BYTES = (size_t)WT_MT * WT_BK * 2;     // 4 KB
constexpr size_t WT_LSTAGE = WT_ACT_BYTES + WT_I8_BYTES;       // activation first (1024-aligned)
constexpr size_t WT_Q_BYTES = (size_t)WT_ROWS * WT_BK * 2;     // 16 KB
constexpr size_t WT_CSTAGE = WT_Q_BYTES + WT_ACT_BYTES;        // 20 KB, both 1024-aligned
constexpr size_t WT_OFF_C = WT_LSTAGES * WT_LSTAGE;            // 120 KB
constexpr size_t WT_OFF_S = WT_OFF_C + WT_CSTAGES * WT_CSTAGE; // sums [WT_SRING][32] fp32
constexpr size_t WT_OFF_X = WT_OFF_S + (size_t)WT_SRING * WT_MT * 4;  // up-row exchange [64][33] fp32
constexpr size_t WT_OFF_BAR = WT_OFF_X + (size_t)64 * 33 * 4;
constexpr int WT_NBAR = 2 * WT_LSTAGES + 2 * WT_CSTAGES + 2 * WT_SLOTS + WT_SRING;
constexpr size_t WT_SMEM = WT_OFF_BAR + WT_NBAR * 8 + 16 + 1024 /* alignment */;

constexpr uint32_t kIdescW8 = idesc_bf16(WT_ROWS, WT_MT, false);

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile with
// 128-byte rows (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// bf16 bits of the integer q in [0, 255] (exact): the float 2^23 + q minus 2^23.
__device__ __forceinline__ uint32_t u8_bf16_pair(uint32_t word, int b0) {
  const float f0 = __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7540u | (unsigned)b0)) - 8388608.f;
  const float f1 = __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7540u | (unsigned)(b0 + 1))) - 8388608.f;
  return __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);  // high halves: element b0 low
}

__device__ __forceinline__ void ep_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int EPI>
__global__ void __launch_bounds__(WT_THREADS, 1)
    gemm_w8_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_a,
                      SkinnyArgs a) {
  constexpr bool PAIR = EPI == EPI_SWIGLU;
  constexpr int TN = PAIR ? WT_ROWS / 2 : WT_ROWS;  // output columns per tile
  extern __shared__ uint8_t wt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(wt_smem_raw) + 1023) & ~uintptr_t(1023));
  float* sS = reinterpret_cast<float*>(smem + WT_OFF_S);
  float* xch = reinterpret_cast<float*>(smem + WT_OFF_X);
  uint64_t* lfull = reinterpret_cast<uint64_t*>(smem + WT_OFF_BAR);  // TMA -> converters
  uint64_t* lempty = lfull + WT_LSTAGES;                             // converters -> TMA
  uint64_t* cfull = lempty + WT_LSTAGES;                             // converters -> MMA
  uint64_t* cempty = cfull + WT_CSTAGES;                             // MMA (commit) -> converters
  uint64_t* tfull = cempty + WT_CSTAGES;                             // MMA (commit) -> epilogue
  uint64_t* tempty = tfull + WT_SLOTS;                               // epilogue -> MMA
  uint64_t* sfull = tempty + WT_SLOTS;                               // converters -> epilogue (sums)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfull + WT_SRING);
  __shared__ int s_last;
  int* err = a.err;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TN;
  const int nkt = a.K / WT_BK, kpc = a.ktiles_per_split;
  const int kt0 = blockIdx.y * kpc, kt1 = min(nkt, kt0 + kpc), nloc = kt1 - kt0;

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < WT_LSTAGES; ++s) { mbar_init(&lfull[s], 1); mbar_init(&lempty[s], 8); }
    for (int s = 0; s < WT_CSTAGES; ++s) { mbar_init(&cfull[s], 8); mbar_init(&cempty[s], 1); }
    for (int j = 0; j < WT_SLOTS; ++j) { mbar_init(&tfull[j], 1); mbar_init(&tempty[j], 4); }
    for (int j = 0; j < WT_SRING; ++j) mbar_init(&sfull[j], 8);
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(tmem_slot, WT_TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------ TMA: int8 codes need nothing from the previous kernel
    if (lane == 0) {
      for (int i = 0; i < nloc; ++i) {
        const int s = i % WT_LSTAGES, kx = (kt0 + i) * WT_BK;
        if (i >= WT_LSTAGES && !mbar_wait(&lempty[s], (uint32_t)((i / WT_LSTAGES - 1) & 1), err, 11)) break;
        uint8_t* st = smem + s * WT_LSTAGE;
        mbar_expect_tx(&lfull[s], (uint32_t)WT_LSTAGE);
        if (PAIR) {
          tma_load_2d(st + WT_ACT_BYTES, &map_w, kx, n0, &lfull[s]);
          tma_load_2d(st + WT_ACT_BYTES + WT_I8_BYTES / 2, &map_w, kx, a.N + n0, &lfull[s]);
        } else {
          tma_load_2d(st + WT_ACT_BYTES, &map_w, kx, n0, &lfull[s]);
        }
        if (i == 0) pdl_wait();  // the activations come from the previous kernel
        tma_load_2d(st, &map_a, kx, 0, &lfull[s]);
      }
      if (nloc == 0) pdl_wait();
    }
    pdl_launch();
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    pdl_launch();
    if (lane == 0) {
      for (int i = 0; i < nloc; ++i) {
        const int c = i % WT_CSTAGES, j = i % WT_SLOTS, v = i / WT_SLOTS;
        if (!mbar_wait(&cfull[c], (uint32_t)((i / WT_CSTAGES) & 1), err, 12)) break;
        if (v > 0 && !mbar_wait(&tempty[j], (uint32_t)((v - 1) & 1), err, 13)) break;
        fence_after();
        const uint32_t sq = smem_u32(smem + WT_OFF_C + c * WT_CSTAGE);
        const uint32_t sa = sq + (uint32_t)WT_Q_BYTES;
        const uint32_t d = tmem + (uint32_t)(j * WT_MT);
#pragma unroll
        for (int kk = 0; kk < WT_BK / 16; ++kk)
          mma_bf16(d, sw128_desc(sq + kk * 32), sw128_desc(sa + kk * 32), kIdescW8, kk != 0);
        mma_commit(&cempty[c]);
        mma_commit(&tfull[j]);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ converters (256 threads)
    pdl_launch();
    const int ct = threadIdx.x - 6 * 32;
    for (int i = 0; i < nloc; ++i) {
      const int s = i % WT_LSTAGES, c = i % WT_CSTAGES;
      if (!mbar_wait(&lfull[s], (uint32_t)((i / WT_LSTAGES) & 1), err, 14)) break;
      if (i >= WT_CSTAGES && !mbar_wait(&cempty[c], (uint32_t)((i / WT_CSTAGES - 1) & 1), err, 15)) break;
      const uint8_t* st = smem + s * WT_LSTAGE;
      uint8_t* cq = smem + WT_OFF_C + c * WT_CSTAGE;
      // Every shared-memory read of the group is issued before the first store
      // (the stores could alias the reads as far as the compiler knows, and
      // would otherwise serialise them).
      // codes: task t = (row t / 4, 16-byte chunk t % 4) -> bf16 chunks 2 (t % 4), + 1 of the row
      uint4 w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int t = ct + 256 * u;
        w[u] = *reinterpret_cast<const uint4*>(st + WT_ACT_BYTES + (t >> 2) * WT_BK + (t & 3) * 16);
      }
      const uint4 act = reinterpret_cast<const uint4*>(st)[ct];  // activation chunk ct (of 256)
      // group sums of the activation rows (the first four converter warps):
      // row m = ct / 4 sums its logical chunks 2p, 2p + 1
      const int m = (ct & 127) >> 2, p = ct & 3;
      uint4 sv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) sv[h] = *reinterpret_cast<const uint4*>(st + sw128_off(m, 2 * p + h));
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int t = ct + 256 * u, r = t >> 2, j = t & 3;
        uint4 lo, hi;
        lo.x = u8_bf16_pair(w[u].x, 0); lo.y = u8_bf16_pair(w[u].x, 2);
        lo.z = u8_bf16_pair(w[u].y, 0); lo.w = u8_bf16_pair(w[u].y, 2);
        hi.x = u8_bf16_pair(w[u].z, 0); hi.y = u8_bf16_pair(w[u].z, 2);
        hi.z = u8_bf16_pair(w[u].w, 0); hi.w = u8_bf16_pair(w[u].w, 2);
        *reinterpret_cast<uint4*>(cq + sw128_off(r, 2 * j)) = lo;
        *reinterpret_cast<uint4*>(cq + sw128_off(r, 2 * j + 1)) = hi;
      }
      // activation tile copied as is (same swizzled layout)
      reinterpret_cast<uint4*>(cq + WT_Q_BYTES)[ct] = act;
      if (ct < 128) {
        float sum = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[8];
          Vec16<bf16>::unpack(sv[h], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) sum += x[e];
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        // Ring of WT_SRING entries: group i is converted only after the MMA of
        // group i - WT_CSTAGES completed, which the MMA issued only after the
        // epilogue released group i - WT_CSTAGES - WT_SLOTS = i - 12; entry
        // i % 16 was last written for group i - 16, already consumed.
        if (p == 0) sS[(i % WT_SRING) * WT_MT + m] = sum;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {  // one arrival per converter warp on each
        mbar_arrive_cta(&lempty[s]);
        mbar_arrive_cta(&cfull[c]);
        mbar_arrive_cta(&sfull[i % WT_SRING]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue: warp q, TMEM lanes 32q.. = tile rows
    // (the workspace, counters and output may still be in use by the previous kernel)
    pdl_wait();
    pdl_launch();
    const int row = warp * 32 + lane;  // tile row
    const int col = PAIR ? n0 + (row & 63) : n0 + row;
    const bool live = col < a.N;
    const size_t wrow = PAIR && row >= 64 ? (size_t)a.N + col : (size_t)col;
    const unsigned short* SC = static_cast<const unsigned short*>(a.scale);
    const unsigned short* BI = static_cast<const unsigned short*>(a.bias);
    const int gpr = a.K / a.group;
    auto sb_of = [&](int i) -> uint32_t {
      if (!live || i >= nloc) return 0u;
      const size_t gi = wrow * gpr + (size_t)((kt0 + i) * WT_BK) / a.group;
      return (uint32_t)SC[gi] | ((uint32_t)BI[gi] << 16);
    };
    float acc[WT_MT];
#pragma unroll
    for (int m = 0; m < WT_MT; ++m) acc[m] = 0.f;
    bool ok = true;
    // group i: accumulate slot i % 8 with the group's scale and bias (sb)
    auto step = [&](int i, uint32_t sb) {
      const int j = i % WT_SLOTS, v = i / WT_SLOTS;
      int okl = ok;
      if (lane == 0 && ok)
        okl = mbar_wait(&tfull[j], (uint32_t)(v & 1), err, 16) &&
              mbar_wait(&sfull[i % WT_SRING], (uint32_t)((i / WT_SRING) & 1), err, 17);
      __syncwarp();
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      fence_after();
      uint32_t d[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * WT_MT), d);
      const float scl = __uint_as_float(sb << 16), bia = __uint_as_float(sb & 0xffff0000u);
      const float4* S4 = reinterpret_cast<const float4*>(sS + (i % WT_SRING) * WT_MT);
#pragma unroll
      for (int q = 0; q < WT_MT / 4; ++q) {
        const float4 sv = S4[q];
        acc[4 * q] = fmaf(bia, sv.x, fmaf(scl, __uint_as_float(d[4 * q]), acc[4 * q]));
        acc[4 * q + 1] = fmaf(bia, sv.y, fmaf(scl, __uint_as_float(d[4 * q + 1]), acc[4 * q + 1]));
        acc[4 * q + 2] = fmaf(bia, sv.z, fmaf(scl, __uint_as_float(d[4 * q + 2]), acc[4 * q + 2]));
        acc[4 * q + 3] = fmaf(bia, sv.w, fmaf(scl, __uint_as_float(d[4 * q + 3]), acc[4 * q + 3]));
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&tempty[j]);
    };
    // the scattered scale / bias loads come from HBM: keep four groups in flight
    uint32_t sb0 = sb_of(0), sb1 = sb_of(1), sb2 = sb_of(2), sb3 = sb_of(3);
    for (int i = 0; i < nloc; i += 4) {
      uint32_t sb = sb0;
      sb0 = sb_of(i + 4);
      step(i, sb);
      if (i + 1 < nloc) { sb = sb1; sb1 = sb_of(i + 5); step(i + 1, sb); }
      if (i + 2 < nloc) { sb = sb2; sb2 = sb_of(i + 6); step(i + 2, sb); }
      if (i + 3 < nloc) { sb = sb3; sb3 = sb_of(i + 7); step(i + 3, sb); }
    }

    auto finish = [&](int m, int c, float g, float u) {
      const size_t o = (size_t)m * a.ldo + c;
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
    if (gridDim.y == 1) {
      if (PAIR) {  // up rows (warps 2, 3) hand their sums to the gate rows (warps 0, 1)
        if (row >= 64)
#pragma unroll
          for (int m = 0; m < WT_MT; ++m) xch[(row - 64) * 33 + m] = acc[m];
        ep_sync();
        if (row < 64 && live && ok)
#pragma unroll
          for (int m = 0; m < WT_MT; ++m)
            if (m < a.M) finish(m, col, acc[m], xch[row * 33 + m]);
      } else if (live && ok) {
#pragma unroll
        for (int m = 0; m < WT_MT; ++m)
          if (m < a.M) finish(m, col, acc[m], 0.f);
      }
    } else {
      const int ldw = PAIR ? 2 * a.N : a.N;
      const size_t slice = (size_t)a.M * ldw;
      if (live) {
        float* wsp = a.ws + blockIdx.y * slice + (PAIR && row >= 64 ? (size_t)a.N + col : (size_t)col);
#pragma unroll
        for (int m = 0; m < WT_MT; ++m)
          if (m < a.M) __stcg(wsp + (size_t)m * ldw, acc[m]);
      }
      __threadfence();
      ep_sync();
      if (threadIdx.x == 0) s_last = atomicAdd(a.counters + blockIdx.x, 1) == (int)gridDim.y - 1;
      ep_sync();
      if (s_last) {
        __threadfence();
        // four columns per item, the splits' slices loaded eight at a time
        // (independent loads) and added in split order
        for (int idx = threadIdx.x; idx < a.M * (TN / 4); idx += 128) {
          const int m = idx / (TN / 4), c = n0 + (idx % (TN / 4)) * 4;
          if (c >= a.N) continue;
          const float* pg = a.ws + (size_t)m * ldw + c;
          float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
          for (int k0 = 0; k0 < (int)gridDim.y; k0 += 8) {
            float4 gv[8], uv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k0 + k < (int)gridDim.y) {
                gv[k] = __ldcg(reinterpret_cast<const float4*>(pg + (k0 + k) * slice));
                if (PAIR) uv[k] = __ldcg(reinterpret_cast<const float4*>(pg + (k0 + k) * slice + a.N));
              }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k0 + k < (int)gridDim.y) {
                g.x += gv[k].x; g.y += gv[k].y; g.z += gv[k].z; g.w += gv[k].w;
                if (PAIR) { u.x += uv[k].x; u.y += uv[k].y; u.z += uv[k].z; u.w += uv[k].w; }
              }
            }
          }
          if (ok) {
            finish(m, c, g.x, u.x);
            finish(m, c + 1, g.y, u.y);
            finish(m, c + 2, g.z, u.z);
            finish(m, c + 3, g.w, u.w);
          }
        }
        if (threadIdx.x == 0) a.counters[blockIdx.x] = 0;
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 5) {
    fence_after();
    tmem_dealloc(tmem, WT_TMEM_COLS);
  }
}

// 2-D uint8 map over a row-major [rows, cols] matrix (row pitch cols bytes),
// box {64 bytes, box_rows rows}, no swizzle, zero fill.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[2] = {cols, rows}, s[1] = {cols};
  cuuint32_t box[2] = {(cuuint32_t)WT_BK, box_rows}, estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), d, s, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI>
cudaError_t wt_launch(const LaunchCtx& c, const CUtensorMap& mw, const CUtensorMap& ma, const SkinnyArgs& a,
                      dim3 grid) {
  const cudaError_t e = set_max_smem((const void*)gemm_w8_tc_kernel<EPI>, (int)WT_SMEM);
  if (e != cudaSuccess) return e;
  return launch_k(gemm_w8_tc_kernel<EPI>, grid, dim3(WT_THREADS), WT_SMEM, c, mw, ma, a);
}

}  // namespace

bool gemm_w8_tc_supported(int M, int N, int K, int group, int epilogue) {
  if (!encode_fn()) return false;
  return M >= 1 && M <= WT_MT && N >= 4 && N % 4 == 0 && K % WT_BK == 0 && group % WT_BK == 0 && K % group == 0 &&
         (epilogue == EPI_STORE || epilogue == EPI_STORE_F32 || epilogue == EPI_RESIDUAL || epilogue == EPI_SWIGLU);
}

cudaError_t launch_gemm_w8_tc(const LaunchCtx& c, SkinnyArgs a) {
  if (!gemm_w8_tc_supported(a.M, a.N, a.K, a.group, a.epilogue)) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.a) & 15) || (reinterpret_cast<uintptr_t>(a.w) & 15) || (a.lda % 8))
    return cudaErrorInvalidValue;
  const bool pair = a.epilogue == EPI_SWIGLU;
  const int tn = pair ? WT_ROWS / 2 : WT_ROWS, tiles = (a.N + tn - 1) / tn, nkt = a.K / WT_BK;
  // K splits so that the tiles fill the SMs once (one CTA per SM), at most 16
  int split = std::max(1, std::min({c.num_sms / tiles, nkt, 16}));
  a.ktiles_per_split = (nkt + split - 1) / split;
  split = (nkt + a.ktiles_per_split - 1) / a.ktiles_per_split;
  if (split > 1 && (!a.ws || !a.counters)) return cudaErrorInvalidValue;
  CUtensorMap mw, ma;
  const uint64_t wrows = pair ? 2ull * a.N : (uint64_t)a.N;
  if (!make_map_u8(&mw, a.w, wrows, (uint64_t)a.K, pair ? WT_ROWS / 2 : WT_ROWS)) return cudaErrorInvalidValue;
  const uint64_t adims[2] = {(uint64_t)a.K, (uint64_t)a.M};
  const uint64_t astr[1] = {(uint64_t)a.lda * 2};
  if (!make_map_bf16(&ma, a.a, 2, adims, astr, WT_MT)) return cudaErrorInvalidValue;
  const dim3 grid(tiles, split);
  switch (a.epilogue) {
    case EPI_STORE: return wt_launch<EPI_STORE>(c, mw, ma, a, grid);
    case EPI_STORE_F32: return wt_launch<EPI_STORE_F32>(c, mw, ma, a, grid);
    case EPI_RESIDUAL: return wt_launch<EPI_RESIDUAL>(c, mw, ma, a, grid);
    case EPI_SWIGLU: return wt_launch<EPI_SWIGLU>(c, mw, ma, a, grid);
  }
  return cudaErrorInvalidValue;
}

}  // namespace q3
