// Prefill attention on the tensor cores (bf16): the causal GQA attention of
// maya2_mlx/backbone.py, Backbone.forward (`scaled_dot_product_attention`
// with `mask="causal"` for T > 1, "attention over keys 0..pos (fp32 softmax,
// one rounding)"; q head h reads kv head h / (H / KV), the repeat_kv of
// rlx_flow/blocks/qwen3_decoder.rs), for query rows whose q/k RMSNorm, RoPE
// and cache append are done.
//
// One CTA owns 128 consecutive query rows of one sequence and one q head, and
// walks the keys 0 .. last position in tiles of 128 (flash attention):
//   S_j = Q K_j^T          tcgen05.mma, M = N = 128, K = head_dim, into tensor
//                          memory (two S buffers, so S_{j+1} is computed while
//                          S_j is in the softmax)
//   P_j = 2^(s log2e/sqrt(D) - m), online row reference m and sum l in fp32,
//                          written to shared memory as two bf16 parts
//                          P = hi + lo (16 significant bits, so the
//                          probabilities keep close to fp32 accuracy) in the
//                          MMA's 128-byte-swizzled A layout; when m moves the
//                          accumulator row is rescaled in tensor memory
//   O  += hi V_j + lo V_j  tcgen05.mma, M = 128, N = head_dim, K = 128, with V
//                          read MN-major straight from its cache layout
//   out = O / l            rounded once to bf16.
// K and V tiles come from the cache by 3-D TMA (head_dim, kv_head * capacity
// + position, sequence) into a 2-stage ring.  Warps 0-7 run the softmax and
// the epilogue: warps w and w + 4 share tensor-memory lanes 32 (w % 4) ..
// +31, i.e. query rows, and split the keys of a tile (and the accumulator
// columns) in halves, exchanging row maxima and sums through shared memory.
// Warp 8 issues TMA, warp 9 the MMAs.
#include <math_constants.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace q3 {

namespace {

using namespace tc;

constexpr int AT_BM = 128, AT_BN = 128;  // query rows per CTA, keys per tile
constexpr int AT_THREADS = 320;          // warps 0-7 softmax / epilogue, 8 TMA, 9 MMA
constexpr int AT_TMA_WARP = 8, AT_MMA_WARP = 9;
constexpr int AT_STAGES = 2;
constexpr uint32_t AT_TMEM_COLS = 512;   // S0 [0, 128), S1 [128, 256), O [256, 256 + D)
constexpr uint32_t AT_O_COL = 256;

template <int D> struct ATL {
  static constexpr int NC = D / 64;                        // 64-element column blocks of a head row
  static constexpr uint32_t SUB = 128 * 128;               // 128 rows x 128 bytes, one swizzled block
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t KV_OFF = Q_OFF + NC * SUB;
  static constexpr uint32_t STAGE = 2 * NC * SUB;          // K blocks, then V blocks
  static constexpr uint32_t P_OFF = KV_OFF + AT_STAGES * STAGE;
  static constexpr uint32_t PLO_OFF = P_OFF + 2 * SUB;    // P hi, then P lo: 128 rows x 128 keys each
  static constexpr uint32_t RED_OFF = PLO_OFF + 2 * SUB;   // [2][128] row maxima / sums of the key halves
  static constexpr uint32_t BAR_OFF = RED_OFF + 2 * 128 * 4;
  static constexpr size_t SMEM = BAR_OFF + 128 + 1024;     // barriers + 1024-byte alignment slack
};

// 2^x on the special-function unit (PTX ex2.approx; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Barrier of the two softmax warps that own lane quadrant qd (64 threads).
__device__ __forceinline__ void pair_sync(int qd) { asm volatile("bar.sync %0, 64;" ::"r"(qd + 1) : "memory"); }

template <int D>
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, AttnTcArgs a) {
  using L = ATL<D>;
  extern __shared__ uint8_t at_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* o_done = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = a.n_qblocks - 1 - (int)(blockIdx.x / a.H);  // later (longer) query tiles first
  const int h = (int)(blockIdx.x % a.H);
  const AttnQBlock qb = a.qblocks[b];
  const int kvh = h / (a.H / a.KV);
  const int n_tiles = (qb.pos0 + qb.nrows + AT_BN - 1) / AT_BN;

  if (warp == AT_TMA_WARP && lane == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_full, 256);
    mbar_init(o_done, 1);
    mbar_fence_init();
  }
  if (warp == AT_MMA_WARP) tmem_alloc(tmem_slot, AT_TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // q and the appended keys come from the previous kernel
  pdl_launch();

  if (warp == AT_TMA_WARP) {
    if (lane == 0) {  // ---------------------------------------- TMA producer
      mbar_expect_tx(q_full, L::NC * L::SUB);
      for (int c = 0; c < L::NC; ++c) tma_load_2d(smem + L::Q_OFF + c * L::SUB, &map_q, h * D + c * 64, qb.row0, q_full);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % AT_STAGES;
        if (j >= AT_STAGES && !mbar_wait(&kv_empty[s], (uint32_t)((j / AT_STAGES - 1) & 1), a.err, 6)) break;
        uint8_t* st = smem + L::KV_OFF + s * L::STAGE;
        const int row = kvh * a.capacity + j * AT_BN;
        mbar_expect_tx(&kv_full[s], L::STAGE);
        for (int c = 0; c < L::NC; ++c) {
          tma_load_3d(st + c * L::SUB, &map_k, c * 64, row, qb.seq, &kv_full[s]);
          tma_load_3d(st + (L::NC + c) * L::SUB, &map_v, c * 64, row, qb.seq, &kv_full[s]);
        }
      }
    }
  } else if (warp == AT_MMA_WARP) {
    if (lane == 0) {  // ---------------------------------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16(AT_BM, AT_BN, false);
      constexpr uint32_t idesc_o = idesc_bf16(AT_BM, D, true);
      const uint32_t q_addr = smem_u32(smem + L::Q_OFF);
      const uint32_t p_addr = smem_u32(smem + L::P_OFF);
      const uint32_t plo_addr = smem_u32(smem + L::PLO_OFF);
      bool ok = mbar_wait(q_full, 0, a.err, 7);
      auto issue_s = [&](int j) {
        const int s = j % AT_STAGES;
        if (!mbar_wait(&kv_full[s], (uint32_t)((j / AT_STAGES) & 1), a.err, 8)) return false;
        fence_after();
        const uint32_t k_addr = smem_u32(smem + L::KV_OFF + s * L::STAGE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * L::SUB + (ks % 4) * 32;
          mma_bf16(tmem + (j & 1) * AT_BN, sw128_desc(q_addr + off), sw128_desc(k_addr + off), idesc_s, ks > 0);
        }
        mma_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles && !issue_s(j + 1)) break;
        if (!mbar_wait(p_full, (uint32_t)(j & 1), a.err, 9)) break;
        fence_after();
        const uint32_t v_addr = smem_u32(smem + L::KV_OFF + (j % AT_STAGES) * L::STAGE + L::NC * L::SUB);
#pragma unroll
        for (int ks = 0; ks < AT_BN / 16; ++ks) {
          const uint32_t off = (ks / 4) * L::SUB + (ks % 4) * 32;
          const uint64_t vd = sw128_desc_mn(v_addr + ks * 2048, L::SUB);
          mma_bf16(tmem + AT_O_COL, sw128_desc(p_addr + off), vd, idesc_o, (j | ks) != 0);
          mma_bf16(tmem + AT_O_COL, sw128_desc(plo_addr + off), vd, idesc_o, 1);
        }
        mma_commit(o_done);
        mma_commit(&kv_empty[j % AT_STAGES]);
      }
    }
  } else {  // -------------------------------------------------- softmax / epilogue
    const int qd = warp & 3, hf = warp >> 2;  // lane quadrant (rows), key / column half
    const int r = qd * 32 + lane;              // query row of the tile = tensor-memory lane
    const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
    const int q_pos = qb.pos0 + r;
    constexpr int HK = AT_BN / 2, HD = D / 2;  // keys / accumulator columns per half
    uint8_t* Ph = smem + L::P_OFF + hf * L::SUB;   // this half's 64 keys = one swizzled block
    uint8_t* Pl = smem + L::PLO_OFF + hf * L::SUB;
    float* red = reinterpret_cast<float*>(smem + L::RED_OFF);  // [2][128]
    const float c = a.scale_log2;
    float m = -CUDART_INF_F, l = 0.f;  // l: this half's share of the row sum
    // After a failed (timed-out) wait a warp stops waiting but keeps to the
    // loop, so that the pair barriers of both halves stay matched.
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      int okl = ok;
      if (lane == 0 && ok) okl = mbar_wait(&s_full[j & 1], (uint32_t)((j >> 1) & 1), a.err, 10);
      __syncwarp();
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      fence_after();
      float s[HK];
#pragma unroll
      for (int q = 0; q < HK / 32; ++q)
        tmem_ld32(tl + (j & 1) * AT_BN + hf * HK + q * 32, reinterpret_cast<uint32_t*>(s + q * 32));
      const int k0 = j * AT_BN + hf * HK;
      if (k0 + HK - 1 > q_pos) {  // causal mask near the diagonal
#pragma unroll
        for (int k = 0; k < HK; ++k)
          if (k0 + k > q_pos) s[k] = -CUDART_INF_F;
      }
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < HK; ++k) mx = fmaxf(mx, s[k]);
      red[hf * 128 + r] = mx;
      pair_sync(qd);
      const float t_max = fmaxf(red[r], red[128 + r]) * c;
      pair_sync(qd);  // both halves have read the maxima before they are overwritten
      // Lazy rescaling: the exponent reference m moves only when the tile's
      // maximum exceeds it by more than 2^8, so probabilities stay below 256
      // and the accumulator is rarely touched; O / l is unchanged by the
      // choice of m.  (Both halves take the same decision from the same maxima.)
      const bool move = t_max > m + 8.f;
      const float m_use = move ? t_max : m;
      const float alpha = move ? ex2(m - m_use) : 1.f;  // 0 on the first tile
#pragma unroll
      for (int k = 0; k < HK; ++k) s[k] = ex2(fmaf(s[k], c, -m_use));
      // P = hi + lo: hi = P with its low 16 bits cleared (a bf16 value),
      // lo = P - hi (exact) likewise truncated, so hi + lo carries 16
      // significant bits; l sums exactly the values the MMAs use.
      float sum = 0.f;
      uint32_t ph[HK / 2], pl[HK / 2];
#pragma unroll
      for (int k = 0; k < HK; k += 2) {
        const uint32_t h0 = __float_as_uint(s[k]) & 0xffff0000u, h1 = __float_as_uint(s[k + 1]) & 0xffff0000u;
        const uint32_t l0 = __float_as_uint(s[k] - __uint_as_float(h0)) & 0xffff0000u;
        const uint32_t l1 = __float_as_uint(s[k + 1] - __uint_as_float(h1)) & 0xffff0000u;
        sum += (__uint_as_float(h0) + __uint_as_float(l0)) + (__uint_as_float(h1) + __uint_as_float(l1));
        ph[k / 2] = __byte_perm(h0, h1, 0x7632);
        pl[k / 2] = __byte_perm(l0, l1, 0x7632);
      }
      l = l * alpha + sum;
      if (j > 0) {  // P.V of the previous tile must be done: it reads P and accumulates into O
        int oko = ok;
        if (lane == 0 && ok) oko = mbar_wait(o_done, (uint32_t)((j - 1) & 1), a.err, 11);
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, oko, 0) != 0;
        fence_after();
        if (ok && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int q = 0; q < HD / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(tl + AT_O_COL + hf * HD + q * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tl + AT_O_COL + hf * HD + q * 32, o);
          }
          tmem_wait_st();
        }
      }
      // row r of this half's P blocks (128-byte swizzle: 16-byte chunk cc of
      // row r sits at chunk cc ^ (r & 7) of its 128-byte line)
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint32_t off = (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(Ph + off) = make_uint4(ph[cc * 4], ph[cc * 4 + 1], ph[cc * 4 + 2], ph[cc * 4 + 3]);
        *reinterpret_cast<uint4*>(Pl + off) = make_uint4(pl[cc * 4], pl[cc * 4 + 1], pl[cc * 4 + 2], pl[cc * 4 + 3]);
      }
      // Last tile: its value rows past the block's last key hold whatever the
      // cache held there; their probabilities are 0, but 0 * (a non-finite
      // value) is not 0 in the P.V product, so those rows are zeroed first
      // (half hf clears column block hf; a whole 128-byte row is the same row
      // under the swizzle).  The tile has landed: S of this tile was computed.
      const int last_key = qb.pos0 + qb.nrows - 1;
      if (j == n_tiles - 1 && j * AT_BN + AT_BN - 1 > last_key && hf < L::NC) {
        const int st = j % AT_STAGES;
        if (ok && lane == 0) mbar_wait(&kv_full[st], (uint32_t)((j / AT_STAGES) & 1), a.err, 13);
        __syncwarp();
        for (int c = hf; c < L::NC; c += 2) {
          if (j * AT_BN + r > last_key) {
            uint4* vrow = reinterpret_cast<uint4*>(smem + L::KV_OFF + st * L::STAGE + (L::NC + c) * L::SUB +
                                                   (size_t)r * 128);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) vrow[cc] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async();  // P's (and zeroed V rows') generic-proxy stores before the MMA's reads
      fence_before();
      mbar_arrive_cta(p_full);
      m = m_use;
    }
    if (ok) {
      int oko = 1;
      if (lane == 0) oko = mbar_wait(o_done, (uint32_t)((n_tiles - 1) & 1), a.err, 12);
      __syncwarp();
      ok = __shfl_sync(0xffffffffu, oko, 0) != 0;
    }
    // (both halves reach this exchange, failed or not, so the pair barrier matches)
    red[hf * 128 + r] = l;
    pair_sync(qd);
    const float inv = 1.f / (red[r] + red[128 + r]);
    if (ok) {
      fence_after();
      bf16* dst = static_cast<bf16*>(a.out) + (size_t)(qb.row0 + r) * a.H * D + (size_t)h * D + hf * HD;
#pragma unroll
      for (int q = 0; q < HD / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(tl + AT_O_COL + hf * HD + q * 32, o);
        if (r < qb.nrows) {
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(o[i]) * inv;
#pragma unroll
          for (int v = 0; v < 4; ++v) reinterpret_cast<uint4*>(dst + q * 32)[v] = Vec16<bf16>::pack(f + 8 * v);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == AT_MMA_WARP) {
    fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

template <int D>
cudaError_t at_launch(const LaunchCtx& c, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const AttnTcArgs& a) {
  auto kern = attn_tc_kernel<D>;
  cudaError_t e = set_max_smem((const void*)kern, (int)ATL<D>::SMEM);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(a.n_qblocks * a.H), dim3(AT_THREADS), ATL<D>::SMEM, c, mq, mk, mv, a);
}

}  // namespace

bool attn_tc_supported(int D) { return (D == 64 || D == 128) && encode_fn() != nullptr; }
int attn_tc_rows() { return AT_BM; }

cudaError_t launch_attn_tc(const LaunchCtx& c, const AttnTcArgs& a) {
  if (!attn_tc_supported(a.D) || a.n_qblocks < 1 || a.T < 1) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  const uint64_t qd[2] = {(uint64_t)a.H * a.D, (uint64_t)a.T};
  const uint64_t qs[1] = {(uint64_t)a.H * a.D * 2};
  const uint64_t kd[3] = {(uint64_t)a.D, (uint64_t)a.KV * a.capacity, (uint64_t)a.max_seqs};
  const uint64_t ks[2] = {(uint64_t)a.D * 2, (uint64_t)a.seq_stride * 2};
  if (!make_map_bf16(&mq, a.q, 2, qd, qs, AT_BM) || !make_map_bf16(&mk, a.kc, 3, kd, ks, AT_BN) ||
      !make_map_bf16(&mv, a.vc, 3, kd, ks, AT_BN))
    return cudaErrorInvalidValue;
  return a.D == 128 ? at_launch<128>(c, mq, mk, mv, a) : at_launch<64>(c, mq, mk, mv, a);
}

}  // namespace q3
