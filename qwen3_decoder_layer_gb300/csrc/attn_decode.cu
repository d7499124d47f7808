// Decode attention over the static KV cache with the per-head q/k RMSNorm,
// RoPE and cache append fused in (maya2_mlx/backbone.py, Backbone.forward:
// "q, k = per-head RMSNorm (two roundings), RoPE in fp32 on the cos/sin
// table, attention over keys 0..pos (fp32 softmax, one rounding)"; GQA as the
// repeat_kv of rlx_flow/blocks/qwen3_decoder.rs).
//
// Split-K ("flash-decoding"): the keys of each query block (rows of one
// sequence, x G query heads of kv head j) are cut into chunks of SUBS
// sub-chunks of CK keys.  A work item is one (query block, chunk, kv head);
// each block of the grid walks a contiguous range of the item list (kv head
// on y), so that most consecutive items continue the same query block.
//
// Warp-specialised block.  One producer warp streams the sub-chunks of the
// block's items, in order, into a 4-stage shared-memory ring (one item) with
// TMA bulk copies (full / empty mbarriers).  It reads only cached positions,
// which no kernel in flight writes, so it starts at launch without waiting
// for the qkv projection.  Sixteen consumer warps: warps 0..NQ-1 first
// normalise and rotate the NQ query vectors of the item; then every warp
// takes its own CK/4 keys of one sub-chunk and runs them end to end -- keys
// appended in this call computed from the qkv row (and stored to the cache
// by the item owning the row), scores, a warp-local softmax, P.V -- with no
// block barrier, producing a warp partial (m, l, o).  A block barrier, one
// merge of the 16 partials per RUN of consecutive items of one query block
// (queries staged once per run, each warp carrying its online-softmax state
// (m, l, o) across the run), and the run's partial goes to global memory.
// The last run of a (query block, kv head) -- found with an atomic counter,
// no waiting -- merges the runs: M = max m_c,
// out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c, rounded once to the
// model dtype.
#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace q3 {

namespace {

using namespace dec;

constexpr int AD_CWARPS = 16;                    // consumer warps
constexpr int AD_CTHREADS = AD_CWARPS * 32;      // 512
constexpr int AD_THREADS = AD_CTHREADS + 32;     // + producer warp
constexpr int AD_NQ_MAX = 8;
constexpr int AD_SUBS = 4;                       // sub-chunks per item
constexpr int AD_STAGES_MAX = 6;                 // ring stages (one sub-chunk each), at most
constexpr int AD_WPS = AD_CWARPS / AD_SUBS;      // warps per sub-chunk

template <typename Dt> struct ADT {
  static constexpr int CK = sizeof(Dt) == 2 ? 64 : 32;  // 16 KB per K or V sub-chunk at head_dim 128
};

template <typename Dt, int D, int NQ> struct ADLayout {
  static constexpr int CK = ADT<Dt>::CK;
  static constexpr int KW = CK / AD_WPS;  // keys per warp
  static constexpr size_t TILE = (size_t)CK * D * sizeof(Dt);
  static constexpr size_t STAGE = 2 * TILE;
  // ring stages: one item (AD_SUBS stages), plus two when shared memory
  // allows, so that a block's next item streams in while this one computes
  static constexpr int STAGES = NQ <= 2 ? AD_STAGES_MAX : AD_SUBS;
  static constexpr size_t OFF_QS = STAGES * STAGE;                                // [NQ][D] queries
  static constexpr size_t OFF_PS = OFF_QS + (size_t)NQ * D * 4;                   // [warp][NQ][KW] scores / p
  static constexpr int WPITCH = D + 4;                                            // o[D], m, l, pad
  static constexpr size_t OFF_WP = OFF_PS + (size_t)AD_CWARPS * NQ * KW * 4;      // [warp][NQ][WPITCH] partials
  static constexpr size_t WP_FLOATS = (size_t)AD_CWARPS * NQ * WPITCH;
  static constexpr int MPITCH = AD_CWARPS + 2;                                    // weights of the warps, M, L
  static constexpr size_t OFF_MRG = OFF_WP + WP_FLOATS * 4;                       // [NQ][MPITCH] merge scratch
  static constexpr size_t OFF_BAR = (OFF_MRG + (size_t)NQ * MPITCH * 4 + 15) & ~size_t(15);
  static constexpr size_t TOTAL = OFF_BAR + 2 * STAGES * 8 + 16 + 1024;  // + slack to align the base to 1024
  // cluster variant: this CTA's merged partial [NQ][D + 2] (o, then m and l),
  // and what the other CTAs of the cluster (up to 16, at least 8) push to it:
  // their m [16][NQ], l [16][NQ] and values of this CTA's output slice
  // [16][RX_SHARE]
  static constexpr int CPITCH = D + 2;
  static constexpr size_t OFF_CP = (TOTAL + 15) & ~size_t(15);
  static constexpr int RX_SHARE = (NQ * D + 7) / 8;
  static constexpr size_t OFF_RX = (OFF_CP + (size_t)NQ * CPITCH * 4 + 15) & ~size_t(15);
  static constexpr size_t RX_FLOATS = (size_t)16 * (2 * NQ + RX_SHARE);
  static constexpr size_t TOTAL_CL = OFF_RX + RX_FLOATS * 4 + 1024;
  static_assert(TOTAL_CL <= 227 * 1024, "cluster-kernel shared memory exceeds 227 KB");
};

// A K or V tile in shared memory as the TMA writes it: each cached position's
// row of D elements is R = D * sizeof(Dt) / 128 consecutive 128-byte lines
// (the tile is one contiguous piece of the cache, one copy), and the 16-byte
// chunk c of line L sits at chunk c ^ (L & 7) of that line (128-byte
// swizzle: row-wise 16-byte accesses of a warp, e.g. ldmatrix over 8 rows,
// spread over the bank groups).  p: the warp's first row (a multiple of 8
// lines into the 1024-byte aligned tile).
// (SWZ = false: the rows as they lie in the cache, unswizzled, filled by bulk
// copies of the valid keys only; the CUDA-core warp form reads whole rows of
// consecutive lanes and has no bank conflicts there.)
template <typename Dt, int D, bool SWZ>
struct KVT {
  static constexpr int R = D * (int)sizeof(Dt) / 128;
  uint8_t* p;
  __device__ __forceinline__ uint8_t* chunk(int r, int c) const {
    if (!SWZ) return p + r * (D * (int)sizeof(Dt)) + c * 16;
    const int line = r * R + (c >> 3);
    return p + line * 128 + (((c & 7) ^ (line & 7)) << 4);
  }
  // element e of row r; the elements after it up to the end of its 16-byte chunk follow it
  __device__ __forceinline__ Dt* elem(int r, int e) const {
    const int off = e * (int)sizeof(Dt);
    return reinterpret_cast<Dt*>(chunk(r, off >> 4) + (off & 15));
  }
};
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
// The K and V tiles of CK cached positions from row `row` (kv head x capacity
// + position) of sequence `seq`, one tensor load each, completing on `bar`.
// The box is always whole: lines past the valid keys hold other cache
// contents or zeros, and are masked.
template <typename Dt, int D>
__device__ __forceinline__ void load_kv_tiles(uint8_t* stage, const CUtensorMap* mk, const CUtensorMap* mv, int row,
                                              int seq, uint64_t* bar) {
  constexpr int CK = ADT<Dt>::CK, R = D * (int)sizeof(Dt) / 128;
  constexpr uint32_t TILE = (uint32_t)CK * D * sizeof(Dt);
  mbar_expect_tx(bar, 2 * TILE);
  tc::tma_load_3d(stage, mk, 0, row * R, seq, bar);
  tc::tma_load_3d(stage + TILE, mv, 0, row * R, seq, bar);
}

// Named barrier over the consumer warps only.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(AD_CTHREADS) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Thread-block cluster: rank of this CTA, CTAs in the cluster, a barrier over
// every thread of the cluster (release / acquire), and loads from another
// CTA's shared memory (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_cluster(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// L2 prefetch of this block's share of [p, p + bytes) over the whole grid.
__device__ __forceinline__ void prefetch_grid_share(const void* p, size_t bytes) {
  if (!p || !bytes) return;
  const int nb = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
  const size_t per = ((bytes + nb - 1) / nb + 15) & ~size_t(15);
  for (size_t b0 = per * b, b1 = min(per * (b + 1), bytes); b0 < b1; b0 += 65536)
    prefetch_l2(static_cast<const char*>(p) + b0, (uint32_t)min(b1 - b0, (size_t)65536));
}

// Keys of an item: [key0, key0 + nkeys) in nsub sub-chunks.
struct ItemKeys {
  int key0, nkeys, nsub;
};
template <typename Dt>
__device__ __forceinline__ ItemKeys item_keys(const AttnItem& item, const AttnQBlock& qb) {
  constexpr int CK = ADT<Dt>::CK;
  ItemKeys r;
  r.key0 = item.chunk * CK * AD_SUBS;
  r.nkeys = min(CK * AD_SUBS, qb.pos0 + qb.nrows - r.key0);
  r.nsub = (r.nkeys + CK - 1) / CK;
  return r;
}

// Sum over the LPK lanes of a key group of each lane's NS per-step partial
// dot products, as a reduce-scatter: at each halving the lane pair keeps
// opposite halves of its remaining steps and adds the partner's copy, so
// NS - 1 shuffles leave each lane the full sum of step sub_l / (LPK / NS);
// the lanes that share that step then add among themselves.
template <int NS, int LPK>
__device__ __forceinline__ float rs_sum(float (&v)[NS], int sub_l) {
#pragma unroll
  for (int c = NS, h = LPK / 2; c > 1; c >>= 1, h >>= 1) {
    const bool up = (sub_l & h) != 0;
#pragma unroll
    for (int k = 0; k < c / 2; ++k) {
      const float send = up ? v[k] : v[k + c / 2];
      const float keep = up ? v[k + c / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, h);
    }
  }
  float r = v[0];
#pragma unroll
  for (int h = LPK / (2 * NS); h >= 1; h >>= 1) r += __shfl_xor_sync(0xffffffffu, r, h);
  return r;
}

// A warp's nk keys (rows of Kt, first absolute position kb) against the nq
// staged queries: scores (scaled, causally masked at pos0 + i / G), folded
// into the warp's running softmax state (m, l and o rescaled) and left as
// probabilities in ps[i * KW + u] for the P.V pass.  LPK lanes share a key
// (EPV elements each), KPS keys per step.  Up to four queries: every lane
// keeps its partial dot product of each step and the partials are summed
// across the key group once, after the last step (rs_sum); the queries sit
// in registers when there are at most two.  Eight queries: one butterfly per
// (step, query), the registers being needed for the state.
template <typename Dt, int D, int NQ, int KW>
__device__ __forceinline__ void warp_scores_softmax(KVT<Dt, D, false> Kt, const float* qs, float* ps, int nk, int nq, int kb,
                                                    int pos0, int G, float scale, float (&m_w)[NQ], float (&l_w)[NQ],
                                                    float (&o_w)[NQ][D / 32]) {
  constexpr int EPV = 16 / sizeof(Dt);
  constexpr int LPK = D / EPV;
  constexpr int KPS = 32 / LPK;
  constexpr int NS = KW / KPS;
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31, sub_l = lane % LPK, kq = lane / LPK;
  if constexpr (NQ <= 4) {
    static_assert(NS <= LPK && (NS & (NS - 1)) == 0, "steps per key group");
    constexpr bool QREG = NQ <= 2;
    float qr[QREG ? NQ : 1][EPV];
    if constexpr (QREG) {
#pragma unroll
      for (int i = 0; i < NQ; ++i)
#pragma unroll
        for (int e = 0; e < EPV / 4; ++e) {
          const float4 q4 = reinterpret_cast<const float4*>(qs + i * D + sub_l * EPV)[e];
          qr[i][4 * e] = q4.x; qr[i][4 * e + 1] = q4.y; qr[i][4 * e + 2] = q4.z; qr[i][4 * e + 3] = q4.w;
        }
    }
    float dp[NQ][NS];
#pragma unroll
    for (int st = 0; st < NS; ++st) {
      const int u = st * KPS + kq;
      float kv[EPV];
      if (u < nk) {
        Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(Kt.chunk(u, sub_l)), kv);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) kv[e] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int e = 0; e < EPV / 4; ++e) {
          float4 q4;
          if constexpr (QREG) {
            q4 = make_float4(qr[i][4 * e], qr[i][4 * e + 1], qr[i][4 * e + 2], qr[i][4 * e + 3]);
          } else {
            q4 = reinterpret_cast<const float4*>(qs + i * D + sub_l * EPV)[e];
          }
          d0 = fmaf(q4.x, kv[4 * e], d0);
          d1 = fmaf(q4.y, kv[4 * e + 1], d1);
          d0 = fmaf(q4.z, kv[4 * e + 2], d0);
          d1 = fmaf(q4.w, kv[4 * e + 3], d1);
        }
        dp[i][st] = d0 + d1;
      }
    }
    // lane (kq, sub_l) now reduces to the score of key u; LPK / NS lanes hold each key
    const int u = (sub_l / (LPK / NS)) * KPS + kq;
    const bool first = (sub_l % (LPK / NS)) == 0;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      float sv = rs_sum<NS, LPK>(dp[i], sub_l);
      sv = (u < nk && i < nq && kb + u <= pos0 + i / G) ? sv * scale : -CUDART_INF_F;
      const float m_new = fmaxf(m_w[i], warp_max(sv));
      const float p = (sv == -CUDART_INF_F) ? 0.f : expf(sv - m_new);
      const float alpha = (m_w[i] == -CUDART_INF_F) ? 0.f : expf(m_w[i] - m_new);
      const float ls = warp_sum(first ? p : 0.f);
      if (first) ps[i * KW + u] = p;
      if (m_new != -CUDART_INF_F) {
        l_w[i] = fmaf(l_w[i], alpha, ls);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o_w[i][e] *= alpha;
        m_w[i] = m_new;
      }
    }
    __syncwarp();
  } else {
#pragma unroll
    for (int st = 0; st < NS; ++st) {
      const int u = st * KPS + kq;
      float kv[EPV];
      if (u < nk) {
        Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(Kt.chunk(u, sub_l)), kv);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) kv[e] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const float4* qp = reinterpret_cast<const float4*>(qs + i * D + sub_l * EPV);
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int e = 0; e < EPV / 4; ++e) {
          const float4 q4 = qp[e];
          d0 = fmaf(q4.x, kv[4 * e], d0);
          d1 = fmaf(q4.y, kv[4 * e + 1], d1);
          d0 = fmaf(q4.z, kv[4 * e + 2], d0);
          d1 = fmaf(q4.w, kv[4 * e + 3], d1);
        }
        float d = d0 + d1;
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (sub_l == 0) ps[i * KW + u] = (u < nk && i < nq && kb + u <= pos0 + i / G) ? d * scale : -CUDART_INF_F;
      }
    }
    __syncwarp();
    // online softmax update of the warp's running state (lanes over keys)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const float sv = lane < KW ? ps[i * KW + lane] : -CUDART_INF_F;
      const float mx = warp_max(sv);
      const float m_new = fmaxf(m_w[i], mx);
      const float p = (sv == -CUDART_INF_F) ? 0.f : expf(sv - m_new);
      const float alpha = (m_w[i] == -CUDART_INF_F) ? 0.f : expf(m_w[i] - m_new);
      const float ls = warp_sum(p);
      if (lane < KW) ps[i * KW + lane] = p;
      if (m_new != -CUDART_INF_F) {
        l_w[i] = fmaf(l_w[i], alpha, ls);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o_w[i][e] *= alpha;
        m_w[i] = m_new;
      }
    }
    __syncwarp();
  }
}

// A warp's online-softmax state over its keys and its partial (m, l, o) for
// the merge.  Two forms with the same interface:
//  * WarpAttnSimt: CUDA cores (every dtype); scores as above, then P.V with
//    lane l holding head elements l*D/32 .. +D/32 of every query.
//  * WarpAttnMma: bf16 with 4 or 8 query vectors (GQA groups of 4-8 heads, or
//    several rows of a sequence), where the per-key work is a small dense
//    product: S^T[16 keys x 8 queries] = K Q^T and O^T[D x 8] += V^T P^T on
//    warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in, fp32
//    accumulate; bf16 products are exact in fp32).  P enters the MMA as three
//    bf16 parts hi + mid + lo, which hold all 24 bits of the fp32
//    probability, so P.V keeps the accuracy of the CUDA-core form.  Lane L holds
//    queries 2(L%4), 2(L%4)+1: its scores for keys L/4 and L/4+8, and its
//    output columns t*16 + L/4 (+8) of every 16-dim tile t.
template <typename Dt, int D, int NQ, int KW>
struct WarpAttnSimt {
  static constexpr bool kSwizzled = false;  // reads K / V tiles as the cache lays them out
  static constexpr int DPL = D / 32;
  float m[NQ], l[NQ], o[NQ][DPL];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      m[i] = -CUDART_INF_F;
      l[i] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[i][e] = 0.f;
    }
  }
  __device__ __forceinline__ void load_q(const float*, int) {}
  __device__ __forceinline__ void attend(KVT<Dt, D, false> Kt, KVT<Dt, D, false> Vt, const float* qs, float* ps, int nk, int nq, int kb,
                                         int pos0, int G, float scale) {
    const int lane = threadIdx.x & 31;
    warp_scores_softmax<Dt, D, NQ, KW>(Kt, qs, ps, nk, nq, kb, pos0, G, scale, m, l, o);
#pragma unroll 4
    for (int u = 0; u < nk; ++u) {
      float v[DPL];
      load_lane_vec<Dt, DPL>(Vt.elem(u, lane * DPL), v);
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const float p = ps[i * KW + u];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[i][e] = fmaf(p, v[e], o[i][e]);
      }
    }
  }
  // partial of this warp -> mine[i * pitch + d] (o), [D] (m), [D + 1] (l)
  __device__ __forceinline__ void store(float* mine, int pitch) const {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      store_lane_vec<DPL>(mine + i * pitch + lane * DPL, o[i]);
      if (lane == 0) { mine[i * pitch + D] = m[i]; mine[i * pitch + D + 1] = l[i]; }
    }
  }
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// two fp32 values that are bf16 values -> one bf16x2 word (first in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

template <int D, int NQ>
struct WarpAttnMma {
  static constexpr bool kSwizzled = true;  // reads K / V tiles 128-byte swizzled (ldmatrix over 8 rows)
  static constexpr int NT = D / 16;  // 16-dim tiles (k-steps of the scores, m-tiles of the output)
  float m[2], l[2];
  float o[NT][4];
  uint32_t qf[NT][2];                // B fragments of Q^T, per 16-dim k-step
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int j = 0; j < 2; ++j) { m[j] = -CUDART_INF_F; l[j] = 0.f; }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[t][e] = 0.f;
  }
  // Q^T fragments from the staged queries (fp32 values of bf16 numbers: exact)
  __device__ __forceinline__ void load_q(const float* qs, int nq) {
    const int lane = threadIdx.x & 31, n = lane >> 2, c = (lane & 3) * 2;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (n < nq) {
        const float* q = qs + n * D + t * 16 + c;
        qf[t][0] = pack_bf16x2(q[0], q[1]);
        qf[t][1] = pack_bf16x2(q[8], q[9]);
      } else {
        qf[t][0] = qf[t][1] = 0u;
      }
    }
  }
  __device__ __forceinline__ void attend(KVT<__nv_bfloat16, D, true> Kt, KVT<__nv_bfloat16, D, true> Vt, const float*, float*, int nk, int nq,
                                         int kb, int pos0, int G, float scale) {
    const int lane = threadIdx.x & 31, r0 = lane >> 2, q0 = (lane & 3) * 2;
    // value rows past this warp's keys hold whatever the stage held: zero them
    // (their probabilities are 0, but 0 * a non-finite value is not)
    if (nk < 16) {
      for (int c = lane; c < (16 - nk) * (D / 8); c += 32)
        *reinterpret_cast<uint4*>(Vt.chunk(nk + c / (D / 8), c % (D / 8))) = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
    }
    // S^T = K Q^T: rows = keys r0, r0 + 8; columns = queries q0, q0 + 1
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;  // ldmatrix row of this lane
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint32_t a[4];
      ldsm_x4(a, Kt.chunk(mrow, t * 2 + mcol / 8));
      mma_bf16_16816(s, a, qf[t][0], qf[t][1]);
    }
    float mx[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int q = q0 + j;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = r0 + 8 * h;
        const bool ok = k < nk && q < nq && kb + k <= pos0 + q / G;
        s[2 * h + j] = ok ? s[2 * h + j] * scale : -CUDART_INF_F;
      }
      float v = fmaxf(s[j], s[2 + j]);
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      mx[j] = v;
    }
    // probabilities (fp32)
    float p[4], alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float m_new = fmaxf(m[j], mx[j]);
      alpha[j] = (m[j] == -CUDART_INF_F) ? 0.f : expf(m[j] - m_new);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        p[2 * h + j] = (s[2 * h + j] == -CUDART_INF_F) ? 0.f : expf(s[2 * h + j] - m_new);
      float sum = p[j] + p[2 + j];
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      sum += __shfl_xor_sync(0xffffffffu, sum, 8);
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      if (m_new != -CUDART_INF_F) {
        l[j] = fmaf(l[j], alpha[j], sum);
        m[j] = m_new;
      } else {
        alpha[j] = 1.f;
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      o[t][0] *= alpha[0]; o[t][2] *= alpha[0];
      o[t][1] *= alpha[1]; o[t][3] *= alpha[1];
    }
    // P^T as the B operand: lane L needs P[query L/4][keys 2(L%4), +1, +8, +9],
    // held by lanes 8(L%4) + (L/4)/2 (keys 2(L%4), +8) and that + 4 (the odd keys)
    const int src = (lane & 3) * 8 + (lane >> 3);
    const int par = (lane >> 2) & 1;  // which of the source's two queries
    float g[2][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      g[0][e] = __shfl_sync(0xffffffffu, p[e], src);
      g[1][e] = __shfl_sync(0xffffffffu, p[e], src + 4);
    }
    const float pk0 = par ? g[0][1] : g[0][0], pk1 = par ? g[1][1] : g[1][0];
    const float pk8 = par ? g[0][3] : g[0][2], pk9 = par ? g[1][3] : g[1][2];
    // p = hi + mid + lo exactly: each part the top 8 significant bits of what
    // is left (the differences are exact in fp32)
    auto top = [](float v) { return __uint_as_float(__float_as_uint(v) & 0xffff0000u); };
    const float h0 = top(pk0), h1 = top(pk1), h8 = top(pk8), h9 = top(pk9);
    const float m0 = top(pk0 - h0), m1 = top(pk1 - h1), m8 = top(pk8 - h8), m9 = top(pk9 - h9);
    const uint32_t bh0 = pack_bf16x2(h0, h1), bh1 = pack_bf16x2(h8, h9);
    const uint32_t bm0 = pack_bf16x2(m0, m1), bm1 = pack_bf16x2(m8, m9);
    const uint32_t bl0 = pack_bf16x2(pk0 - h0 - m0, pk1 - h1 - m1);
    const uint32_t bl1 = pack_bf16x2(pk8 - h8 - m8, pk9 - h9 - m9);
    // O^T += V^T P^T: A = V^T tile (16 dims x 16 keys) by a transposing ldmatrix
    const int vrow = (lane & 7) + (lane >> 4) * 8, vcol = ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint32_t a[4];
      ldsm_x4_t(a, Vt.chunk(vrow, t * 2 + vcol / 8));
      mma_bf16_16816(o[t], a, bh0, bh1);
      mma_bf16_16816(o[t], a, bm0, bm1);
      mma_bf16_16816(o[t], a, bl0, bl1);
    }
  }
  __device__ __forceinline__ void store(float* mine, int pitch) const {
    const int lane = threadIdx.x & 31, r0 = lane >> 2, q0 = (lane & 3) * 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int q = q0 + j;
      if (q >= NQ) continue;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        mine[q * pitch + t * 16 + r0] = o[t][j];
        mine[q * pitch + t * 16 + r0 + 8] = o[t][2 + j];
      }
      if (r0 == 0) { mine[q * pitch + D] = m[j]; mine[q * pitch + D + 1] = l[j]; }
    }
  }
};

// The warp state a kernel instance uses.
template <typename Dt, int D, int NQ, int KW>
struct WarpAttnOf {
  using type = WarpAttnSimt<Dt, D, NQ, KW>;
};
template <int D, int NQ>
struct WarpAttnOf<__nv_bfloat16, D, NQ, 16> {
  using type = typename std::conditional<(NQ >= 4), WarpAttnMma<D, NQ>, WarpAttnSimt<__nv_bfloat16, D, NQ, 16>>::type;
};

// The last block to finish a (query block, kv head) combines its nc chunk
// partials: M = max m_c, out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c,
// rounded once to the model dtype.  Every partial is first loaded into
// shared memory in one pass of independent loads (m, l into wp; o into
// `ostage` when given, which must hold nc * nq * D floats), so that the
// combine costs one round trip to L2 rather than one per chunk.
template <typename Dt, int D, int NQ>
__device__ void combine_parts(const AttnDecArgs& a, const AttnQBlock& qb, int j, int nc, int nq, int G, float* wp,
                              float* mrg, float* ostage) {
  using LY = ADLayout<Dt, D, NQ>;
  constexpr int MP = LY::MPITCH;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t pbase = (size_t)qb.part_base * a.KV + j;  // partial of chunk c: (pbase + c * KV) * nq_max
  auto pidx = [&](int c, int i) { return (pbase + (size_t)c * a.KV) * a.nq_max + i; };
  const bool staged = 2 * (size_t)nc * nq <= LY::WP_FLOATS;
  float* fm = wp;            // [c][i]: chunk maxima, then their weights e^(m_c - M_i)
  float* fl = wp + nc * nq;  // [c][i]: chunk normalisers
  __threadfence();
  if (staged) {
    for (int idx = tid; idx < nc * nq; idx += AD_CTHREADS) {
      const int c = idx / nq, i = idx % nq;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + pidx(c, i));
      fm[idx] = ml.x;
      fl[idx] = ml.y;
    }
  }
  if (ostage) {
    const int per = nq * D / 4;  // float4 per chunk (queries of one chunk are contiguous)
    for (int idx = tid; idx < nc * per; idx += AD_CTHREADS) {
      const int c = idx / per, r = idx - c * per;
      reinterpret_cast<float4*>(ostage)[idx] = __ldcg(reinterpret_cast<const float4*>(a.part_o + pidx(c, 0) * D) + r);
    }
  }
  csync();
  // per-query max and normaliser (warp per query, lanes over chunks)
  for (int i = warp; i < nq; i += AD_CWARPS) {
    auto mval = [&](int c) { return staged ? fm[c * nq + i] : __ldcg(a.part_ml + pidx(c, i) * 2); };
    auto lval = [&](int c) { return staged ? fl[c * nq + i] : __ldcg(a.part_ml + pidx(c, i) * 2 + 1); };
    float M = -CUDART_INF_F;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, mval(c));
    M = warp_max(M);
    float Lsum = 0.f;
    for (int c = lane; c < nc; c += 32) {
      const float m = mval(c);
      const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
      Lsum = fmaf(lval(c), f, Lsum);
      if (staged) fm[c * nq + i] = f;
    }
    Lsum = warp_sum(Lsum);
    if (lane == 0) { mrg[i * MP + AD_CWARPS] = M; mrg[i * MP + AD_CWARPS + 1] = Lsum; }
  }
  csync();
  // out[i][d] = sum_c f[c][i] o_c[i][d] / L_i, one thread per output element
  for (int idx = tid; idx < nq * D; idx += AD_CTHREADS) {
    const int i = idx / D, d = idx % D;
    const float M = mrg[i * MP + AD_CWARPS];
    float v = 0.f;
#pragma unroll 4
    for (int c = 0; c < nc; ++c) {
      float f;
      if (staged) {
        f = fm[c * nq + i];
      } else {
        const float m = __ldcg(a.part_ml + pidx(c, i) * 2);
        f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
      }
      v = fmaf(ostage ? ostage[(size_t)c * nq * D + idx] : __ldcg(a.part_o + pidx(c, i) * D + d), f, v);
    }
    const int row = qb.row0 + i / G, head = j * G + i % G;
    static_cast<Dt*>(a.out)[((size_t)row * a.H + head) * D + d] = from_f<Dt>(v / mrg[i * MP + AD_CWARPS + 1]);
  }
}

template <typename Dt, int D, int NQ>
__global__ void __launch_bounds__(AD_THREADS, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, AttnDecArgs a) {
  extern __shared__ __align__(128) uint8_t ad_smem_raw[];
  uint8_t* ad_smem = align1024(ad_smem_raw);  // the K/V tiles' swizzle is relative to 1024-byte blocks
  using LY = ADLayout<Dt, D, NQ>;
  constexpr int CK = LY::CK;
  constexpr int KW = LY::KW;
  constexpr bool SWZ = WarpAttnOf<Dt, D, NQ, KW>::type::kSwizzled;  // K / V tiles swizzled (tensor loads)            // keys per warp
  constexpr int DPL = D / 32;           // head elements per lane
  constexpr int WP = LY::WPITCH;
  constexpr int MP = LY::MPITCH;
  float* qs = reinterpret_cast<float*>(ad_smem + LY::OFF_QS);
  float* ps_all = reinterpret_cast<float*>(ad_smem + LY::OFF_PS);
  float* wp = reinterpret_cast<float*>(ad_smem + LY::OFF_WP);
  float* mrg = reinterpret_cast<float*>(ad_smem + LY::OFF_MRG);
  uint64_t* full = reinterpret_cast<uint64_t*>(ad_smem + LY::OFF_BAR);
  uint64_t* empty = full + LY::STAGES;
  __shared__ int s_flag, s_fail;
  __shared__ int s_issued[AD_STAGES_MAX];  // uses of each stage issued so far
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int qkv_ld = (a.H + 2 * a.KV) * D;
  const int n_items = *a.n_items;
  auto tiles = [&](int s) { return ad_smem + (size_t)s * LY::STAGE; };

  if (tid == 0) {
    for (int s = 0; s < LY::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], AD_WPS);
    }
    mbar_fence_init();
    s_fail = 0;
  }
  if (tid < LY::STAGES) s_issued[tid] = 0;
  __syncthreads();

  if (warp == AD_CWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int g = 0;
      // at most one item per block: item x; else the contiguous range (as the consumers)
      const int it_lo = n_items <= (int)gridDim.x ? (int)blockIdx.x
                                                  : (int)(blockIdx.x * (unsigned)n_items / gridDim.x);
      const int it_hi = n_items <= (int)gridDim.x ? min((int)blockIdx.x + 1, n_items)
                                                  : (int)((blockIdx.x + 1) * (unsigned)n_items / gridDim.x);
      for (int it = it_lo; it < it_hi; ++it) {
        const AttnItem item = a.items[it];
        const AttnQBlock qb = a.qblocks[item.qb];
        const ItemKeys ik = item_keys<Dt>(item, qb);
        for (int sub = 0; sub < ik.nsub; ++sub, ++g) {
          const int s = g % LY::STAGES;
          if (g >= LY::STAGES && !mbar_wait(&empty[s], (uint32_t)((g / LY::STAGES - 1) & 1), a.err, 2)) {
            s_fail = 1;
            return;
          }
          const int k0 = ik.key0 + sub * CK;
          if constexpr (SWZ) {
            load_kv_tiles<Dt, D>(tiles(s), &map_k, &map_v, j * a.capacity + k0, qb.seq, &full[s]);
          } else {
            const int nk = min(CK, ik.key0 + ik.nkeys - k0);
            const size_t off = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + k0) * D;
            const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
            mbar_expect_tx(&full[s], 2 * bytes);
            tma_load_1d(tiles(s), static_cast<const Dt*>(a.kc) + off, bytes, &full[s]);
            tma_load_1d(tiles(s) + LY::TILE, static_cast<const Dt*>(a.vc) + off, bytes, &full[s]);
          }
          *(volatile int*)&s_issued[s] = g / LY::STAGES + 1;
        }
      }
      // L2 prefetch of this block's share of the next kernels' operands
      prefetch_grid_share(a.pf, a.pf_bytes);
      prefetch_grid_share(a.pf2, a.pf2_bytes);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch();
  const Dt* qkv = static_cast<const Dt*>(a.qkv);
  float* ps = ps_all + (size_t)warp * NQ * KW;  // this warp's scores / probabilities
  const int wsub = warp / AD_WPS;               // sub-chunk of this warp
  const int wk0 = (warp % AD_WPS) * KW;         // its first key inside the sub-chunk
  int g = 0;                                    // block-wide sub-chunk sequence position
  // This block owns items [lo(x), lo(x + 1)) of kv head j, lo(x) = x n / gx:
  // runs of consecutive chunks of one query block, so the queries are staged
  // once per run and each warp carries its online-softmax state (m, l, o)
  // across the run's chunks.  One partial per run; the last run of a query
  // block (an atomic counter over its runs) combines them.
  const int gx = gridDim.x;
  auto lo_of = [&](int x) { return (int)((unsigned)x * (unsigned)n_items / (unsigned)gx); };  // n_items * gx < 2^32
  // (with at most one item per block, block x takes item x)
  const int it_lo = n_items <= gx ? (int)blockIdx.x : lo_of(blockIdx.x);
  const int it_hi = n_items <= gx ? min((int)blockIdx.x + 1, n_items) : lo_of(blockIdx.x + 1);
  typename WarpAttnOf<Dt, D, NQ, KW>::type ws;  // this warp's online-softmax state
  auto reset_state = [&]() { ws.reset(); };
  reset_state();
  __shared__ int s_run[2];  // this block's run index within the query block, number of runs

  // merge the warps' states of the run over query block b into its partial;
  // the last run of b combines
  auto flush = [&](int b, bool last) {
    const AttnQBlock qb = a.qblocks[b];
    const int nq = qb.nrows * G;
    ws.store(wp + (size_t)warp * NQ * WP, WP);
    if (tid == 0) {  // runs of b: blocks with a non-empty range meeting b's items [part_base, part_base + n_chunks)
      const int s0 = qb.part_base, s1 = qb.part_base + qb.n_chunks;
      if (n_items <= gx) {  // one item per block: the run index is the item's chunk
        s_run[0] = it_lo - s0;
        s_run[1] = s1 - s0;
      } else {  // every range is non-empty; the block holding item i is ceil((i + 1) gx / n) - 1
        auto owner = [&](int i) { return (int)(((unsigned)(i + 1) * (unsigned)gx + n_items - 1) / (unsigned)n_items) - 1; };
        const int x0 = owner(s0);
        s_run[0] = (int)blockIdx.x - x0;
        s_run[1] = owner(s1 - 1) - x0 + 1;
      }
    }
    csync();
    if (s_fail) return;
    const size_t part0 = ((size_t)(qb.part_base + s_run[0]) * a.KV + j) * a.nq_max;
    if (warp < nq) {
      const int i = warp;
      const float m = lane < AD_CWARPS ? wp[((size_t)lane * NQ + i) * WP + D] : -CUDART_INF_F;
      const float M = warp_max(m);
      const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
      const float L = warp_sum(lane < AD_CWARPS ? f * wp[((size_t)lane * NQ + i) * WP + D + 1] : 0.f);
      if (lane < AD_CWARPS) mrg[i * MP + lane] = f;
      if (lane == 0) {
        a.part_ml[(part0 + i) * 2] = M;
        a.part_ml[(part0 + i) * 2 + 1] = L;
      }
    }
    csync();
    for (int idx = tid; idx < nq * D; idx += AD_CTHREADS) {
      const int i = idx / D, d = idx % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < AD_CWARPS; ++w) v = fmaf(wp[((size_t)w * NQ + i) * WP + d], mrg[i * MP + w], v);
      a.part_o[(part0 + i) * D + d] = v;
    }
    __threadfence();
    csync();
    if (tid == 0) {
      const int prev = atomicAdd(a.counters + (size_t)b * a.KV + j, 1);
      s_flag = (prev == s_run[1] - 1);
    }
    csync();
    if (s_flag) {
      const int nc = s_run[1];
      // the ring is idle once this block's last run is flushed
      const bool os = last && (size_t)nc * nq * D <= LY::STAGES * LY::STAGE / 4;
      combine_parts<Dt, D, NQ>(a, qb, j, nc, nq, G, wp, mrg, os ? reinterpret_cast<float*>(ad_smem) : nullptr);
      if (tid == 0) a.counters[(size_t)b * a.KV + j] = 0;
    }
    csync();
  };

  int cur = -1;  // query block of the current run
  for (int it = it_lo; it < it_hi; ++it) {
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const ItemKeys ik = item_keys<Dt>(item, qb);
    const int nq = qb.nrows * G;  // <= NQ
    if (item.qb != cur) {
      if (cur >= 0) {
        flush(cur, false);
        if (s_fail) break;
        reset_state();
      }
      cur = item.qb;
      // queries: RMSNorm + RoPE of this block's q heads of kv group j (warp per query)
      if (warp < NQ) {
        const int i = warp;
        float x[DPL];
        if (i < nq) {
          const int row = qb.row0 + i / G, hh = j * G + i % G;
          const Dt* src = qkv + (size_t)row * qkv_ld + (size_t)hh * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) x[e] = to_f(src[e]);
          norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.q_gain), a.cos_t, a.sin_t, qb.pos0 + i / G, a.eps);
        } else {
#pragma unroll
          for (int e = 0; e < DPL; ++e) x[e] = 0.f;
        }
        store_lane_vec<DPL>(qs + i * D + lane * DPL, x);
      }
      csync();
      ws.load_q(qs, nq);
    }

    // ---- this warp's keys of the item, folded into its running state
    if (wsub < ik.nsub) {
      const int s = (g + wsub) % LY::STAGES;
      const int key0 = ik.key0 + wsub * CK;                     // sub-chunk's first key
      const int nk = min(KW, ik.key0 + ik.nkeys - key0 - wk0);  // this warp's keys (may be <= 0)
      const KVT<Dt, D, SWZ> Kt{tiles(s) + (size_t)wk0 * D * sizeof(Dt)};
      const KVT<Dt, D, SWZ> Vt{tiles(s) + LY::TILE + (size_t)wk0 * D * sizeof(Dt)};
      // A warp may reach a stage before the previous use of it has landed
      // (it skips the sub-chunks a shorter item does not have): wait until the
      // producer has issued this use, so that the parity wait below cannot
      // match the previous phase.
      int landed = 1;
      if (lane == 0) {
        const int use = (g + wsub) / LY::STAGES;
        const long long t0 = clock64();
        while (*(volatile int*)&s_issued[s] <= use) {
          if (clock64() - t0 > (1ll << 31)) {
            atomicExch(a.err, 2);
            landed = 0;
            break;
          }
        }
        if (landed) landed = mbar_wait(&full[s], (uint32_t)(use & 1), a.err, 2);
      }
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, landed, 0)) {
        s_fail = 1;
      } else if (nk > 0) {
        const int kb = key0 + wk0;  // absolute position of this warp's first key
        // keys appended by this call among this warp's keys
        const int n0 = max(kb, qb.seg_pos0), n1 = min(kb + nk, qb.seg_pos0 + qb.seg_n);
        for (int u = n0; u < n1; ++u) {
          const int row = qb.seg_row0 + (u - qb.seg_pos0);
          float x[DPL], v[DPL];
          const Dt* ksrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + j) * D + lane * DPL;
          const Dt* vsrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + a.KV + j) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) { x[e] = to_f(ksrc[e]); v[e] = to_f(vsrc[e]); }
          norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.k_gain), a.cos_t, a.sin_t, u, a.eps);
          const bool owner = row >= qb.row0 && row < qb.row0 + qb.nrows;
          const size_t goff = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + u) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            Kt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(x[e]);
            Vt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(v[e]);
            if (owner) {
              static_cast<Dt*>(a.kc)[goff + e] = from_f<Dt>(x[e]);
              static_cast<Dt*>(a.vc)[goff + e] = from_f<Dt>(v[e]);
            }
          }
        }
        __syncwarp();
        ws.attend(Kt, Vt, qs, ps, nk, nq, kb, qb.pos0, G, a.scale);
      }
      // this warp is done with its part of the stage (its smem writes ordered
      // before the producer's next copy into it)
      __syncwarp();
      fence_proxy_async();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    g += ik.nsub;
  }
  if (cur >= 0 && !s_fail) flush(cur, true);
}

// One item per block and step of the persistent loop (used when the grid has
// at least as many blocks as items, e.g. batch-1 decode): the queries are
// staged and the warp partials merged for every item.
template <typename Dt, int D, int NQ>
__global__ void __launch_bounds__(AD_THREADS, 1)
    attn_decode_item_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, AttnDecArgs a) {
  extern __shared__ __align__(128) uint8_t ad_smem_raw[];
  uint8_t* ad_smem = align1024(ad_smem_raw);  // the K/V tiles' swizzle is relative to 1024-byte blocks
  using LY = ADLayout<Dt, D, NQ>;
  constexpr int CK = LY::CK;
  constexpr int KW = LY::KW;
  constexpr bool SWZ = WarpAttnOf<Dt, D, NQ, KW>::type::kSwizzled;  // K / V tiles swizzled (tensor loads)            // keys per warp
  constexpr int DPL = D / 32;           // head elements per lane
  constexpr int WP = LY::WPITCH;
  constexpr int MP = LY::MPITCH;
  float* qs = reinterpret_cast<float*>(ad_smem + LY::OFF_QS);
  float* ps_all = reinterpret_cast<float*>(ad_smem + LY::OFF_PS);
  float* wp = reinterpret_cast<float*>(ad_smem + LY::OFF_WP);
  float* mrg = reinterpret_cast<float*>(ad_smem + LY::OFF_MRG);
  uint64_t* full = reinterpret_cast<uint64_t*>(ad_smem + LY::OFF_BAR);
  uint64_t* empty = full + LY::STAGES;
  __shared__ int s_flag, s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int qkv_ld = (a.H + 2 * a.KV) * D;
  const int n_items = *a.n_items;
  auto tiles = [&](int s) { return ad_smem + (size_t)s * LY::STAGE; };

  if (tid == 0) {
    for (int s = 0; s < LY::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], AD_WPS);
    }
    mbar_fence_init();
    s_fail = 0;
  }
  __syncthreads();

  if (warp == AD_CWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int g = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const AttnItem item = a.items[it];
        const AttnQBlock qb = a.qblocks[item.qb];
        const ItemKeys ik = item_keys<Dt>(item, qb);
        for (int sub = 0; sub < ik.nsub; ++sub, ++g) {
          const int s = g % LY::STAGES;
          if (g >= LY::STAGES && !mbar_wait(&empty[s], (uint32_t)((g / LY::STAGES - 1) & 1), a.err, 2)) {
            s_fail = 1;
            return;
          }
          const int k0 = ik.key0 + sub * CK;
          if constexpr (SWZ) {
            load_kv_tiles<Dt, D>(tiles(s), &map_k, &map_v, j * a.capacity + k0, qb.seq, &full[s]);
          } else {
            const int nk = min(CK, ik.key0 + ik.nkeys - k0);
            const size_t off = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + k0) * D;
            const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
            mbar_expect_tx(&full[s], 2 * bytes);
            tma_load_1d(tiles(s), static_cast<const Dt*>(a.kc) + off, bytes, &full[s]);
            tma_load_1d(tiles(s) + LY::TILE, static_cast<const Dt*>(a.vc) + off, bytes, &full[s]);
          }
        }
      }
      // L2 prefetch of this block's share of the next kernels' operands
      prefetch_grid_share(a.pf, a.pf_bytes);
      prefetch_grid_share(a.pf2, a.pf2_bytes);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch();
  const Dt* qkv = static_cast<const Dt*>(a.qkv);
  float* ps = ps_all + (size_t)warp * NQ * KW;  // this warp's scores / probabilities
  const int wsub = warp / AD_WPS;               // sub-chunk of this warp
  const int wk0 = (warp % AD_WPS) * KW;         // its first key inside the sub-chunk
  int g = 0;                                    // block-wide sub-chunk sequence position
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const AttnItem item = a.items[it];
    const AttnQBlock qb = a.qblocks[item.qb];
    const ItemKeys ik = item_keys<Dt>(item, qb);
    const int nq = qb.nrows * G;  // <= NQ

    // queries: RMSNorm + RoPE of this block's q heads of kv group j (warp per query)
    if (warp < NQ) {
      const int i = warp;
      float x[DPL];
      if (i < nq) {
        const int row = qb.row0 + i / G, hh = j * G + i % G;
        const Dt* src = qkv + (size_t)row * qkv_ld + (size_t)hh * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) x[e] = to_f(src[e]);
        norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.q_gain), a.cos_t, a.sin_t, qb.pos0 + i / G, a.eps);
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) x[e] = 0.f;
      }
      store_lane_vec<DPL>(qs + i * D + lane * DPL, x);
    }
    csync();

    // ---- this warp's keys, end to end
    typename WarpAttnOf<Dt, D, NQ, KW>::type ws;
    ws.reset();
    ws.load_q(qs, nq);
    if (wsub < ik.nsub) {
      const int s = (g + wsub) % LY::STAGES;
      const int key0 = ik.key0 + wsub * CK;                     // sub-chunk's first key
      const int nk = min(KW, ik.key0 + ik.nkeys - key0 - wk0);  // this warp's keys (may be <= 0)
      const KVT<Dt, D, SWZ> Kt{tiles(s) + (size_t)wk0 * D * sizeof(Dt)};
      const KVT<Dt, D, SWZ> Vt{tiles(s) + LY::TILE + (size_t)wk0 * D * sizeof(Dt)};
      int landed = 1;
      if (lane == 0) landed = mbar_wait(&full[s], (uint32_t)(((g + wsub) / LY::STAGES) & 1), a.err, 2);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, landed, 0)) {
        s_fail = 1;
      } else if (nk > 0) {
        const int kb = key0 + wk0;  // absolute position of this warp's first key
        // keys appended by this call among this warp's keys
        const int n0 = max(kb, qb.seg_pos0), n1 = min(kb + nk, qb.seg_pos0 + qb.seg_n);
        for (int u = n0; u < n1; ++u) {
          const int row = qb.seg_row0 + (u - qb.seg_pos0);
          float x[DPL], v[DPL];
          const Dt* ksrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + j) * D + lane * DPL;
          const Dt* vsrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + a.KV + j) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) { x[e] = to_f(ksrc[e]); v[e] = to_f(vsrc[e]); }
          norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.k_gain), a.cos_t, a.sin_t, u, a.eps);
          const bool owner = row >= qb.row0 && row < qb.row0 + qb.nrows;
          const size_t goff = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + u) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) {
            Kt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(x[e]);
            Vt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(v[e]);
            if (owner) {
              static_cast<Dt*>(a.kc)[goff + e] = from_f<Dt>(x[e]);
              static_cast<Dt*>(a.vc)[goff + e] = from_f<Dt>(v[e]);
            }
          }
        }
        __syncwarp();
        ws.attend(Kt, Vt, qs, ps, nk, nq, kb, qb.pos0, G, a.scale);
      }
      // this warp is done with its part of the stage (its smem writes ordered
      // before the producer's next copy into it)
      __syncwarp();
      fence_proxy_async();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // warp partial -> shared memory
    ws.store(wp + (size_t)warp * NQ * WP, WP);
    g += ik.nsub;
    csync();
    if (s_fail) break;

    // merge the 16 warp partials into this item's partial; warp i: lanes over
    // the warp partials of query i
    const size_t part0 = ((size_t)(qb.part_base + item.chunk) * a.KV + j) * a.nq_max;
    if (warp < nq) {
      const int i = warp;
      const float m = lane < AD_CWARPS ? wp[((size_t)lane * NQ + i) * WP + D] : -CUDART_INF_F;
      const float M = warp_max(m);
      const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
      const float L = warp_sum(lane < AD_CWARPS ? f * wp[((size_t)lane * NQ + i) * WP + D + 1] : 0.f);
      if (lane < AD_CWARPS) mrg[i * MP + lane] = f;
      if (lane == 0) {
        a.part_ml[(part0 + i) * 2] = M;
        a.part_ml[(part0 + i) * 2 + 1] = L;
      }
    }
    csync();
    for (int idx = tid; idx < nq * D; idx += AD_CTHREADS) {
      const int i = idx / D, d = idx % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < AD_CWARPS; ++w) v = fmaf(wp[((size_t)w * NQ + i) * WP + d], mrg[i * MP + w], v);
      a.part_o[(part0 + i) * D + d] = v;
    }
    __threadfence();
    csync();
    if (tid == 0) {
      const int prev = atomicAdd(a.counters + (size_t)item.qb * a.KV + j, 1);
      s_flag = (prev == qb.n_chunks - 1);
    }
    csync();
    if (s_flag) {
      const int nc = qb.n_chunks;
      // the ring is idle once this block's last item has been consumed
      const bool os = it + (int)gridDim.x >= n_items && (size_t)nc * nq * D <= LY::STAGES * LY::STAGE / 4;
      combine_parts<Dt, D, NQ>(a, qb, j, nc, nq, G, wp, mrg, os ? reinterpret_cast<float*>(ad_smem) : nullptr);
      if (tid == 0) a.counters[(size_t)item.qb * a.KV + j] = 0;
    }
    csync();
  }
}

// One (query block, kv head) per thread-block cluster (batch-1 and small
// batches): the cluster's CTAs split the block's keys 0..last into equal runs
// of whole sub-chunks, each CTA loads its whole run into its ring at launch
// (every stage used once, no refills), its warps compute as in the kernels
// above, the warp partials merge into the CTA's partial in shared memory, and
// after a cluster barrier each CTA combines one slice of the output elements
// from all the CTAs' partials through distributed shared memory:
// out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c, rounded once.  No
// partial goes through global memory and no CTA waits on another's atomic.
template <typename Dt, int D, int NQ>
__global__ void __launch_bounds__(AD_THREADS, 1)
    attn_decode_cluster_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, AttnDecArgs a) {
  extern __shared__ __align__(128) uint8_t ad_smem_raw[];
  uint8_t* ad_smem = align1024(ad_smem_raw);  // the K/V tiles' swizzle is relative to 1024-byte blocks
  using LY = ADLayout<Dt, D, NQ>;
  constexpr int CK = LY::CK;
  constexpr int KW = LY::KW;
  constexpr bool SWZ = WarpAttnOf<Dt, D, NQ, KW>::type::kSwizzled;  // K / V tiles swizzled (tensor loads)
  constexpr int DPL = D / 32;
  constexpr int WP = LY::WPITCH;
  constexpr int MP = LY::MPITCH;
  constexpr int CP = LY::CPITCH;
  float* qs = reinterpret_cast<float*>(ad_smem + LY::OFF_QS);
  float* ps_all = reinterpret_cast<float*>(ad_smem + LY::OFF_PS);
  float* wp = reinterpret_cast<float*>(ad_smem + LY::OFF_WP);
  float* mrg = reinterpret_cast<float*>(ad_smem + LY::OFF_MRG);
  float* cp = reinterpret_cast<float*>(ad_smem + LY::OFF_CP);
  uint64_t* full = reinterpret_cast<uint64_t*>(ad_smem + LY::OFF_BAR);
  __shared__ int s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = blockIdx.y;
  const int G = a.H / a.KV;
  const int qkv_ld = (a.H + 2 * a.KV) * D;
  const uint32_t rank = cluster_rank(), ncl = cluster_size();
  const AttnQBlock qb = a.qblocks[blockIdx.x / ncl];
  const int nq = qb.nrows * G;  // <= NQ
  // this CTA's keys: whole sub-chunks, [k_lo, k_hi) of 0 .. last position
  const int n_keys = qb.pos0 + qb.nrows;
  const int per = ((n_keys + (int)ncl - 1) / (int)ncl + CK - 1) / CK * CK;
  const int k_lo = min((int)rank * per, n_keys), k_hi = min(k_lo + per, n_keys);
  int nsub = (k_hi - k_lo + CK - 1) / CK;  // <= LY::STAGES (the host checks attn_decode_cluster_keys)
  auto tiles = [&](int s) { return ad_smem + (size_t)s * LY::STAGE; };

  if (tid == 0) {
    for (int s = 0; s < LY::STAGES; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    s_fail = 0;
    if (nsub > LY::STAGES) {  // a run longer than the ring: refuse rather than overrun it
      atomicExch(a.err, 14);
      s_fail = 1;
    }
  }
  if (nsub > LY::STAGES) nsub = 0;
  __syncthreads();

  if (warp == AD_CWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int sub = 0; sub < nsub && sub < LY::STAGES; ++sub) {
        const int k0 = k_lo + sub * CK;
        if constexpr (SWZ) {
          load_kv_tiles<Dt, D>(tiles(sub), &map_k, &map_v, j * a.capacity + k0, qb.seq, &full[sub]);
        } else {
          const int nk = min(CK, k_hi - k0);
          const size_t off = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + k0) * D;
          const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
          mbar_expect_tx(&full[sub], 2 * bytes);
          tma_load_1d(tiles(sub), static_cast<const Dt*>(a.kc) + off, bytes, &full[sub]);
          tma_load_1d(tiles(sub) + LY::TILE, static_cast<const Dt*>(a.vc) + off, bytes, &full[sub]);
        }
      }
      // L2 prefetch of this CTA's share of the next kernels' operands
      prefetch_grid_share(a.pf, a.pf_bytes);
      prefetch_grid_share(a.pf2, a.pf2_bytes);
    }
  } else {
    // ---------------------------------------------------------- consumers
    pdl_wait();
    pdl_launch();
    const Dt* qkv = static_cast<const Dt*>(a.qkv);
    float* ps = ps_all + (size_t)warp * NQ * KW;
    const int wsub = warp / AD_WPS;
    const int wk0 = (warp % AD_WPS) * KW;
    if (warp < NQ) {  // queries: RMSNorm + RoPE (warp per query)
      const int i = warp;
      float x[DPL];
      if (i < nq) {
        const int row = qb.row0 + i / G, hh = j * G + i % G;
        const Dt* src = qkv + (size_t)row * qkv_ld + (size_t)hh * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) x[e] = to_f(src[e]);
        norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.q_gain), a.cos_t, a.sin_t, qb.pos0 + i / G, a.eps);
      } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) x[e] = 0.f;
      }
      store_lane_vec<DPL>(qs + i * D + lane * DPL, x);
    }
    csync();
    typename WarpAttnOf<Dt, D, NQ, KW>::type ws;
    ws.reset();
    ws.load_q(qs, nq);
    for (int sub = wsub; sub < nsub; sub += AD_SUBS) {
      const int key0 = k_lo + sub * CK;
      const int nk = min(KW, k_hi - key0 - wk0);
      const KVT<Dt, D, SWZ> Kt{tiles(sub) + (size_t)wk0 * D * sizeof(Dt)};
      const KVT<Dt, D, SWZ> Vt{tiles(sub) + LY::TILE + (size_t)wk0 * D * sizeof(Dt)};
      int landed = 1;
      if (lane == 0) landed = mbar_wait(&full[sub], 0u, a.err, 2);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, landed, 0)) {
        s_fail = 1;
        break;
      }
      if (nk <= 0) continue;
      const int kb = key0 + wk0;
      const int n0 = max(kb, qb.seg_pos0), n1 = min(kb + nk, qb.seg_pos0 + qb.seg_n);
      for (int u = n0; u < n1; ++u) {  // keys appended by this call: from the qkv row
        const int row = qb.seg_row0 + (u - qb.seg_pos0);
        float x[DPL], v[DPL];
        const Dt* ksrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + j) * D + lane * DPL;
        const Dt* vsrc = qkv + (size_t)row * qkv_ld + (size_t)(a.H + a.KV + j) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) { x[e] = to_f(ksrc[e]); v[e] = to_f(vsrc[e]); }
        norm_rope_head<Dt, D>(x, static_cast<const Dt*>(a.k_gain), a.cos_t, a.sin_t, u, a.eps);
        const bool owner = row >= qb.row0 && row < qb.row0 + qb.nrows;
        const size_t goff = (size_t)qb.seq * a.seq_stride + ((size_t)j * a.capacity + u) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          Kt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(x[e]);
          Vt.elem(u - kb, lane * DPL)[e] = from_f<Dt>(v[e]);
          if (owner) {
            static_cast<Dt*>(a.kc)[goff + e] = from_f<Dt>(x[e]);
            static_cast<Dt*>(a.vc)[goff + e] = from_f<Dt>(v[e]);
          }
        }
      }
      __syncwarp();
      ws.attend(Kt, Vt, qs, ps, nk, nq, kb, qb.pos0, G, a.scale);
    }
    // warp partials -> the CTA's partial cp[i] = (sum_w f_w o_w, M, sum_w f_w l_w)
    ws.store(wp + (size_t)warp * NQ * WP, WP);
    csync();
    if (warp < NQ) {
      const int i = warp;
      const float m = lane < AD_CWARPS ? wp[((size_t)lane * NQ + i) * WP + D] : -CUDART_INF_F;
      const float M = warp_max(m);
      const float f = (m == -CUDART_INF_F) ? 0.f : expf(m - M);
      const float L = warp_sum(lane < AD_CWARPS ? f * wp[((size_t)lane * NQ + i) * WP + D + 1] : 0.f);
      if (lane < AD_CWARPS) mrg[i * MP + lane] = f;
      if (lane == 0) { cp[i * CP + D] = M; cp[i * CP + D + 1] = L; }
    }
    csync();
    for (int idx = tid; idx < NQ * D; idx += AD_CTHREADS) {
      const int i = idx / D, d = idx % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < AD_CWARPS; ++w) v = fmaf(wp[((size_t)w * NQ + i) * WP + d], mrg[i * MP + w], v);
      cp[i * CP + d] = v;
    }
    csync();
    // push: every CTA's m and l of each query, and to CTA d the values of d's
    // slice of the nq x D outputs, stored into d's receive area (remote
    // stores; the cluster barrier's release / acquire orders them before
    // d's reads, and nothing reads another CTA's memory after it)
    const int total = nq * D;
    const int share = (total + (int)ncl - 1) / (int)ncl;
    const uint32_t rx = smem_u32(ad_smem + LY::OFF_RX);
    constexpr int RS = LY::RX_SHARE;
    const int nml = (int)ncl * 2 * nq;
    for (int t = tid; t < nml + total; t += AD_CTHREADS) {
      if (t < nml) {
        const int d = t / (2 * nq), r = t % (2 * nq), i = r >> 1, which = r & 1;
        const uint32_t off = (uint32_t)((which * 16 + (int)rank) * NQ + i) * 4u;  // m [16][NQ], then l [16][NQ]
        st_cluster(cluster_map(rx + off, (uint32_t)d), cp[i * CP + D + which]);
      } else {
        const int idx = t - nml, d = idx / share, k = idx - d * share;
        const uint32_t off = (uint32_t)(32 * NQ + (int)rank * RS + k) * 4u;
        st_cluster(cluster_map(rx + off, (uint32_t)d), cp[(idx / D) * CP + idx % D]);
      }
    }
  }
  // every CTA's pushes are in the receivers' shared memory after this
  __syncwarp();
  cluster_sync_all();
  {
    // This CTA's slice of the nq x D outputs from what the cluster pushed
    // here: the maxima and sums over the CTAs, then the weighted sums in CTA
    // order.
    const float* rx = reinterpret_cast<const float*>(ad_smem + LY::OFF_RX);
    const float* cm = rx;               // [16][NQ] m of CTA c
    const float* cl = rx + 16 * NQ;     // [16][NQ] l of CTA c
    const float* rv = rx + 32 * NQ;     // [16][RX_SHARE] values of CTA c
    constexpr int RS = LY::RX_SHARE;
    float* sM = wp;                     // [NQ] max over CTAs, then [NQ] the sum (scratch: warp partials)
    const int total = nq * D;
    const int share = (total + (int)ncl - 1) / (int)ncl;
    const int o0 = min(total, (int)rank * share), n_out = min(total, o0 + share) - o0;
    if (tid < nq) {
      float M = -CUDART_INF_F;
      for (uint32_t c = 0; c < ncl; ++c) M = fmaxf(M, cm[c * NQ + tid]);
      float L = 0.f;
      for (uint32_t c = 0; c < ncl; ++c) {
        const float m = cm[c * NQ + tid];
        L = fmaf(cl[c * NQ + tid], (m == -CUDART_INF_F) ? 0.f : expf(m - M), L);
      }
      sM[tid] = M;
      sM[NQ + tid] = L;
    }
    __syncthreads();
    if (!s_fail) {
      for (int t = tid; t < n_out; t += AD_THREADS) {
        const int idx = o0 + t, i = idx / D, d = idx % D;
        float v = 0.f;
        for (uint32_t c = 0; c < ncl; ++c) {
          const float m = cm[c * NQ + i];
          v = fmaf(rv[c * RS + t], (m == -CUDART_INF_F) ? 0.f : expf(m - sM[i]), v);
        }
        const int row = qb.row0 + i / G, head = j * G + i % G;
        static_cast<Dt*>(a.out)[((size_t)row * a.H + head) * D + d] = from_f<Dt>(v / sM[NQ + i]);
      }
    }
  }
}

// 3-D map over one layer's K or V cache [sequence][kv head x capacity][D],
// each position's row seen as D * sizeof(Dt) / 128 lines of 128 bytes: boxes
// of CK positions' lines (one contiguous piece of the cache), 128-byte
// swizzle, zeros out of bounds.
template <typename Dt>
bool make_kv_map(CUtensorMap* m, const void* base, int D, const AttnDecArgs& a) {
  tc::EncodeTiledFn fn = tc::encode_fn();
  const int R = D * (int)sizeof(Dt) / 128;
  if (!fn || a.n_seqs < 1 || R < 1) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(128 / sizeof(Dt)), (cuuint64_t)R * a.KV * a.capacity, (cuuint64_t)a.n_seqs};
  const cuuint64_t strides[2] = {128, (cuuint64_t)a.seq_stride * sizeof(Dt)};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / sizeof(Dt)), (cuuint32_t)(R * ADT<Dt>::CK), 1}, estr[3] = {1, 1, 1};
  return fn(m, sizeof(Dt) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Dt, int D, int NQ>
cudaError_t ad_launch(const LaunchCtx& c, const AttnDecArgs& a) {
  using LY = ADLayout<Dt, D, NQ>;
  CUtensorMap mk, mv;
  if ((reinterpret_cast<uintptr_t>(a.kc) & 15) || (reinterpret_cast<uintptr_t>(a.vc) & 15) ||
      !make_kv_map<Dt>(&mk, a.kc, D, a) || !make_kv_map<Dt>(&mv, a.vc, D, a))
    return cudaErrorInvalidValue;
  if (a.cluster > 1) {
    // 8..16 CTAs: each receive area holds the slices of at least 8 CTAs' shares
    if (a.cluster < 8 || a.cluster > 16) return cudaErrorInvalidValue;
    auto ck = attn_decode_cluster_kernel<Dt, D, NQ>;
    cudaError_t e = set_max_smem((const void*)ck, (int)LY::TOTAL_CL);
    if (e != cudaSuccess) return e;
    if (a.cluster > 8) {
      e = cudaFuncSetAttribute(ck, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid_x, a.KV);
    cfg.blockDim = dim3(AD_THREADS);
    cfg.dynamicSmemBytes = LY::TOTAL_CL;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, ck, mk, mv, a);
  }
  auto kern = a.runs ? attn_decode_kernel<Dt, D, NQ> : attn_decode_item_kernel<Dt, D, NQ>;
  cudaError_t e = set_max_smem((const void*)kern, (int)LY::TOTAL);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(a.grid_x, a.KV), dim3(AD_THREADS), LY::TOTAL, c, mk, mv, a);
}

template <typename Dt, int D>
cudaError_t ad_nq(const LaunchCtx& c, const AttnDecArgs& a) {
  if (a.nq <= 1) return ad_launch<Dt, D, 1>(c, a);
  if (a.nq <= 2) return ad_launch<Dt, D, 2>(c, a);
  if (a.nq <= 4) return ad_launch<Dt, D, 4>(c, a);
  return ad_launch<Dt, D, 8>(c, a);
}

}  // namespace

// Keys one cluster of `cl` CTAs can take for a query block of nq query
// vectors (every CTA holds its whole run in its ring).
int attn_decode_cluster_keys(int dt, int nq, int cl) {
  const int ck = dt == DT_BF16 ? ADT<bf16>::CK : ADT<float>::CK;
  const int stages = nq <= 2 ? AD_STAGES_MAX : AD_SUBS;
  return cl * stages * ck;
}

namespace {
template <typename Dt, int D, int NQ>
int ad_cluster_fit(int cl, int kv, int clusters_x) {
  using LY = ADLayout<Dt, D, NQ>;
  auto ck = attn_decode_cluster_kernel<Dt, D, NQ>;
  if (set_max_smem((const void*)ck, (int)LY::TOTAL_CL) != cudaSuccess) return 0;
  if (cl > 8 && cudaFuncSetAttribute(ck, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl * clusters_x, kv);
  cfg.blockDim = dim3(AD_THREADS);
  cfg.dynamicSmemBytes = LY::TOTAL_CL;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ck, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}
template <typename Dt, int D>
int ad_cluster_fit_nq(int nq, int cl, int kv, int clusters_x) {
  if (nq <= 1) return ad_cluster_fit<Dt, D, 1>(cl, kv, clusters_x);
  if (nq <= 2) return ad_cluster_fit<Dt, D, 2>(cl, kv, clusters_x);
  if (nq <= 4) return ad_cluster_fit<Dt, D, 4>(cl, kv, clusters_x);
  return ad_cluster_fit<Dt, D, 8>(cl, kv, clusters_x);
}
}  // namespace

// How many clusters of `cl` CTAs of the cluster kernel can be resident at
// once on the current device (0 if the launch shape is not possible).
int attn_decode_cluster_capacity(int dt, int D, int nq, int cl, int kv, int clusters_x) {
  if (D == 128) return dt == DT_BF16 ? ad_cluster_fit_nq<bf16, 128>(nq, cl, kv, clusters_x)
                                     : ad_cluster_fit_nq<float, 128>(nq, cl, kv, clusters_x);
  if (D == 64) return dt == DT_BF16 ? ad_cluster_fit_nq<bf16, 64>(nq, cl, kv, clusters_x)
                                    : ad_cluster_fit_nq<float, 64>(nq, cl, kv, clusters_x);
  return 0;
}

int attn_decode2_chunk(int dt) { return (dt == DT_BF16 ? ADT<bf16>::CK : ADT<float>::CK) * AD_SUBS; }
int attn_decode2_nq_max() { return AD_NQ_MAX; }

cudaError_t launch_attn_decode2(const LaunchCtx& c, int dt, const AttnDecArgs& a) {
  if (a.nq < 1 || a.nq > AD_NQ_MAX) return cudaErrorInvalidValue;
  if (a.D == 128) return dt == DT_BF16 ? ad_nq<bf16, 128>(c, a) : ad_nq<float, 128>(c, a);
  if (a.D == 64) return dt == DT_BF16 ? ad_nq<bf16, 64>(c, a) : ad_nq<float, 64>(c, a);
  return cudaErrorInvalidValue;
}

}  // namespace q3
