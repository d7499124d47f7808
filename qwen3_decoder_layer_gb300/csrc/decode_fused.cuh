// A whole decode step (T <= 4 rows, dense layers) of the Qwen3 stack forward
// (maya2_mlx/backbone.py, Backbone.forward: per layer h = R(h + pend), y =
// RMSNorm(h), qkv = y Wqkv^T, per-head q/k RMSNorm + RoPE, cache append,
// attention over keys 0..pos, h = R(h + R(attn Wo^T)), y2 = RMSNorm(h),
// pend = R(R(R(silu(g)) * u) Wd^T); final RMSNorm) in ONE persistent kernel.
//
// Why: at batch 1 every linear and the attention are a few microseconds of
// HBM streaming each, and the boundary between two kernels (drain, launch,
// prologue) costs about as much again.  Here one CTA per SM stays resident
// for the whole step:
//
//  * A producer warp streams, in a fixed order, every byte this CTA will
//    read from HBM in the step -- its share of the weight rows of each linear
//    of each layer and its share of the KV cache -- through a ring of
//    shared-memory slots with TMA bulk copies (full / empty mbarriers).  None
//    of it depends on the step's activations, so the producer never waits
//    for a phase to finish: while the consumers sit at a grid barrier, the
//    ring fills with the next phase's weights and HBM keeps streaming.
//  * Sixteen consumer warps run the phases of each layer --
//      QKV  (RMSNorm prologue, rows of the fused q|k|v weight),
//      ATTN (q/k RMSNorm + RoPE, cache append, split-K attention over 256-key
//            items: each warp runs 16 keys end to end -- scores, a warp-local
//            softmax, P.V -- then one merge per item; the last item of a
//            (query block, kv head) combines the chunks),
//      O    (rows of Wo with the residual add and the row sums of squares),
//      GU   (RMSNorm prologue from those sums, gate|up row pairs, SiLU * up),
//      DOWN (rows of Wd with the residual add and sums of squares)
//    -- separated by grid barriers (an atomic counter; the launch is
//    cooperative, so all CTAs are resident).  Every phase's input (a few KB
//    per row) is staged in shared memory in the model dtype.
//  * After the last layer the final RMSNorm is spread over all CTAs.
//
// Every wait is bounded; a wait that gives up records an error code and
// raises an abort flag that makes every other wait return at once, so the
// kernel always terminates.
#pragma once
#include <math_constants.h>

#include <algorithm>

#include "common.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace q3 {

namespace fused {

using namespace dec;

constexpr int FD_CW = 15;               // consumer warps (16 warps in all: 4 per scheduler, 128 registers each)
constexpr int FD_CT = FD_CW * 32;       // 512 consumer threads
constexpr int FD_THREADS = FD_CT + 32;  // + producer warp
constexpr int FD_KW = 16;               // keys per attention unit (one warp)
constexpr int FD_ITEM = FD_KW * FD_CW;  // 240 keys per attention item
constexpr int FD_NQ = 8;                // query vectors (rows x G) per query block
constexpr int FD_RM = 4;                // weight rows per GEMV unit (at most)
constexpr int FD_MAXQB = 4;

// ---------------------------------------------------------------- schedule
struct QBlk {
  int seq, row0, nrows, pos0, seg_row0, seg_pos0, seg_n, n_chunks, part_base;
};
struct Sched {
  int nqb, n_items;
  QBlk qb[FD_MAXQB];
};

// Query blocks of the step's rows (rows of one sequence are consecutive):
// blocks of at most FD_NQ / G rows of one sequence.
__device__ inline void make_sched(const FusedArgs& a, Sched& S) {
  const int G = a.H / a.KV, rpb = FD_NQ / G;
  S.nqb = 0;
  int parts = 0, items = 0;
  for (int t = 0; t < a.T;) {
    int n = 1;
    while (t + n < a.T && a.row_seq[t + n] == a.row_seq[t]) ++n;
    for (int r = 0; r < n; r += rpb) {
      QBlk& q = S.qb[S.nqb++];
      q.seq = a.row_seq[t];
      q.row0 = t + r;
      q.nrows = min(rpb, n - r);
      q.pos0 = a.row_pos[t + r];
      q.seg_row0 = t;
      q.seg_pos0 = a.row_pos[t];
      q.seg_n = n;
      q.n_chunks = (q.pos0 + q.nrows + FD_ITEM - 1) / FD_ITEM;
      q.part_base = parts;
      parts += q.n_chunks;
      items += q.n_chunks * a.KV;
    }
    t += n;
  }
  S.n_items = items;
}
// Item i -> (query block, chunk, kv head).
__device__ __forceinline__ void item_of(const Sched& S, int KV, int i, int& b, int& ch, int& j) {
  b = 0;
  while (i >= S.qb[b].n_chunks * KV) {
    i -= S.qb[b].n_chunks * KV;
    ++b;
  }
  ch = i / KV;
  j = i % KV;
}
__device__ __forceinline__ int item_keys(const QBlk& q, int ch) { return min(FD_ITEM, q.pos0 + q.nrows - ch * FD_ITEM); }

// A CTA's share of the N rows of a linear: rows [r0, r1), in units of rpu rows.
struct Span {
  int r0, r1, rpu, nu;
};
__device__ __forceinline__ Span span_of(int N, int rpu, int c, int nc) {
  Span s;
  s.r0 = (int)((long long)N * c / nc);
  s.r1 = (int)((long long)N * (c + 1) / nc);
  s.rpu = rpu;
  s.nu = (s.r1 - s.r0 + rpu - 1) / rpu;
  return s;
}
// Rows per unit: as many as fit a slot, at most FD_RM (pairs: FD_RM / 2).
__host__ __device__ __forceinline__ int rows_per_unit(int slot_bytes, int row_bytes, bool pair) {
  int r = slot_bytes / (row_bytes * (pair ? 2 : 1));
  const int m = pair ? FD_RM / 2 : FD_RM;
  return r < 1 ? 0 : (r > m ? m : r);
}

// ---------------------------------------------------------------- shared memory layout
template <int D> struct FDL {
  // union area (phase input rows, or attention scratch) is placed after the ring
  static constexpr int WPITCH = D + 4;  // warp partial: o[D], m, l, pad
  static constexpr size_t ATT_QS = 0;                                             // [NQ][D]
  static constexpr size_t ATT_PS = ATT_QS + (size_t)FD_NQ * D * 4;                // [warp][NQ][KW]
  static constexpr size_t ATT_WP = ATT_PS + (size_t)FD_CW * FD_NQ * FD_KW * 4;    // [warp][NQ][WPITCH]
  static constexpr size_t ATT_MRG = ATT_WP + (size_t)FD_CW * FD_NQ * WPITCH * 4;  // [NQ][CW + 2]
  static constexpr size_t ATT_BYTES = ATT_MRG + (size_t)FD_NQ * (FD_CW + 2) * 4;
  static constexpr size_t WP_FLOATS = (size_t)FD_CW * FD_NQ * WPITCH;
};

__host__ __device__ __forceinline__ size_t fd_align(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct FDGeom {
  size_t ring, uni, misc, total;
};
__host__ __device__ inline FDGeom fd_geom(const FusedArgs& a, size_t att_bytes) {
  FDGeom g;
  g.ring = (size_t)a.n_slots * a.slot_bytes;
  g.uni = fd_align((size_t)a.u_bytes > att_bytes ? (size_t)a.u_bytes : att_bytes, 128);
  g.misc = (size_t)a.n_slots * 16 + 1024;  // full/empty barriers, reductions, flags
  g.total = g.ring + g.uni + g.misc;
  return g;
}

// ---------------------------------------------------------------- sync helpers
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(FD_CT) : "memory"); }
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool aborted(const FusedArgs& a) { return *(volatile unsigned*)(a.sync + 1) != 0; }
__device__ __forceinline__ void raise_abort(const FusedArgs& a, int code) {
  atomicExch(a.err, code);
  atomicExch(a.sync + 1, 1u);
}
// Bounded, abort-aware wait for phase `parity` of an mbarrier.
__device__ inline bool fwait(uint64_t* bar, uint32_t parity, const FusedArgs& a, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (int it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (aborted(a)) return false;
      if (clock64() - t0 > (1ll << 31)) {
        raise_abort(a, code);
        return false;
      }
    }
  }
}
// Warp-wide wait for ring unit gg (slot gg % ns, use gg / ns): lane 0 first
// waits until the producer has issued that use of the slot (issued[slot] >
// use), then for the slot's full barrier.  The first step matters: a warp
// may reach a unit more than one slot-use ahead of the oldest unit not yet
// consumed (warps take units 15 apart, the ring may hold fewer), and a
// parity wait on a barrier two phases behind would pass at once.
__device__ __forceinline__ bool unit_wait(uint64_t* full, const int* issued, int ns, int gg, const FusedArgs& a,
                                          int code, bool live) {
  int ok = live;
  if ((threadIdx.x & 31) == 0 && live) {
    const int slot = gg % ns, use = gg / ns;
    const long long t0 = clock64();
    for (int it = 1; *(volatile const int*)&issued[slot] <= use; ++it) {
      if ((it & 255) == 0) {
        if (aborted(a)) { ok = 0; break; }
        if (clock64() - t0 > (1ll << 31)) {
          raise_abort(a, code);
          ok = 0;
          break;
        }
      }
    }
    if (ok) ok = fwait(&full[slot], (uint32_t)(use & 1), a, code);
  }
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Grid barrier among the consumer warps of all CTAs: the k-th barrier of the
// step waits for the counter to reach k * gridDim.x.
__device__ inline void grid_barrier(const FusedArgs& a, unsigned k) {
  csync();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.sync, 1u);
    const unsigned target = k * gridDim.x;
    const long long t0 = clock64();
    for (int it = 1;; ++it) {
      if (ld_acquire(a.sync) >= target) break;
      if ((it & 63) == 0) {
        if (aborted(a)) break;
        if (clock64() - t0 > (1ll << 31)) {
          raise_abort(a, 20);
          break;
        }
      }
    }
    __threadfence();
  }
  csync();
}
// Sum of an F2 over the consumer threads (red: 2 * FD_CW floats); all get it.
__device__ __forceinline__ F2 f2_csum(F2 v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = f2_warp_sum(v);
  csync();
  if (lane == 0) { red[2 * warp] = v.hi; red[2 * warp + 1] = v.lo; }
  csync();
  F2 t;
  t.hi = lane < FD_CW ? red[2 * lane] : 0.f;
  t.lo = lane < FD_CW ? red[2 * lane + 1] : 0.f;
  return f2_warp_sum(t);
}

// Loads of data other CTAs wrote during this launch: through L2 only.
template <typename Dt> __device__ __forceinline__ uint4 ldcg16(const Dt* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }
template <typename Dt> __device__ __forceinline__ float ldcg_e(const Dt* p);
template <> __device__ __forceinline__ float ldcg_e<float>(const float* p) { return __ldcg(p); }
template <> __device__ __forceinline__ float ldcg_e<bf16>(const bf16* p) {
  const unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(p));
  return __uint_as_float((uint32_t)u << 16);
}
template <typename Dt> __device__ __forceinline__ void stcg_e(Dt* p, float v);
template <> __device__ __forceinline__ void stcg_e<float>(float* p, float v) { __stcg(p, v); }
template <> __device__ __forceinline__ void stcg_e<bf16>(bf16* p, float v) {
  __stcg(reinterpret_cast<unsigned short*>(p), (unsigned short)(__float_as_uint(rd<bf16>(v)) >> 16));
}

// ---------------------------------------------------------------- staging
// xs[t][k] = RMSNorm(src[t]) * gain (the two roundings), with each row's
// scale from `sumsq` (double, precomputed) or, if sumsq is null, computed
// here over the row.  src_plain: src is this launch's input (not written by
// other CTAs).
template <typename Dt>
__device__ void stage_norm(Dt* xs, const Dt* src, const Dt* gain, const double* sumsq, int T, int K, float eps,
                           float* red, F2* s_rs) {
  constexpr int V = Vec16<Dt>::N;
  const int tid = threadIdx.x;
  if (sumsq) {
    if (tid < T) s_rs[tid] = rms_scale2(f2_from_double(__ldcg(sumsq + tid)), K, eps);
  } else {
    for (int t = 0; t < T; ++t) {
      F2 ss = {0.f, 0.f};
      for (int k = tid * V; k < K; k += FD_CT * V) {
        float v[V];
        Vec16<Dt>::unpack(ldcg16(src + (size_t)t * K + k), v);
#pragma unroll
        for (int e = 0; e < V; ++e) f2_add_sq(ss, v[e]);
      }
      ss = f2_csum(ss, red);
      if (tid == 0) s_rs[t] = rms_scale2(ss, K, eps);
    }
  }
  csync();
  const int nch = T * K / V;
  for (int c = tid; c < nch; c += FD_CT) {
    const int t = c * V / K, k = c * V - t * K;
    float hv[V], gv[V], o[V];
    Vec16<Dt>::unpack(ldcg16(src + (size_t)c * V), hv);
    Vec16<Dt>::unpack(ld16(gain + k), gv);
    const F2 rs = s_rs[t];
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] = rms_apply2<Dt>(hv[e], rs, gv[e]);
    *reinterpret_cast<uint4*>(xs + (size_t)c * V) = Vec16<Dt>::pack(o);
  }
  csync();
}
template <typename Dt>
__device__ void stage_copy(Dt* xs, const Dt* src, int T, int K) {
  constexpr int V = Vec16<Dt>::N;
  for (int c = threadIdx.x; c < T * K / V; c += FD_CT)
    *reinterpret_cast<uint4*>(xs + (size_t)c * V) = ldcg16(src + (size_t)c * V);
  csync();
}

// ---------------------------------------------------------------- GEMV unit
// Dot products of up to FD_RM weight rows (in a slot) with the NT staged
// input rows; row r lives at slot + (r < nr ? r : up_off + (r - nr)) * rb
// (pair units: nr gate rows, then nr up rows).  res[r][t] in every lane.
template <typename Dt, int WF, int NT>
__device__ __forceinline__ void unit_dot(const uint8_t* slot, int nrows, int nr, size_t up_bytes, int rb,
                                         const Dt* xs, int K, const void* sc, const void* bi, int group,
                                         int grow0, int grow_up0, float (&res)[FD_RM][NT]) {
  using W = WRow<Dt, WF>;
  constexpr int XV = Vec16<Dt>::N;
  const int lane = threadIdx.x & 31;
  float acc[FD_RM][NT];
#pragma unroll
  for (int r = 0; r < FD_RM; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  const int nvec = K / W::EPV;
  for (int v = lane; v < nvec; v += 32) {
    const int k0 = v * W::EPV;
    float xv[NT][W::EPV];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < W::EPV / XV; ++q)
        Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(xs + (size_t)t * K + k0 + q * XV), xv[t] + q * XV);
#pragma unroll
    for (int r = 0; r < FD_RM; ++r) {
      if (r < nrows) {
        const size_t off = r < nr ? (size_t)r * rb : up_bytes + (size_t)(r - nr) * rb;
        const uint4 q = *reinterpret_cast<const uint4*>(slot + off + (size_t)v * 16);
        float w[W::EPV];
        W::get(q, w, sc, bi, K, group, (size_t)(r < nr ? grow0 + r : grow_up0 + (r - nr)), k0);
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int e = 0; e < W::EPV; ++e) acc[r][t] = fmaf(w[e], xv[t][e], acc[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < FD_RM; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) res[r][t] = warp_sum(acc[r][t]);
}

// ---------------------------------------------------------------- the kernel
struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int ns, sb;
};

template <typename Dt, int WF, int NT, int D, int NQ>
__global__ void __launch_bounds__(FD_THREADS, 1) decode_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(128) uint8_t fd_smem[];
  using LY = FDL<D>;
  constexpr int DPL = D / 32;
  constexpr int EPV = 16 / sizeof(Dt);
  constexpr int LPK = D / EPV;
  constexpr int KPS = 32 / LPK;
  constexpr int WPc = LY::WPITCH;
  constexpr int MP = FD_CW + 2;
  const FDGeom geo = fd_geom(a, LY::ATT_BYTES);
  Ring ring;
  ring.base = fd_smem;
  ring.ns = a.n_slots;
  ring.sb = a.slot_bytes;
  uint8_t* uni = fd_smem + geo.ring;
  ring.full = reinterpret_cast<uint64_t*>(uni + geo.uni);
  ring.empty = ring.full + a.n_slots;
  float* red = reinterpret_cast<float*>(ring.empty + a.n_slots);  // 64 floats
  F2* s_rs = reinterpret_cast<F2*>(red + 64);                      // [4]
  float* ssq_red = red + 72;                                       // [FD_CW][4][2]
  __shared__ Sched S;
  __shared__ int s_flag;
  __shared__ int s_issued[64];  // uses of each ring slot issued so far

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, nc = gridDim.x;
  const int H = a.H, KV = a.KV, G = H / KV, hid = a.hidden, I = a.I;
  const int qkv_n = (H + 2 * KV) * D;
  const int wbytes = WF == W_U8 ? 1 : (int)sizeof(Dt);
  const int rb_hid = hid * wbytes, rb_o = H * D * wbytes, rb_i = I * wbytes;
  const int rpu_qkv = rows_per_unit(a.slot_bytes, rb_hid, false);
  const int rpu_o = rows_per_unit(a.slot_bytes, rb_o, false);
  const int rpu_gu = rows_per_unit(a.slot_bytes, rb_hid, true);
  const int rpu_dn = rows_per_unit(a.slot_bytes, rb_i, false);
  const Span sp_qkv = span_of(qkv_n, rpu_qkv, c, nc);
  const Span sp_o = span_of(hid, rpu_o, c, nc);
  const Span sp_gu = span_of(I, rpu_gu, c, nc);
  const Span sp_dn = span_of(hid, rpu_dn, c, nc);
  const size_t kv_unit = (size_t)FD_KW * D * sizeof(Dt);  // K (then V) bytes of one attention unit

  if (tid < 64) s_issued[tid] = 0;
  if (tid == 0) {
    make_sched(a, S);
    for (int s = 0; s < a.n_slots; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // ================================================================ producer
  if (warp == FD_CW) {
    if (lane != 0) return;
    int g = 0;
    bool ok = true;
    auto slot_for = [&](int gg) -> uint8_t* { return ring.base + (size_t)(gg % ring.ns) * ring.sb; };
    auto acquire = [&](int gg) -> bool {
      if (gg < ring.ns) return true;
      return fwait(&ring.empty[gg % ring.ns], (uint32_t)((gg / ring.ns - 1) & 1), a, 21);
    };
    auto rows_units = [&](const Span& sp, const void* w, int rb, bool pair, int n_up) {
      for (int u = 0; u < sp.nu && ok; ++u, ++g) {
        if (!(ok = acquire(g))) break;
        const int r = sp.r0 + u * sp.rpu, n = min(sp.rpu, sp.r1 - r);
        uint8_t* dst = slot_for(g);
        uint64_t* bar = &ring.full[g % ring.ns];
        const uint32_t bytes = (uint32_t)(n * rb);
        mbar_expect_tx(bar, pair ? 2 * bytes : bytes);
        tma_load_1d(dst, static_cast<const char*>(w) + (size_t)r * rb, bytes, bar);
        if (pair) tma_load_1d(dst + (size_t)sp.rpu * rb, static_cast<const char*>(w) + (size_t)(n_up + r) * rb, bytes, bar);
        *(volatile int*)&s_issued[g % ring.ns] = g / ring.ns + 1;
      }
    };
    for (int l = 0; l < a.L && ok; ++l) {
      const FusedLayer& Lw = a.layers[l];
      rows_units(sp_qkv, Lw.qkv, rb_hid, false, 0);
      const Dt* kc = static_cast<const Dt*>(a.kc) + (size_t)l * a.layer_stride;
      const Dt* vc = static_cast<const Dt*>(a.vc) + (size_t)l * a.layer_stride;
      for (int it = c; it < S.n_items && ok; it += nc) {
        int b, ch, j;
        item_of(S, KV, it, b, ch, j);
        const QBlk& q = S.qb[b];
        const int nkeys = item_keys(q, ch);
        for (int u = 0; u * FD_KW < nkeys && ok; ++u, ++g) {
          if (!(ok = acquire(g))) break;
          const int k0 = ch * FD_ITEM + u * FD_KW, nk = min(FD_KW, ch * FD_ITEM + nkeys - k0);
          const size_t off = (size_t)q.seq * a.seq_stride + ((size_t)j * a.capacity + k0) * D;
          uint8_t* dst = slot_for(g);
          uint64_t* bar = &ring.full[g % ring.ns];
          const uint32_t bytes = (uint32_t)(nk * D * sizeof(Dt));
          mbar_expect_tx(bar, 2 * bytes);
          tma_load_1d(dst, kc + off, bytes, bar);
          tma_load_1d(dst + kv_unit, vc + off, bytes, bar);
          *(volatile int*)&s_issued[g % ring.ns] = g / ring.ns + 1;
        }
      }
      rows_units(sp_o, Lw.o, rb_o, false, 0);
      rows_units(sp_gu, Lw.gu, rb_hid, true, I);
      rows_units(sp_dn, Lw.down, rb_i, false, 0);
    }
    // leave no copy in flight: the last issued unit of each slot has landed
    for (int gg = max(0, g - ring.ns); gg < g; ++gg)
      fwait(&ring.full[gg % ring.ns], (uint32_t)((gg / ring.ns) & 1), a, 22);
    return;
  }

  // ================================================================ consumers
  Dt* xs = reinterpret_cast<Dt*>(uni);
  float* qs = reinterpret_cast<float*>(uni + LY::ATT_QS);
  float* ps = reinterpret_cast<float*>(uni + LY::ATT_PS) + (size_t)warp * FD_NQ * FD_KW;
  float* wp = reinterpret_cast<float*>(uni + LY::ATT_WP);
  float* mrg = reinterpret_cast<float*>(uni + LY::ATT_MRG);
  Dt* hbuf = static_cast<Dt*>(a.h);
  Dt* qkvb = static_cast<Dt*>(a.qkv);
  Dt* attnb = static_cast<Dt*>(a.attn);
  Dt* mb = static_cast<Dt*>(a.mbuf);
  const int T = a.T;
  int g = 0;
  unsigned nbar = 0;
  bool live = true;

  // Weight-row phase: units k = warp, warp + 16, ... of the span; `epi`
  // consumes res[r][t] for row r of the unit (global row gr).
  auto gemv_phase = [&](const Span& sp, int rb, bool pair, int K, const void* sc, const void* bi, int n_up,
                        auto&& epi) {
    for (int u = warp; u < sp.nu; u += FD_CW) {
      const int gg = g + u;
      live = unit_wait(ring.full, s_issued, ring.ns, gg, a, 23, live);
      const int r0 = sp.r0 + u * sp.rpu, n = min(sp.rpu, sp.r1 - r0);
      float res[FD_RM][NT];
      if (live) {
        const uint8_t* slot = ring.base + (size_t)(gg % ring.ns) * ring.sb;
        unit_dot<Dt, WF, NT>(slot, pair ? 2 * n : n, n, (size_t)sp.rpu * rb, rb, xs, K, sc, bi, a.group, r0,
                             n_up + r0, res);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&ring.empty[gg % ring.ns]);
      if (live) epi(r0, n, res);
    }
    g += sp.nu;
  };

  // Residual epilogue: h[t][row] = R(h + R(v)); squares of the new values.
  F2 ssq[NT];
  auto residual_epi = [&](int r0, int n, float (&res)[FD_RM][NT]) {
#pragma unroll
    for (int r = 0; r < FD_RM; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (r < n && lane == r * NT + t) {
          Dt* p = hbuf + (size_t)t * hid + r0 + r;
          const float hn = rd<Dt>(ldcg_e<Dt>(p) + rd<Dt>(res[r][t]));
          stcg_e<Dt>(p, hn);
          f2_add_sq(ssq[t], hn);
        }
  };
  // Per-CTA sum of the squares -> sumsq[slot][t].
  auto flush_ssq = [&](double* dst) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const F2 v = f2_warp_sum(ssq[t]);
      if (lane == 0) { ssq_red[(warp * 4 + t) * 2] = v.hi; ssq_red[(warp * 4 + t) * 2 + 1] = v.lo; }
      ssq[t] = F2{0.f, 0.f};
    }
    csync();
    if (tid < NT) {
      F2 s = {0.f, 0.f};
      for (int w = 0; w < FD_CW; ++w) s = f2_add(s, F2{ssq_red[(w * 4 + tid) * 2], ssq_red[(w * 4 + tid) * 2 + 1]});
      atomicAdd(dst + tid, (double)s.hi + (double)s.lo);
    }
  };
#pragma unroll
  for (int t = 0; t < NT; ++t) ssq[t] = F2{0.f, 0.f};

  for (int l = 0; l < a.L; ++l) {
    const FusedLayer& Lw = a.layers[l];
    // ------------------------------------------------------------ QKV
    if (l == 0) {
      if (c == 0) {  // h = x; the step's sums of squares start at zero
        const Dt* x = static_cast<const Dt*>(a.x);
        for (int i = tid; i < T * hid / EPV; i += FD_CT)
          __stcg(reinterpret_cast<uint4*>(hbuf) + i, ldcg16(x + (size_t)i * EPV));
        for (int i = tid; i < (2 * a.L + 1) * T; i += FD_CT) a.sumsq[i] = 0.0;
      }
      stage_norm<Dt>(xs, static_cast<const Dt*>(a.x), static_cast<const Dt*>(Lw.in_norm), nullptr, T, hid, a.eps,
                     red, s_rs);
    } else {
      stage_norm<Dt>(xs, hbuf, static_cast<const Dt*>(Lw.in_norm), a.sumsq + (size_t)(2 * l) * T, T, hid, a.eps,
                     red, s_rs);
    }
    gemv_phase(sp_qkv, rb_hid, false, hid, Lw.qkv_s, Lw.qkv_b, 0, [&](int r0, int n, float (&res)[FD_RM][NT]) {
#pragma unroll
      for (int r = 0; r < FD_RM; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (r < n && lane == r * NT + t) stcg_e<Dt>(qkvb + (size_t)t * qkv_n + r0 + r, res[r][t]);
    });
    grid_barrier(a, ++nbar);

    // ------------------------------------------------------------ ATTN
    {
      Dt* kc = static_cast<Dt*>(a.kc) + (size_t)l * a.layer_stride;
      Dt* vc = static_cast<Dt*>(a.vc) + (size_t)l * a.layer_stride;
      for (int it = c; it < S.n_items; it += nc) {
        int b, ch, j;
        item_of(S, KV, it, b, ch, j);
        const QBlk q = S.qb[b];
        const int nkeys = item_keys(q, ch);
        const int nunits = (nkeys + FD_KW - 1) / FD_KW;
        const int nq = q.nrows * G;
        if (warp < NQ) {  // queries: RMSNorm + RoPE (warp per query vector)
          float x[DPL];
          if (warp < nq) {
            const int row = q.row0 + warp / G, hh = j * G + warp % G;
            const Dt* src = qkvb + (size_t)row * qkv_n + (size_t)hh * D + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) x[e] = ldcg_e<Dt>(src + e);
            norm_rope_head<Dt, D>(x, static_cast<const Dt*>(Lw.q_norm), a.cos_t, a.sin_t, q.pos0 + warp / G, a.eps);
          } else {
#pragma unroll
            for (int e = 0; e < DPL; ++e) x[e] = 0.f;
          }
          store_lane_vec<DPL>(qs + warp * D + lane * DPL, x);
        }
        csync();
        float m_w[NQ], l_w[NQ], o_w[NQ][DPL];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          m_w[i] = -CUDART_INF_F;
          l_w[i] = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) o_w[i][e] = 0.f;
        }
        if (warp < nunits) {
          const int gg = g + warp;
          live = unit_wait(ring.full, s_issued, ring.ns, gg, a, 24, live);
          uint8_t* slot = ring.base + (size_t)(gg % ring.ns) * ring.sb;
          Dt* Kt = reinterpret_cast<Dt*>(slot);
          Dt* Vt = reinterpret_cast<Dt*>(slot + kv_unit);
          const int kb = ch * FD_ITEM + warp * FD_KW;  // position of this warp's first key
          const int nk = min(FD_KW, ch * FD_ITEM + nkeys - kb);
          if (live) {
            // keys appended in this step among this warp's keys
            const int n0 = max(kb, q.seg_pos0), n1 = min(kb + nk, q.seg_pos0 + q.seg_n);
            for (int u = n0; u < n1; ++u) {
              const int row = q.seg_row0 + (u - q.seg_pos0);
              float x[DPL], v[DPL];
              const Dt* ksrc = qkvb + (size_t)row * qkv_n + (size_t)(H + j) * D + lane * DPL;
              const Dt* vsrc = qkvb + (size_t)row * qkv_n + (size_t)(H + KV + j) * D + lane * DPL;
#pragma unroll
              for (int e = 0; e < DPL; ++e) { x[e] = ldcg_e<Dt>(ksrc + e); v[e] = ldcg_e<Dt>(vsrc + e); }
              norm_rope_head<Dt, D>(x, static_cast<const Dt*>(Lw.k_norm), a.cos_t, a.sin_t, u, a.eps);
              const bool owner = row >= q.row0 && row < q.row0 + q.nrows;
              const size_t goff = (size_t)q.seq * a.seq_stride + ((size_t)j * a.capacity + u) * D + lane * DPL;
#pragma unroll
              for (int e = 0; e < DPL; ++e) {
                Kt[(u - kb) * D + lane * DPL + e] = from_f<Dt>(x[e]);
                Vt[(u - kb) * D + lane * DPL + e] = from_f<Dt>(v[e]);
                if (owner) {
                  kc[goff + e] = from_f<Dt>(x[e]);
                  vc[goff + e] = from_f<Dt>(v[e]);
                }
              }
            }
            __syncwarp();
            // scores: LPK lanes per key, KPS keys per step
            const int sub_l = lane % LPK, kq = lane / LPK;
#pragma unroll
            for (int st = 0; st < FD_KW / KPS; ++st) {
              const int u = st * KPS + kq;
              float kv[EPV];
              if (u < nk) {
                Vec16<Dt>::unpack(*reinterpret_cast<const uint4*>(Kt + (size_t)u * D + sub_l * EPV), kv);
              } else {
#pragma unroll
                for (int e = 0; e < EPV; ++e) kv[e] = 0.f;
              }
#pragma unroll
              for (int i = 0; i < NQ; ++i) {
                if (i < nq) {
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
                  if (sub_l == 0)
                    ps[i * FD_KW + u] = (u < nk && kb + u <= q.pos0 + i / G) ? d * a.scale : -CUDART_INF_F;
                }
              }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
              if (i < nq) {
                const float sv = lane < FD_KW ? ps[i * FD_KW + lane] : -CUDART_INF_F;
                const float mm = warp_max(sv);
                const float p = (sv == -CUDART_INF_F) ? 0.f : expf(sv - mm);
                const float ll = warp_sum(p);
                if (lane < FD_KW) ps[i * FD_KW + lane] = p;
                m_w[i] = mm;
                l_w[i] = ll;
              }
            }
            __syncwarp();
            for (int u = 0; u < nk; ++u) {
              float v[DPL];
              load_lane_vec<Dt, DPL>(Vt + (size_t)u * D + lane * DPL, v);
#pragma unroll
              for (int i = 0; i < NQ; ++i) {
                if (i < nq) {
                  const float p = ps[i * FD_KW + u];
#pragma unroll
                  for (int e = 0; e < DPL; ++e) o_w[i][e] = fmaf(p, v[e], o_w[i][e]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive1(&ring.empty[gg % ring.ns]);
        }
        float* mine = wp + (size_t)warp * FD_NQ * WPc;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          if (i < nq) {
            store_lane_vec<DPL>(mine + i * WPc + lane * DPL, o_w[i]);
            if (lane == 0) { mine[i * WPc + D] = m_w[i]; mine[i * WPc + D + 1] = l_w[i]; }
          }
        }
        g += nunits;
        csync();
        // merge the warp partials into the item's partial
        const size_t part0 = ((size_t)(q.part_base + ch) * KV + j) * FD_NQ;
        if (warp < nq) {
          const int i = warp;
          const float mm = lane < FD_CW ? wp[((size_t)lane * FD_NQ + i) * WPc + D] : -CUDART_INF_F;
          const float M = warp_max(mm);
          const float f = (mm == -CUDART_INF_F) ? 0.f : expf(mm - M);
          const float L = warp_sum(lane < FD_CW ? f * wp[((size_t)lane * FD_NQ + i) * WPc + D + 1] : 0.f);
          if (lane < FD_CW) mrg[i * MP + lane] = f;
          if (lane == 0) {
            __stcg(a.part_ml + (part0 + i) * 2, M);
            __stcg(a.part_ml + (part0 + i) * 2 + 1, L);
          }
        }
        csync();
        for (int idx = tid; idx < nq * D; idx += FD_CT) {
          const int i = idx / D, d = idx % D;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < FD_CW; ++w) v = fmaf(wp[((size_t)w * FD_NQ + i) * WPc + d], mrg[i * MP + w], v);
          __stcg(a.part_o + (part0 + i) * D + d, v);
        }
        __threadfence();
        csync();
        if (tid == 0) {
          const int prev = atomicAdd(a.counters + b * KV + j, 1);
          s_flag = (prev == q.n_chunks - 1);
        }
        csync();
        if (s_flag) {  // last chunk of (query block, kv head): combine
          __threadfence();
          const int ncs = q.n_chunks;
          const size_t pbase = (size_t)q.part_base * KV + j;
          for (int i = warp; i < nq; i += FD_CW) {
            float M = -CUDART_INF_F;
            for (int cc = lane; cc < ncs; cc += 32)
              M = fmaxf(M, __ldcg(a.part_ml + ((pbase + (size_t)cc * KV) * FD_NQ + i) * 2));
            M = warp_max(M);
            float Ls = 0.f;
            for (int cc = lane; cc < ncs; cc += 32) {
              const size_t p = (pbase + (size_t)cc * KV) * FD_NQ + i;
              const float mm = __ldcg(a.part_ml + p * 2);
              Ls = fmaf(__ldcg(a.part_ml + p * 2 + 1), (mm == -CUDART_INF_F) ? 0.f : expf(mm - M), Ls);
            }
            Ls = warp_sum(Ls);
            if (lane == 0) { mrg[i * MP + FD_CW] = M; mrg[i * MP + FD_CW + 1] = Ls; }
          }
          csync();
          for (int idx = tid; idx < nq * D; idx += FD_CT) {
            const int i = idx / D, d = idx % D;
            const float M = mrg[i * MP + FD_CW];
            float v = 0.f;
            for (int cc = 0; cc < ncs; ++cc) {
              const size_t p = (pbase + (size_t)cc * KV) * FD_NQ + i;
              const float mm = __ldcg(a.part_ml + p * 2);
              if (mm != -CUDART_INF_F) v = fmaf(__ldcg(a.part_o + p * D + d), expf(mm - M), v);
            }
            const int row = q.row0 + i / G, head = j * G + i % G;
            stcg_e<Dt>(attnb + ((size_t)row * H + head) * D + d, v / mrg[i * MP + FD_CW + 1]);
          }
          if (tid == 0) a.counters[b * KV + j] = 0;
        }
        csync();
      }
    }
    grid_barrier(a, ++nbar);

    // ------------------------------------------------------------ O
    stage_copy<Dt>(xs, attnb, T, H * D);
    gemv_phase(sp_o, rb_o, false, H * D, Lw.o_s, Lw.o_b, 0, residual_epi);
    flush_ssq(a.sumsq + (size_t)(2 * l + 1) * T);
    grid_barrier(a, ++nbar);

    // ------------------------------------------------------------ GU
    stage_norm<Dt>(xs, hbuf, static_cast<const Dt*>(Lw.post_norm), a.sumsq + (size_t)(2 * l + 1) * T, T, hid,
                   a.eps, red, s_rs);
    gemv_phase(sp_gu, rb_hid, true, hid, Lw.gu_s, Lw.gu_b, I, [&](int r0, int n, float (&res)[FD_RM][NT]) {
      // rows 0..n-1 are gate rows, n..2n-1 the matching up rows
#pragma unroll
      for (int r = 0; r < FD_RM / 2; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (r < n && lane == r * NT + t) {
            float gv = 0.f, uv = 0.f;
#pragma unroll
            for (int rr = 0; rr < FD_RM; ++rr) {
              if (rr == r) gv = res[rr][t];
              if (rr == r + n) uv = res[rr][t];
            }
            const float gg = rd<Dt>(gv), up = rd<Dt>(uv);
            stcg_e<Dt>(mb + (size_t)t * I + r0 + r, rd<Dt>(silu_f(gg)) * up);
          }
    });
    grid_barrier(a, ++nbar);

    // ------------------------------------------------------------ DOWN
    stage_copy<Dt>(xs, mb, T, I);
    gemv_phase(sp_dn, rb_i, false, I, Lw.down_s, Lw.down_b, 0, residual_epi);
    flush_ssq(a.sumsq + (size_t)(2 * l + 2) * T);
    grid_barrier(a, ++nbar);
  }

  // ---------------------------------------------------------------- final RMSNorm
  {
    const double* ss = a.sumsq + (size_t)(2 * a.L) * T;
    const Dt* gain = static_cast<const Dt*>(a.final_norm);
    Dt* out = static_cast<Dt*>(a.out);
    const int nch = T * hid / EPV;
    for (int cidx = c * FD_CT + tid; cidx < nch; cidx += nc * FD_CT) {
      const int t = cidx * EPV / hid, k = cidx * EPV - t * hid;
      const F2 rs = rms_scale2(f2_from_double(__ldcg(ss + t)), hid, a.eps);
      float hv[EPV], gv[EPV], o[EPV];
      Vec16<Dt>::unpack(ldcg16(hbuf + (size_t)cidx * EPV), hv);
      Vec16<Dt>::unpack(ld16(gain + k), gv);
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[e] = rms_apply2<Dt>(hv[e], rs, gv[e]);
      *reinterpret_cast<uint4*>(out + (size_t)cidx * EPV) = Vec16<Dt>::pack(o);
    }
  }
}

// Cooperative launch of one instantiation (head_dim 128).
template <typename Dt, int WF, int NT, int NQ>
cudaError_t fd_launch(const LaunchCtx& ctx, const FusedArgs& a, int grid, size_t smem) {
  auto kern = decode_fused_kernel<Dt, WF, NT, 128, NQ>;
  static size_t configured = 0;  // dynamic shared memory the kernel is enabled for
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, FD_THREADS, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(FD_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// The instantiations of one (activation dtype, weight format): T rows and
// NQ = 2 (one row, G <= 2) or 8 query vectors per block.
template <typename Dt, int WF>
cudaError_t fd_dispatch(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq) {
  if (a.T == 1 && nq <= 2) return fd_launch<Dt, WF, 1, 2>(c, a, grid, smem);
  switch (a.T) {
    case 1: return fd_launch<Dt, WF, 1, 8>(c, a, grid, smem);
    case 2: return fd_launch<Dt, WF, 2, 8>(c, a, grid, smem);
    case 3: return fd_launch<Dt, WF, 3, 8>(c, a, grid, smem);
    case 4: return fd_launch<Dt, WF, 4, 8>(c, a, grid, smem);
  }
  return cudaErrorInvalidValue;
}

cudaError_t fused_launch_bf16(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq);
cudaError_t fused_launch_bf16_u8(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq);
cudaError_t fused_launch_f32(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq);

}  // namespace fused
}  // namespace q3
