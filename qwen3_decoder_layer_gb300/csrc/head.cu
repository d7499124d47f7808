// The steps on either side of the decoder stack:
//  * embedding rows (maya2_mlx/backbone.py, Backbone.embed_tokens: the rows of
//    the embedding table at the token ids, in the model dtype);
//  * the pooled sentence vector (@mlx-bun/inference qwen3.ts, embedPooled: the
//    last row's final-norm hidden state over its L2 norm, the square, sum,
//    square root and divide each an array operation in the model dtype).
// The output head itself (Backbone.cb0_logits) is a GEMV / GEMM with the
// EPI_STORE_RF32 epilogue of gemv.cu and gemm_simt.cu.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

template <typename Dt>
__global__ void __launch_bounds__(256) embed_gather_kernel(EmbedArgs a) {
  constexpr int V = Vec16<Dt>::N;
  pdl_wait();
  pdl_launch();
  const int t = blockIdx.x;
  const Dt* src = static_cast<const Dt*>(a.table) + (size_t)a.ids[t] * a.hidden;
  Dt* dst = static_cast<Dt*>(a.out) + (size_t)t * a.hidden;
  for (int k = threadIdx.x * V; k < a.hidden; k += blockDim.x * V)
    *reinterpret_cast<uint4*>(dst + k) = ld16(src + k);
}

// One block: sq = R(v v) per element, ss = R(sum sq) with the sum accumulated
// in fp32 (fixed order: per-thread partials, then the block tree), n =
// R(sqrt(ss)), out = R(v / n) with a correctly rounded fp32 division.
template <typename Dt>
__global__ void __launch_bounds__(256) l2_pool_kernel(L2PoolArgs a) {
  __shared__ float red[32];
  pdl_wait();
  pdl_launch();
  const Dt* v = static_cast<const Dt*>(a.row);
  float part = 0.f;
  for (int k = threadIdx.x; k < a.hidden; k += blockDim.x) {
    const float x = to_f(v[k]);
    part += rd<Dt>(x * x);
  }
  const float ss = rd<Dt>(block_sum(part, red));
  const float nrm = rd<Dt>(__fsqrt_rn(ss));
  Dt* out = static_cast<Dt*>(a.out);
  for (int k = threadIdx.x; k < a.hidden; k += blockDim.x) out[k] = from_f<Dt>(__fdiv_rn(to_f(v[k]), nrm));
}

// The bounded-wait self test: an mbarrier expecting one arrival that never
// comes.  mbar_wait gives up after its limit (about a second), writes the code
// and the kernel returns; nothing traps and the context stays usable.
__global__ void wait_probe_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, err, kWaitProbeCode);
  }
}

}  // namespace

cudaError_t launch_wait_probe(cudaStream_t s, int* err) {
  wait_probe_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_embed_gather(const LaunchCtx& c, int dt, const EmbedArgs& a) {
  if (a.n < 1) return cudaSuccess;
  if (dt == DT_BF16) return launch_k(embed_gather_kernel<bf16>, dim3(a.n), dim3(256), 0, c, a);
  return launch_k(embed_gather_kernel<float>, dim3(a.n), dim3(256), 0, c, a);
}

cudaError_t launch_l2_pool(const LaunchCtx& c, int dt, const L2PoolArgs& a) {
  if (dt == DT_BF16) return launch_k(l2_pool_kernel<bf16>, dim3(1), dim3(256), 0, c, a);
  return launch_k(l2_pool_kernel<float>, dim3(1), dim3(256), 0, c, a);
}

}  // namespace q3
