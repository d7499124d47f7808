// Instantiations of the fused decode step for bf16 activations.
#include "decode_fused.cuh"

namespace q3 {
namespace fused {

cudaError_t fused_launch_bf16(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq) {
  return fd_dispatch<bf16, W_DT>(c, a, grid, smem, nq);
}

}  // namespace fused
}  // namespace q3
