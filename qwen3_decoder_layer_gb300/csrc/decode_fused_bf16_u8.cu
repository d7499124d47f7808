// Instantiations of the fused decode step for bf16 activations with int8 weights.
#include "decode_fused.cuh"

namespace q3 {
namespace fused {

cudaError_t fused_launch_bf16_u8(const LaunchCtx& c, const FusedArgs& a, int grid, size_t smem, int nq) {
  return fd_dispatch<bf16, W_U8>(c, a, grid, smem, nq);
}

}  // namespace fused
}  // namespace q3
