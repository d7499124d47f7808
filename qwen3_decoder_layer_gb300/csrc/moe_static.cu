// qwen3_moe_layer_static: the MoE block of qwen3_moe_layer with its scratch
// memory (router logits, the expert histogram and permutation, the expert
// activations and the per-slot expert outputs) held in a fixed-size array in
// device global memory that belongs to this library's image, so that a call
// allocates nothing.  The KV cache and weights are untouched; only the
// handle's configuration and weight pointers are read.
//
// The array is a host-side stand-in in host code, not a device address: the
// address the kernels get comes from cudaGetSymbolAddress, looked up once per
// device (with that device current) on the first call there and kept.
#include <cuda_runtime.h>

#include <mutex>

#include "qwen3.h"

namespace q3 {
int handle_device(const qwen3_handle* h);
qwen3_status report_error(qwen3_handle* h, qwen3_status s, const char* msg);
qwen3_status moe_layer_on_scratch(qwen3_handle* h, int32_t layer, const void* y, int32_t T, void* out,
                                  int32_t* topk_idx, float* topk_w, void* stream, void* scratch,
                                  size_t scratch_bytes);
}  // namespace q3

namespace {

// 4 MiB on every GPU that loads the library, for as long as the process runs.
constexpr size_t kMoeStaticScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_moe_scratch[kMoeStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_moe_scratch, per device ordinal

}  // namespace

extern "C" QWEN3_API qwen3_status qwen3_moe_layer_static(qwen3_handle* h, int32_t layer, const void* y, int32_t T,
                                                         void* out, int32_t* topk_idx, float* topk_w,
                                                         void* stream) {
  if (!h) return QWEN3_E_ARG;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return q3::report_error(h, QWEN3_E_CUDA, "cudaGetDevice failed");
  }
  if (dev != q3::handle_device(h))
    return q3::report_error(h, QWEN3_E_ARG, "the handle's device must be the current device");
  if (dev < 0 || dev >= kMaxDevices)
    return q3::report_error(h, QWEN3_E_UNSUPPORTED, "device ordinal beyond the static scratch table");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_moe_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return q3::report_error(h, QWEN3_E_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return q3::moe_layer_on_scratch(h, layer, y, T, out, topk_idx, topk_w, stream, scratch, kMoeStaticScratchBytes);
}
