// static_scratch.cu -- an entry point for callers that cannot allocate.
//
// Some callers must not allocate device memory at all once they are running:
// a serving process that fixes its whole memory budget at start-up, a plugin
// inside a host framework that owns every device allocation, or code that
// runs where cudaMalloc is forbidden or may fail. They cannot use
// mxfp4_expert_linear (which grows a library-owned buffer) and may have no
// buffer to hand to mxfp4_expert_linear_with_workspace.
//
// mxfp4_expert_linear_static_scratch runs the same kernels with their scratch
// (routing lists and float32 partials) placed in a fixed array compiled into
// the library: kStaticScratchBytes of device memory on every GPU that loads
// the library, held until the process exits. The call allocates nothing.
//
// In host code the array's name is only a host-side stand-in for the device
// symbol: it is not a device address. The device address is looked up once
// per device, with that device current, by cudaGetSymbolAddress, and that
// address is what the kernels receive. The looked-up address is kept for the
// life of the process, so this entry point must not be used on a device
// after cudaDeviceReset (or any other teardown of its primary context).
#include <mutex>

#include "../../include/mxfp4_expert_linear.h"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;   // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (set-up on first
// use per device). Returns MXFP4EL_OK or MXFP4EL_ERR_CUDA.
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4EL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXFP4EL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return MXFP4EL_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return MXFP4EL_OK;
}

}  // namespace
}  // namespace mxfp4el

extern "C" size_t mxfp4_expert_linear_static_scratch_bytes(void) {
  return mxfp4el::kStaticScratchBytes;
}

extern "C" int mxfp4_expert_linear_static_scratch(
    const void* latent_tokens, const uint8_t* packed_weights,
    const uint8_t* scale_bytes, const void* selected_experts,
    const float* mixture_weights, const void* shared_output, void* out,
    int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, int token_dtype,
    int index_dtype, void* stream) {
  // The same checks, in the same order, as the other entry points; only a
  // call they accept can be refused for its size.
  const int rc = mxfp4el::validate_linear(latent_tokens, packed_weights, scale_bytes,
                                          selected_experts, mixture_weights, shared_output,
                                          out, T, E, I, O, K, token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  const size_t need = mxfp4_expert_linear_workspace_size(T, E, I, O, K, token_dtype);
  if (need == (size_t)-1 || need > mxfp4el::kStaticScratchBytes) return MXFP4EL_ERR_TOO_LARGE;
  void* scratch = nullptr;
  if (need > 0) {
    const int arc = mxfp4el::scratch_address(&scratch);
    if (arc != MXFP4EL_OK) return arc;
  }
  return mxfp4_expert_linear_with_workspace(
      latent_tokens, packed_weights, scale_bytes, selected_experts,
      mixture_weights, shared_output, out, T, E, I, O, K, token_dtype,
      index_dtype, scratch, mxfp4el::kStaticScratchBytes, stream);
}
