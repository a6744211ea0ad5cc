// swiglu.cu -- the activation between the two projections of the MXFP4
// SwiGLU expert.
//
// ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
// section 1, the expert shape: down(silu(gate(x)) * up(x)) per routed
// expert, accumulated with the routing weight in float32; the Hy3 decode
// write-up: the gate and up projections stacked along their output rows.)
// The gate/up projection is the routed linear over 2F stacked rows (gate
// rows 0..F-1, up rows F..2F-1), leaving float32 partial results per pair
// and group column. Per pair and intermediate index f:
//   g = sum of the gate row's columns, u = sum of the up row's columns (in
//   column order, as the combine sums them), h = silu(g) * u with
//   silu(g) = g / (1 + exp(-g)), in float32, rounded once to the token dtype.
// The down projection then runs with every pair as its own token; its
// selection is a copy of the ids in which an out-of-range id becomes expert
// 0 with h = 0 (the combine, which reads the original ids, skips that pair),
// so an invalid id is counted once per call.
#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

template <typename Tok, typename Idx>
__global__ void __launch_bounds__(256)
swiglu_kernel(const float* __restrict__ part, int ncol, const Idx* __restrict__ sel, int64_t E,
              int64_t P, int64_t F, Tok* __restrict__ h, int32_t* __restrict__ sel2) {
  pdl_wait();                  // the gate/up projection's partial results are complete
  pdl_launch_dependents();
  const int64_t n = P * F;
  const int64_t row = (int64_t)ncol * 2 * F;       // floats per pair
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pair = idx / F, f = idx - pair * F;
    const long long e = (long long)sel[pair];
    const bool valid = e >= 0 && e < E;
    float v = 0.f;
    if (valid) {
      const float* pp = part + pair * row + f;
      float g = pp[0], u = pp[F];
      for (int c = 1; c < ncol; ++c) {
        g += pp[(int64_t)c * 2 * F];
        u += pp[(int64_t)c * 2 * F + F];
      }
      v = g / (1.f + expf(-g)) * u;
    }
    h[idx] = TokenIO<Tok>::from_f32(v);
    if (f == 0) sel2[pair] = valid ? (int32_t)e : 0;
  }
}

template <typename Tok, typename Idx>
cudaError_t launch_typed(const float* part, int ncol, const Idx* sel, int64_t E, int64_t P,
                         int64_t F, Tok* h, int32_t* sel2, cudaStream_t stream) {
  const int64_t n = P * F;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  return launch_after_previous(swiglu_kernel<Tok, Idx>, dim3((unsigned)blocks), dim3(256), 0,
                               stream, part, ncol, sel, E, P, F, h, sel2);
}

}  // namespace

cudaError_t launch_swiglu(const float* part, int ncol, const void* sel, int index_dtype,
                          int64_t E, int64_t P, int64_t F, int token_dtype, void* h,
                          int32_t* sel2, cudaStream_t stream) {
  if (token_dtype == kTokenBF16) {
    auto* hb = static_cast<__nv_bfloat16*>(h);
    if (index_dtype == kIndexI64)
      return launch_typed(part, ncol, static_cast<const int64_t*>(sel), E, P, F, hb, sel2, stream);
    return launch_typed(part, ncol, static_cast<const int32_t*>(sel), E, P, F, hb, sel2, stream);
  }
  auto* hf = static_cast<float*>(h);
  if (index_dtype == kIndexI64)
    return launch_typed(part, ncol, static_cast<const int64_t*>(sel), E, P, F, hf, sel2, stream);
  return launch_typed(part, ncol, static_cast<const int32_t*>(sel), E, P, F, hf, sel2, stream);
}

}  // namespace mxfp4el
