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
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Four consecutive h values of one pair, stored in the token dtype.
__device__ __forceinline__ void store4(float* h, float4 v) { *reinterpret_cast<float4*>(h) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* h, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(h) = w;
}

template <typename Tok, typename Idx>
__global__ void __launch_bounds__(256)
swiglu_kernel(const float* __restrict__ part, int ncol, const Idx* __restrict__ sel, int64_t E,
              int64_t P, int F, Tok* __restrict__ h, int32_t* __restrict__ sel2) {
  pdl_wait();                  // the gate/up projection's partial results are complete
  pdl_launch_dependents();
  // x: four consecutive intermediate indices f per thread (F is a multiple
  // of 32, so a pair's rows and columns start on 16-byte boundaries); y:
  // pairs, in steps of the grid's height.
  const int f = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  const int64_t col = 2 * (int64_t)F;              // floats per group column of a pair
  for (int64_t pair = blockIdx.y; pair < P; pair += gridDim.y) {
    const long long e = (long long)sel[pair];
    const bool valid = e >= 0 && e < E;
    if (f < F) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (valid) {
        const float* pp = part + pair * ncol * col + f;
        float4 g = __ldg(reinterpret_cast<const float4*>(pp));
        float4 u = __ldg(reinterpret_cast<const float4*>(pp + F));
        for (int c = 1; c < ncol; ++c) {         // group columns in order
          const float4 gc = __ldg(reinterpret_cast<const float4*>(pp + c * col));
          const float4 uc = __ldg(reinterpret_cast<const float4*>(pp + c * col + F));
          g.x += gc.x; g.y += gc.y; g.z += gc.z; g.w += gc.w;
          u.x += uc.x; u.y += uc.y; u.z += uc.z; u.w += uc.w;
        }
        v = make_float4(silu_times(g.x, u.x), silu_times(g.y, u.y), silu_times(g.z, u.z),
                        silu_times(g.w, u.w));
      }
      store4(h + pair * F + f, v);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) sel2[pair] = valid ? (int32_t)e : 0;
  }
}

template <typename Tok, typename Idx>
cudaError_t launch_typed(const float* part, int ncol, const Idx* sel, int64_t E, int64_t P,
                         int64_t F, Tok* h, int32_t* sel2, cudaStream_t stream) {
  if (P == 0 || F == 0) return cudaSuccess;
  const int64_t bx = (F / 4 + 255) / 256;
  // About 16 blocks per SM in all; each block row loops over its pairs.
  const int64_t by = std::max<int64_t>(1, std::min<int64_t>({P, 65535, (152 * 16 + bx - 1) / bx}));
  return launch_after_previous(swiglu_kernel<Tok, Idx>, dim3((unsigned)bx, (unsigned)by),
                               dim3(256), 0, stream, part, ncol, sel, E, P, (int)F, h, sel2);
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
