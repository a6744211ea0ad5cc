// router.cu -- the sigmoid top-K router that feeds the routed expert linear.
//
// ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
// section 1, the sigmoid router; the Hy3 decode write-up, the router after
// its logits.) Per token t and expert e: score = sigmoid(logit[t,e]) in
// float32, choice = score + bias[e]; the K experts of highest choice, highest
// first, ties to the lower index (a stable descending sort); their weights
// are the raw scores (the bias only steers the choice), summed left to right
// in float32, each divided by that sum plus 1e-20 and multiplied by the
// scaling factor.
//
// One warp per token (router_token_warp in router.cuh): an expert whose
// choice is NaN is never taken; slots left without an expert get id -1 and
// weight 0 (the linear skips such pairs).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "router.cuh"

namespace mxfp4el {
namespace {

__global__ void __launch_bounds__(kRouterThreads)
router_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int64_t T,
                   int E, int K, float scaling, int32_t* __restrict__ sel,
                   float* __restrict__ p) {
  extern __shared__ float router_smem[];   // per warp: E raw, E choice, K chosen scores
  pdl_launch_dependents();
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5;
  float* scratch = router_smem + (size_t)warp * router_scratch_floats(E, K);
  for (int64_t t = (int64_t)blockIdx.x * warps + warp; t < T; t += (int64_t)gridDim.x * warps)
    router_token_warp(logits + t * E, bias, E, K, scaling, scratch, sel + t * K, p + t * K);
}

}  // namespace

int router_warps_per_block(int64_t E, int64_t K) {
  const int64_t per_warp = (2 * E + K) * (int64_t)sizeof(float);
  return (int)std::max<int64_t>(0, std::min<int64_t>(kRouterThreads / 32,
                                                     kRouterSmemLimit / per_warp));
}

cudaError_t launch_router(const float* logits, const float* bias, int64_t T, int64_t E,
                          int64_t K, float scaling, int32_t* sel, float* p,
                          cudaStream_t stream) {
  if (T == 0 || K == 0) return cudaSuccess;
  const int warps = router_warps_per_block(E, K);
  if (warps <= 0) return cudaErrorInvalidValue;
  const int64_t blocks = std::min<int64_t>((T + warps - 1) / warps, 152 * 16);
  const size_t smem = (size_t)warps * (2 * E + K) * sizeof(float);
  router_topk_kernel<<<(unsigned)blocks, warps * 32, smem, stream>>>(
      logits, bias, T, (int)E, (int)K, scaling, sel, p);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace mxfp4el
