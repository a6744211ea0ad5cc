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
// One warp per token: the raw and choice scores go to shared memory, then K
// rounds of a warp-wide argmax (greater score, or equal score and lower
// index) each take one expert and mark it taken, in shared memory only. An expert whose choice is NaN is
// never taken; slots left without an expert get id -1 and weight 0 (the
// linear skips such pairs).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + expf(-x)); }

// (c, e) beats (bc, be): greater choice, or equal choice and lower index.
__device__ __forceinline__ bool better(float c, int e, float bc, int be) {
  return c > bc || (c == bc && e < be);
}

__global__ void __launch_bounds__(kRouterThreads)
router_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int64_t T,
                   int E, int K, float scaling, int32_t* __restrict__ sel,
                   float* __restrict__ p) {
  extern __shared__ float router_smem[];   // per warp: E raw, E choice, K chosen scores
  pdl_launch_dependents();
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* raw = router_smem + (size_t)warp * (2 * E + K);
  float* choice = raw + E;
  float* chosen = choice + E;
  for (int64_t t = (int64_t)blockIdx.x * warps + warp; t < T; t += (int64_t)gridDim.x * warps) {
    const float* row = logits + t * E;
    for (int e = lane; e < E; e += 32) {
      const float r = sigmoid_f32(row[e]);
      raw[e] = r;
      choice[e] = r + (bias != nullptr ? bias[e] : 0.f);
    }
    __syncwarp();
    for (int k = 0; k < K; ++k) {
      float bc = -INFINITY;
      int be = 0x7fffffff;
      for (int e = lane; e < E; e += 32) {
        const float c = choice[e];
        if (c == c && better(c, e, bc, be)) {   // c == c: not NaN (taken or invalid)
          bc = c;
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float oc = __shfl_xor_sync(kFullMask, bc, o);
        const int oe = __shfl_xor_sync(kFullMask, be, o);
        if (better(oc, oe, bc, be)) {
          bc = oc;
          be = oe;
        }
      }
      if (lane == 0) {
        const bool found = be != 0x7fffffff;
        sel[t * K + k] = found ? be : -1;
        chosen[k] = found ? raw[be] : 0.f;
        if (found) choice[be] = __int_as_float(0x7fffffff);   // NaN: taken
      }
      __syncwarp();
    }
    if (lane == 0) {
      float total = 0.f;
      for (int k = 0; k < K; ++k) total += chosen[k];        // left to right
      for (int k = 0; k < K; ++k) p[t * K + k] = chosen[k] / (total + 1e-20f) * scaling;
    }
    __syncwarp();
  }
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
