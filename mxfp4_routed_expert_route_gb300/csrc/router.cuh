// router.cuh -- the sigmoid top-K router for one token, by one warp.
//
// ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
// section 1, the sigmoid router; the Hy3 decode write-up, the router after
// its logits.) Per expert e: score = sigmoid(logit[e]) in float32, choice =
// score + bias[e]; the K experts of highest choice, highest first, ties to
// the lower index (a stable descending sort); their weights are the raw
// scores (the bias only steers the choice), summed left to right in float32,
// each divided by that sum plus 1e-20 and multiplied by the scaling factor.
//
// The raw and choice scores go to the warp's shared-memory scratch, then K
// rounds of a warp-wide argmax (greater score, or equal score and lower
// index) each take one expert and mark it taken. An expert whose choice is
// NaN is never taken; slots left without an expert get id -1 and weight 0.
#pragma once

#include "common.cuh"

namespace mxfp4el {

__device__ __forceinline__ float router_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

// (c, e) beats (bc, be): greater choice, or equal choice and lower index.
__device__ __forceinline__ bool router_better(float c, int e, float bc, int be) {
  return c > bc || (c == bc && e < be);
}

// Floats of shared-memory scratch one warp needs.
__host__ __device__ constexpr int64_t router_scratch_floats(int64_t E, int64_t K) {
  return 2 * E + K;
}

// Routes one token with the whole warp. `scratch` holds
// router_scratch_floats(E, K) floats of this warp. Lane 0 writes the K ids
// to sel and the K weights to p.
__device__ __forceinline__ void router_token_warp(const float* __restrict__ row,
                                                  const float* __restrict__ bias, int E, int K,
                                                  float scaling, float* scratch, int32_t* sel,
                                                  float* p) {
  const int lane = threadIdx.x & 31;
  float* raw = scratch;
  float* choice = raw + E;
  float* chosen = choice + E;
  for (int e = lane; e < E; e += 32) {
    const float r = router_sigmoid(row[e]);
    raw[e] = r;
    choice[e] = r + (bias != nullptr ? bias[e] : 0.f);
  }
  __syncwarp();
  for (int k = 0; k < K; ++k) {
    float bc = -INFINITY;
    int be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float c = choice[e];
      if (c == c && router_better(c, e, bc, be)) {   // c == c: not NaN (taken or invalid)
        bc = c;
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float oc = __shfl_xor_sync(kFullMask, bc, o);
      const int oe = __shfl_xor_sync(kFullMask, be, o);
      if (router_better(oc, oe, bc, be)) {
        bc = oc;
        be = oe;
      }
    }
    if (lane == 0) {
      const bool found = be != 0x7fffffff;
      sel[k] = found ? be : -1;
      chosen[k] = found ? raw[be] : 0.f;
      if (found) choice[be] = __int_as_float(0x7fffffff);   // NaN: taken
    }
    __syncwarp();
  }
  if (lane == 0) {
    float total = 0.f;
    for (int k = 0; k < K; ++k) total += chosen[k];        // left to right
    for (int k = 0; k < K; ++k) p[k] = chosen[k] / (total + 1e-20f) * scaling;
  }
  __syncwarp();
}

}  // namespace mxfp4el
