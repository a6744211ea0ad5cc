// gemv.cu -- decode-regime routed expert GEMV.
//
// For every selected expert e and each of its tokens t this computes the
// float32 routed result part[t*K+k, o] = sum_i W_e[o, i] x[t, i] with
// W_e[o, 32g + 2j (+1)] = LUT[low (high) nibble of packed[e,o,g,j]] *
// 2^(scales[e,o,g] - 127) (problem statement "MXFP4 Routed Expert Linear",
// Kimi K3, sections "What is stored in one group" to "Reconstruct the matrix
// in the right orientation").
//
// The kernel is bound by HBM: every byte of a selected expert is read once.
//   * CTA = 8 warps over (expert slot u, tile of 8 R output rows); slots past
//     the number of active experts exit at once.
//   * lane = one 32-value group: a 128-bit load brings its 16 packed bytes,
//     one byte load its scale. R rows per warp keep R loads in flight per lane
//     and let the lane's token values be reused across the R rows.
//   * decode in registers: the hardware E2M1 -> f16x2 conversion, widened to
//     f32, then packed f32x2 FMAs against the token; each group's partial is
//     scaled by its exact power of two and accumulated in float32.
//   * the expert's tokens are taken NT at a time; within a pass the decoded
//     group is reused for every token. A later pass re-reads the rows from L2.
//   * one shuffle reduce-scatter sums the R x NT accumulators across lanes.
#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

// Dot product of one packed group (16 bytes = 32 codes) with 32 token values.
// The result is the unscaled group partial sum_j LUT[code_j] * x_j.
__device__ __forceinline__ float dot_group(const uint4& w, const float (&x)[32]) {
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(words[q], h);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // byte 4q+b holds input positions 8q+2b (low nibble) and 8q+2b+1
      const float2 wf = f16x2_to_f32x2(h[b]);
      const float2 xv = make_float2(x[8 * q + 2 * b], x[8 * q + 2 * b + 1]);
      if (b & 1) a1 = ffma2(wf, xv, a1);
      else       a0 = ffma2(wf, xv, a0);
    }
  }
  return (a0.x + a1.x) + (a0.y + a1.y);
}

template <int V> struct Log2 { static constexpr int value = 1 + Log2<V / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

template <typename Tok, int R, int NT>
__global__ void __launch_bounds__(kGemvThreads, 2)
gemv_kernel(const Tok* __restrict__ x, const uint8_t* __restrict__ packed,
            const uint8_t* __restrict__ scales, RoutePlan plan,
            float* __restrict__ part, int G, int O, int I, int K,
            int row_tiles) {
  constexpr int V = R * NT;
  constexpr int L = Log2<V>::value;
  static_assert((1 << L) == V, "R * NT must be a power of two");

  const int u = blockIdx.x / row_tiles;
  const int tile = blockIdx.x - u * row_tiles;
  if (u >= plan.meta[kMetaNumActive]) return;
  const int e = plan.active[u];
  const int seg_beg = plan.offsets[e];
  const int seg_end = plan.offsets[e + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int o0 = (tile * kGemvWarps + warp) * R;
  if (o0 >= O) return;

  const uint8_t* wrow[R];
  const uint8_t* srow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const size_t row = (size_t)e * O + min(o0 + r, O - 1);   // clamp: stay in bounds
    wrow[r] = packed + row * (size_t)G * 16;
    srow[r] = scales + row * (size_t)G;
  }

  for (int base = seg_beg; base < seg_end; base += NT) {
    const int nt = min(NT, seg_end - base);
    const Tok* xrow[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int pair = plan.pair_list[base + min(j, nt - 1)];
      xrow[j] = x + (size_t)(pair / K) * I;
    }
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;

    for (int g = lane; g < G; g += 32) {
      uint4 w[R];
      E8M0 sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) w[r] = ld_stream_u4(wrow[r] + (size_t)g * 16);
#pragma unroll
      for (int r = 0; r < R; ++r) sc[r] = e8m0(srow[r][g]);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if (j < nt) {
          float xf[32];
          TokenIO<Tok>::load32(xrow[j] + (size_t)g * 32, xf);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float d = dot_group(w[r], xf);
            acc[r * NT + j] = fmaf(d * sc[r].pre, sc[r].factor, acc[r * NT + j]);
          }
        }
      }
    }

    const float total = warp_reduce_scatter<V>(acc, lane);
    if ((lane & ((1 << (5 - L)) - 1)) == 0) {
      const int idx = (lane >> (5 - L)) & (V - 1);
      const int r = idx / NT, j = idx - (idx / NT) * NT;
      if (j < nt && o0 + r < O) {
        const int pair = plan.pair_list[base + j];
        part[(size_t)pair * O + o0 + r] = total;
      }
    }
  }
}

constexpr int kRows = 4;     // output rows per warp
constexpr int kTokens = 4;   // tokens per pass

template <typename Tok>
cudaError_t launch_typed(const Tok* x, const uint8_t* packed, const uint8_t* scales,
                         const RoutePlan& plan, float* part, int64_t T, int64_t E,
                         int64_t I, int64_t O, int64_t K, cudaStream_t stream) {
  const int64_t rows_per_cta = (int64_t)kGemvWarps * kRows;
  const int64_t row_tiles = (O + rows_per_cta - 1) / rows_per_cta;
  const int64_t slots = std::min<int64_t>(E, T * K);
  const int64_t blocks = slots * row_tiles;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  gemv_kernel<Tok, kRows, kTokens><<<(unsigned)blocks, kGemvThreads, 0, stream>>>(
      x, packed, scales, plan, part, (int)(I / 32), (int)O, (int)I, (int)K,
      (int)row_tiles);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const void* x, int token_dtype, const uint8_t* packed,
                        const uint8_t* scales, const RoutePlan& plan,
                        float* part, int64_t T, int64_t E, int64_t I,
                        int64_t O, int64_t K, cudaStream_t stream) {
  if (token_dtype == kTokenBF16)
    return launch_typed(static_cast<const __nv_bfloat16*>(x), packed, scales,
                        plan, part, T, E, I, O, K, stream);
  return launch_typed(static_cast<const float*>(x), packed, scales, plan, part,
                      T, E, I, O, K, stream);
}

}  // namespace mxfp4el
