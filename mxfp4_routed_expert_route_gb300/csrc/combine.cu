// combine.cu -- deterministic combine of the routed results.
//
//   out[t, o] = round( y_shared[t, o] + sum_{k = 0}^{K-1} p[t, k] * part[t*K+k, o] )
//
// where part[t*K+k, o] is itself the sum, in column order c = 0..ncol-1, of
// the partial results the GEMV wrote for the input-group columns.
//
// ("Route, weight, and add the shared path", problem statement "MXFP4 Routed
// Expert Linear", Kimi K3: start from the shared output and add the weighted
// routed contributions.) The sum runs in float32 in slot order k = 0..K-1 and
// is rounded once to the token dtype, so the result does not depend on which
// kernel or which CTA produced each part. Pairs whose expert id is outside
// [0, E) contribute nothing. combine_vec_kernel gives each warp a segment of
// 128 outputs of one token, four per lane with 16-byte loads of the
// partial results; combine_kernel, a grid-stride elementwise pass, serves
// widths that are not a multiple of 4 and unaligned buffers. Both evaluate
// the same expression in the same order.
#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

template <typename Tok, typename Idx>
__global__ void __launch_bounds__(256)
combine_kernel(const Tok* __restrict__ ys, const Idx* __restrict__ sel,
               const float* __restrict__ p, const float* __restrict__ part, int ncol,
               Tok* __restrict__ out, int64_t T, int64_t O, int K, int64_t E) {
  pdl_wait();                  // the GEMV's partial results are complete
  const int64_t n = T * O;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / O;
    const int64_t o = idx - t * O;
    float acc = TokenIO<Tok>::to_f32(ys[idx]);
    for (int k = 0; k < K; ++k) {
      const int64_t pk = t * K + k;
      const long long e = (long long)sel[pk];
      if (e >= 0 && e < E) {
        const float* pp = part + pk * ncol * O + o;
        float v = pp[0];
        for (int c = 1; c < ncol; ++c) v += pp[(int64_t)c * O];
        acc = fmaf(p[pk], v, acc);
      }
    }
    out[idx] = TokenIO<Tok>::from_f32(acc);
  }
}

// Four consecutive token values as float32, and back (rounded once).
__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xffff0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xffff0000u);
}
__device__ __forceinline__ void store4(float* p, const float (&x)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&x)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&a);
  v.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = v;
}

constexpr int kVecLanes = 32;   // one warp per segment of 4 * 32 outputs
constexpr int kSlotBatch = 4;   // slots whose loads are issued together

// Ids and weights of slots [k0, k0 + n) of pair row t*K (n <= kSlotBatch).
struct SlotBatch {
  bool valid[kSlotBatch];
  float w[kSlotBatch];
};
template <typename Idx>
__device__ __forceinline__ SlotBatch load_slots(const Idx* __restrict__ sel,
                                                const float* __restrict__ p, int64_t E,
                                                int64_t pk0, int n) {
  SlotBatch b;
#pragma unroll
  for (int j = 0; j < kSlotBatch; ++j) {
    const long long e = j < n ? (long long)sel[pk0 + j] : -1;
    b.valid[j] = e >= 0 && e < E;
    b.w[j] = j < n ? p[pk0 + j] : 0.f;
  }
  return b;
}

// Adds those slots' partial results to acc in slot order, each slot's
// columns summed in column order first. kCols (the GEMV's partials, ncol > 1):
// the loads go out four columns of the batch (16 vectors) at a time, so a row
// of ncol columns costs ceil(ncol/4) round trips to L2 instead of ncol. One
// column (the tensor-core GEMM's partials, HBM-bound at prefill sizes): one
// vector per slot, few registers, many warps per SM.
constexpr int kColBatch = 4;
template <bool kCols>
__device__ __forceinline__ void add_slots(const SlotBatch& b, const float* __restrict__ part,
                                          int ncol, int64_t O, int64_t pk0, int64_t o,
                                          float (&acc)[4]) {
  const int64_t row = (int64_t)ncol * O;          // floats per pair
  const float* base = part + pk0 * row + o;
  float4 s[kSlotBatch];
  if constexpr (!kCols) {
#pragma unroll
    for (int j = 0; j < kSlotBatch; ++j)
      s[j] = b.valid[j] ? __ldcs(reinterpret_cast<const float4*>(base + j * row))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    for (int c0 = 0; c0 < ncol; c0 += kColBatch) {
      float4 u[kColBatch][kSlotBatch];
#pragma unroll
      for (int cc = 0; cc < kColBatch; ++cc) {
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
          u[cc][j] = b.valid[j] && c0 + cc < ncol
                         ? __ldcs(reinterpret_cast<const float4*>(base + j * row +
                                                                  (int64_t)(c0 + cc) * O))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int cc = 0; cc < kColBatch; ++cc) {
        if (c0 + cc >= ncol) break;
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
          if (c0 + cc == 0) {
            s[j] = u[cc][j];
          } else {
            s[j].x += u[cc][j].x; s[j].y += u[cc][j].y;
            s[j].z += u[cc][j].z; s[j].w += u[cc][j].w;
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kSlotBatch; ++j) {
    if (b.valid[j]) {
      acc[0] = fmaf(b.w[j], s[j].x, acc[0]);
      acc[1] = fmaf(b.w[j], s[j].y, acc[1]);
      acc[2] = fmaf(b.w[j], s[j].z, acc[2]);
      acc[3] = fmaf(b.w[j], s[j].w, acc[3]);
    }
  }
}

template <typename Tok, typename Idx, bool kCols>
__global__ void __launch_bounds__(256)
combine_vec_kernel(const Tok* __restrict__ ys, const Idx* __restrict__ sel,
                   const float* __restrict__ p, const float* __restrict__ part, int ncol,
                   Tok* __restrict__ out, int64_t T, int64_t O, int K, int64_t E,
                   int prefetch) {
  const int64_t nv = O / 4;                         // 4-wide vectors per token row
  const int64_t segs = (nv + kVecLanes - 1) / kVecLanes;
  const int64_t tasks = T * segs;
  const int warps = blockDim.x / 32, lane = threadIdx.x & 31;
  const int64_t first = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
  float acc0[4] = {0.f, 0.f, 0.f, 0.f};
  SlotBatch b0 = {};
  const bool early = prefetch != 0 && first < tasks;
  if (early) {
    const int64_t t = first / segs;
    const int64_t v = (first - t * segs) * kVecLanes + lane;
    if (v < nv) {
      load4(ys + t * O + 4 * v, acc0);
      b0 = load_slots(sel, p, E, t * K, min(kSlotBatch, K));
    }
  }
  pdl_wait();                  // the linear kernel's partial results are complete
  for (int64_t task = first; task < tasks; task += (int64_t)gridDim.x * warps) {
    const int64_t t = task / segs;
    const int64_t v = (task - t * segs) * kVecLanes + lane;
    if (v >= nv) continue;
    const int64_t o = 4 * v;
    const bool pre = early && task == first;
    float acc[4];
    if (pre) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = acc0[i];
    } else {
      load4(ys + t * O + o, acc);
    }
    for (int k0 = 0; k0 < K; k0 += kSlotBatch) {
      const int n = min(kSlotBatch, K - k0);
      const SlotBatch b = pre && k0 == 0 ? b0 : load_slots(sel, p, E, t * K + k0, n);
      add_slots<kCols>(b, part, ncol, O, t * K + k0, o, acc);
    }
    store4(out + t * O + o, acc);
  }
}

template <typename Tok, typename Idx>
cudaError_t launch_typed(const Tok* ys, const Idx* sel, const float* p,
                         const float* part, int ncol, Tok* out, int64_t T, int64_t E,
                         int64_t O, int64_t K, bool prefetch, cudaStream_t stream) {
  const int64_t n = T * O;
  if (n == 0) return cudaSuccess;
  const uintptr_t tok_align = 4 * sizeof(Tok);
  if (O % 4 == 0 && reinterpret_cast<uintptr_t>(ys) % tok_align == 0 &&
      reinterpret_cast<uintptr_t>(out) % tok_align == 0 &&
      reinterpret_cast<uintptr_t>(part) % 16 == 0) {
    const int64_t tasks = T * ((O / 4 + kVecLanes - 1) / kVecLanes);
    const int64_t blocks = std::min<int64_t>((tasks + 7) / 8, 152 * 8);
    // The early loads only shorten the path when each warp has one task
    // (small batches); with many tasks per warp the combine is bandwidth-bound.
    prefetch = prefetch && tasks <= blocks * 8;
    if (ncol > 1)
      return launch_after_previous(combine_vec_kernel<Tok, Idx, true>, dim3((unsigned)blocks),
                                   dim3(256), 0, stream, ys, sel, p, part, ncol, out, T, O,
                                   (int)K, E, prefetch ? 1 : 0);
    return launch_after_previous(combine_vec_kernel<Tok, Idx, false>, dim3((unsigned)blocks),
                                 dim3(256), 0, stream, ys, sel, p, part, ncol, out, T, O, (int)K,
                                 E, prefetch ? 1 : 0);
  }
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  return launch_after_previous(combine_kernel<Tok, Idx>, dim3((unsigned)blocks), dim3(256), 0,
                               stream, ys, sel, p, part, ncol, out, T, O, (int)K, E);
}

template <typename Tok>
cudaError_t launch_by_index(const Tok* ys, const void* sel, int index_dtype,
                            const float* p, const float* part, int ncol, Tok* out,
                            int64_t T, int64_t E, int64_t O, int64_t K, bool prefetch,
                            cudaStream_t stream) {
  if (index_dtype == kIndexI64)
    return launch_typed(ys, static_cast<const int64_t*>(sel), p, part, ncol, out, T,
                        E, O, K, prefetch, stream);
  return launch_typed(ys, static_cast<const int32_t*>(sel), p, part, ncol, out, T, E,
                      O, K, prefetch, stream);
}

}  // namespace

cudaError_t launch_combine(const void* y_shared, const void* sel,
                           int index_dtype, const float* p, const float* part,
                           int ncol, void* out, int token_dtype, int64_t T,
                           int64_t E, int64_t O, int64_t K, bool after_linear,
                           cudaStream_t stream) {
  if (token_dtype == kTokenBF16)
    return launch_by_index(static_cast<const __nv_bfloat16*>(y_shared), sel,
                           index_dtype, p, part, ncol,
                           static_cast<__nv_bfloat16*>(out), T, E, O, K, after_linear, stream);
  return launch_by_index(static_cast<const float*>(y_shared), sel, index_dtype,
                         p, part, ncol, static_cast<float*>(out), T, E, O, K, after_linear,
                         stream);
}

}  // namespace mxfp4el
