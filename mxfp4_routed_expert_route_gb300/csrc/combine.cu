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
// [0, E) contribute nothing. The kernel is a grid-stride elementwise pass.
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

template <typename Tok, typename Idx>
cudaError_t launch_typed(const Tok* ys, const Idx* sel, const float* p,
                         const float* part, int ncol, Tok* out, int64_t T, int64_t E,
                         int64_t O, int64_t K, cudaStream_t stream) {
  const int64_t n = T * O;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  return launch_after_previous(combine_kernel<Tok, Idx>, dim3((unsigned)blocks), dim3(256), 0,
                               stream, ys, sel, p, part, ncol, out, T, O, (int)K, E);
}

template <typename Tok>
cudaError_t launch_by_index(const Tok* ys, const void* sel, int index_dtype,
                            const float* p, const float* part, int ncol, Tok* out,
                            int64_t T, int64_t E, int64_t O, int64_t K,
                            cudaStream_t stream) {
  if (index_dtype == kIndexI64)
    return launch_typed(ys, static_cast<const int64_t*>(sel), p, part, ncol, out, T,
                        E, O, K, stream);
  return launch_typed(ys, static_cast<const int32_t*>(sel), p, part, ncol, out, T, E,
                      O, K, stream);
}

}  // namespace

cudaError_t launch_combine(const void* y_shared, const void* sel,
                           int index_dtype, const float* p, const float* part,
                           int ncol, void* out, int token_dtype, int64_t T,
                           int64_t E, int64_t O, int64_t K, cudaStream_t stream) {
  if (token_dtype == kTokenBF16)
    return launch_by_index(static_cast<const __nv_bfloat16*>(y_shared), sel,
                           index_dtype, p, part, ncol,
                           static_cast<__nv_bfloat16*>(out), T, E, O, K, stream);
  return launch_by_index(static_cast<const float*>(y_shared), sel, index_dtype,
                         p, part, ncol, static_cast<float*>(out), T, E, O, K, stream);
}

}  // namespace mxfp4el
