// prepare.cu -- load-time layout of the experts' MXFP4 weights for the
// routed expert linear's kernels ("MoE Expert Kernels: Grouped Prefill and
// Mixed-Quant Compact Experts", section 2, the weight preparation built once
// at load time; the values are those of "MXFP4 Routed Expert Linear", Kimi
// K3, "What is stored in one group").
//
// The prepared copy holds the same bytes as (packed_weights, scale_bytes),
// reordered so that the tensor-core kernel reads one contiguous block per
// 64-wide K chunk of a 128-row tile:
//
//   block (e, mt, kc), at ((e * mtiles + mt) * nk + kc) * kPrepBlockBytes,
//   mtiles = ceil(O / 128), nk = ceil(G / 2), G = I / 32:
//     bytes [32 m, 32 m + 32): row o = 128 mt + m, its packed bytes of groups
//       2kc and 2kc+1, the 16-byte halves swapped when bit 2 of m is set
//       (the 32-byte swizzle: eight consecutive rows then read eight
//       different shared-memory bank groups);
//     bytes kPrepPackedBytes + 2m, + 2m + 1: its scale bytes of those groups.
//   Rows o >= O of the last tile hold zero codes and the scale bytes of row
//   O - 1; with G odd, the missing group 2kc + 1 = G of the last chunk holds
//   zero codes and the scale byte of group G - 1. Both decode to exact zeros.
//
// After the blocks, 256-byte aligned: the f16 row offsets int16 [E][O] and the
// tile modes uint8 [E][mtiles] of the tensor-core kernel's exact f16 operand
// mode, the same values its per-call tile scan computes.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// One CTA per block (kc, mt, e); thread m moves row m.
__global__ void __launch_bounds__(kPrepRows)
prepare_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales, int G,
               int O, int mtiles, unsigned char* __restrict__ out) {
  const int kc = blockIdx.x, mt = blockIdx.y, e = blockIdx.z, m = threadIdx.x;
  const int nk = gridDim.x;
  unsigned char* blk = out + (((size_t)e * mtiles + mt) * nk + kc) * kPrepBlockBytes;
  const int o = mt * kPrepRows + m;
  const size_t row = (size_t)e * O + min(o, O - 1);
  const int g0 = 2 * kc, g1 = 2 * kc + 1;
  uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
  if (o < O) {
    c0 = *reinterpret_cast<const uint4*>(packed + (row * G + g0) * 16);
    if (g1 < G) c1 = *reinterpret_cast<const uint4*>(packed + (row * G + g1) * 16);
  }
  const uint32_t sw = (uint32_t)(m >> 2) & 1u;
  *reinterpret_cast<uint4*>(blk + m * 32 + sw * 16) = c0;
  *reinterpret_cast<uint4*>(blk + m * 32 + (sw ^ 1u) * 16) = c1;
  const uint8_t s0 = scales[row * G + g0];
  const uint8_t s1 = g1 < G ? scales[row * G + g1] : s0;
  blk[kPrepPackedBytes + 2 * m] = s0;
  blk[kPrepPackedBytes + 2 * m + 1] = s1;
}

}  // namespace

size_t prepared_bytes(int64_t E, int64_t I, int64_t O) {
  const int64_t G = I / 32, nk = (G + 1) / 2, mtiles = (O + kPrepRows - 1) / kPrepRows;
  return align256((size_t)E * mtiles * nk * kPrepBlockBytes) +
         align256((size_t)E * O * sizeof(int16_t)) + align256((size_t)E * mtiles);
}

PreparedView prepared_view(const void* base, int64_t E, int64_t I, int64_t O) {
  const int64_t G = I / 32, nk = (G + 1) / 2, mtiles = (O + kPrepRows - 1) / kPrepRows;
  const unsigned char* b = static_cast<const unsigned char*>(base);
  PreparedView v;
  v.blocks = b;
  size_t off = align256((size_t)E * mtiles * nk * kPrepBlockBytes);
  v.row_off = reinterpret_cast<const int16_t*>(b + off);
  off += align256((size_t)E * O * sizeof(int16_t));
  v.tile_mode = b + off;
  return v;
}

cudaError_t launch_prepare(const uint8_t* packed, const uint8_t* scales, int64_t E, int64_t I,
                           int64_t O, void* prepared, cudaStream_t stream) {
  const int64_t G = I / 32, nk = (G + 1) / 2, mtiles = (O + kPrepRows - 1) / kPrepRows;
  if (E <= 0 || O <= 0) return cudaSuccess;
  if (nk > 0x7fffffff || mtiles > 65535 || E > 65535) return cudaErrorInvalidValue;
  // A plain launch: whatever ran before on the stream (a call still reading
  // an earlier copy in this buffer) finishes first.
  prepare_kernel<<<dim3((unsigned)nk, (unsigned)mtiles, (unsigned)E), kPrepRows, 0, stream>>>(
      packed, scales, (int)G, (int)O, (int)mtiles, static_cast<unsigned char*>(prepared));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launch();
  const PreparedView v = prepared_view(prepared, E, I, O);
  uint8_t* tile_mode = const_cast<uint8_t*>(v.tile_mode);
  int16_t* row_off = const_cast<int16_t*>(v.row_off);
  // The f16 operand modes and row offsets; rows too wide for the scan keep
  // every tile in the bf16 mode.
  if (tile_scan_fits(I)) return launch_tile_scan(scales, E, I, O, 0, tile_mode, row_off, stream);
  return cudaMemsetAsync(tile_mode, 0, (size_t)E * mtiles, stream);
}

}  // namespace mxfp4el
