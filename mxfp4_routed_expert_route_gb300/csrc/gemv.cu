// gemv.cu -- decode-regime routed expert GEMV.
//
// For every selected expert e and each of its tokens t this computes the
// float32 routed result part[t*K+k, o] = sum_i W_e[o, i] x[t, i] with
// W_e[o, 32g + 2j (+1)] = LUT[low (high) nibble of packed[e,o,g,j]] *
// 2^(scales[e,o,g] - 127) (problem statement "MXFP4 Routed Expert Linear",
// Kimi K3, sections "What is stored in one group" to "Reconstruct the matrix
// in the right orientation").
//
// The work is bound by HBM: every byte of a selected expert is read once.
//
// gemv_stream_kernel (the main kernel): persistent CTAs, one per SM. A work
// unit is (selected expert, tile of 16*RW consecutive output rows); the
// tile's packed bytes, and its scale bytes, are contiguous in memory, so a
// producer warp moves each unit with one or two 1D bulk copies (TMA engine)
// into a ring of shared-memory stages guarded by mbarriers. Each CTA takes a
// contiguous range of units, so it reads one expert's token list once and
// streams consecutive memory. Sixteen consumer warps each own RW rows of the
// tile: lane = one 32-value group, decoded in
// registers by the hardware E2M1 -> f16x2 conversion and multiplied against
// the token, then reduced across lanes with one shuffle reduce-scatter. The
// expert's tokens are taken NT at a time straight from shared memory, so a
// unit's weights are read from HBM once whatever the number of tokens.
//
// Arithmetic. fp32 tokens: products and sums in float32 (f32x2 FMAs).
// bf16 tokens: each token is scaled by a power of two 2^sigma_t chosen so
// that max|x_t| 2^sigma_t lies in [2^8, 2^9) and rounded to f16 (exact for
// bf16 values in f16's normal range); within a group the 32 products form
// two f16x2 chains of 8 (fma.rn.f16x2) that are added in f16, so each half
// sums 16 products with at most 8 roundings; the two halves are widened to
// float32, scaled by the group's exact power of two and accumulated in
// float32. The group error is <= 8 * 2^-11 of the sum of |terms| (plus f16
// subnormal rounding, absolute <= 2^-25 * 2^-sigma_t per token value), and
// |partial| <= 16 * 6 * 2^9 keeps every f16 sum inside f16's range.
//
// gemv_direct_kernel: the same arithmetic in float32 straight from global
// memory (no staging), for rows too wide for a shared-memory stage.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr int kConsumerWarps = 15;
constexpr int kStreamThreads = (kConsumerWarps + 1) * 32;
constexpr int kDirectThreads = 256;
constexpr int kDirectWarps = kDirectThreads / 32;
constexpr size_t kMaxStageBytes = 64 * 1024;
constexpr size_t kSmemBudget = 220 * 1024;
constexpr int kMaxStages = 8;
// Dynamic shared memory: the stage barriers, the scale-factor table, then
// (self-routed mode) the routing area and the stages.
constexpr uint32_t kScaleLutOffset = 2 * kMaxStages * sizeof(uint64_t);
constexpr int kScaleLutEntries = 512;
constexpr uint32_t kScaleLutBytes = kScaleLutEntries * sizeof(float2);
constexpr uint32_t kStreamHeadBytes = kScaleLutOffset + kScaleLutBytes;
static_assert(kStreamHeadBytes % 128 == 0, "the routing area and stages stay 128-byte aligned");

template <int V> struct Log2 { static constexpr int value = 1 + Log2<V / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

// ------------------------------------------------------------ group dots ---
// 16 packed bytes -> 16 f16x2 words: word i holds input positions 2i (low
// half, from the low nibble) and 2i+1 (high half).
__device__ __forceinline__ void decode_group(const uint4& v, uint32_t (&w)[16]) {
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(words[q], h);
#pragma unroll
    for (int b = 0; b < 4; ++b) w[4 * q + b] = h[b];
  }
}

// sum_j w_j x_j over one group: two f16x2 chains of 8 products, added in
// f16, then the two halves widened to float32.
__device__ __forceinline__ float dot_group_f16(const uint32_t (&w)[16], const uint32_t (&x)[16]) {
  uint32_t a0 = hmul2(w[0], x[0]);
  uint32_t a1 = hmul2(w[1], x[1]);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    a0 = hfma2(w[2 * i], x[2 * i], a0);
    a1 = hfma2(w[2 * i + 1], x[2 * i + 1], a1);
  }
  const float2 f = f16x2_to_f32x2(hadd2(a0, a1));
  return f.x + f.y;
}

// sum_j w_j x_j over one group in float32 (exact products).
__device__ __forceinline__ float dot_group_f32(const uint32_t (&w)[16], const float (&x)[32]) {
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 wf = f16x2_to_f32x2(w[i]);
    const float2 xv = make_float2(x[2 * i], x[2 * i + 1]);
    if (i & 1) a1 = ffma2(wf, xv, a1);
    else       a0 = ffma2(wf, xv, a0);
  }
  return (a0.x + a1.x) + (a0.y + a1.y);
}

// Token operand of one group, per token dtype.
template <typename Tok> struct GroupToken;

template <> struct GroupToken<float> {      // fp32 tokens, used as they are
  using Elem = float;
  float v[32];
  __device__ __forceinline__ void load(const float* row, int g) {
    TokenIO<float>::load32(row + (size_t)g * 32, v);
  }
  __device__ __forceinline__ float dot(const uint32_t (&w)[16]) const { return dot_group_f32(w, v); }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
  }
};

template <> struct GroupToken<__half> {     // bf16 tokens, pre-scaled to f16
  using Elem = __half;
  uint32_t v[16];
  __device__ __forceinline__ void load(const __half* row, int g) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = ld_u4(row + (size_t)g * 32 + 8 * q);
      v[4 * q + 0] = u.x; v[4 * q + 1] = u.y; v[4 * q + 2] = u.z; v[4 * q + 3] = u.w;
    }
  }
  // The same values from the bf16 tokens: f16(x * up), up = 2^sigma_t, as
  // the token prep rounds them.
  __device__ __forceinline__ void load_scaled(const __nv_bfloat16* row, int g, float up) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = ld_u4(row + (size_t)g * 32 + 8 * q);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16) * up,
                                            __uint_as_float(w[k] & 0xffff0000u) * up);
        v[4 * q + k] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }
  __device__ __forceinline__ float dot(const uint32_t (&w)[16]) const { return dot_group_f16(w, v); }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0u;
  }
};

// ---------------------------------------------------------- token prep -----
__global__ void __launch_bounds__(256)
prep_tokens_kernel(const __nv_bfloat16* __restrict__ x, __half* __restrict__ x16,
                   int* __restrict__ sigma, int T, int I) {
  pdl_launch_dependents();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t < T) prep_token(x, x16, sigma, t, I, threadIdx.x & 31);
  // Finish only after the bucketer before this kernel has: the GEMV waits
  // on this kernel alone.
  pdl_wait();
}

// ------------------------------------------------------- stream kernel -----
struct StreamArgs {
  const void* x;                 // float (fp32 tokens) or __half (pre-scaled)
  const int* sigma;              // per-token power of two, bf16 tokens only
  const uint8_t* packed;
  const uint8_t* scales;
  const uint8_t* scales_end;     // one past the last scale byte
  RoutePlan plan;
  float* part;                   // [T*K, ncol, O]
  unsigned long long* status;    // device status words (timeouts)
  int G, O, I, K;
  int ncol;                      // group columns: ceil(G / 32)
  int nsub;                      // row subsets: consumer warps per column
  int rows_per_tile;             // nsub * RWS
  int row_tiles;
  int stages;
  uint32_t stage_bytes;          // header + packed part + scale part, 128-aligned
  uint32_t packed_stage_bytes;   // rows_per_tile * G * 16 (scales follow)
  // Self-routed mode (small batches): the CTA derives the routing lists
  // from the ids itself, in shared memory, and scales bf16 tokens on load.
  const void* sel;               // (T, K) expert ids, int32 or int64
  int sel_i64;
  int T, E, P;                   // P = T * K
  int fixed_cost;                // split cost of a unit beyond its tokens
  uint32_t route_bytes;          // bytes of the routing area in shared memory
  // Dynamic tail: the contiguous per-CTA ranges cover static_permille/1000
  // of the cost; the units after them form a pool that CTAs claim one at a
  // time from *pool once their own range is done.
  int static_permille;
  int* pool;                     // claim counter (workspace), reset by CTA 0
  // Stage layout. Plain weights: header at 0, the tile's packed rows (16 G
  // bytes each) at 128, its scale span after them. Prepared weights (prep):
  // one slab per K chunk of rows_per_tile rows x 32 bytes (groups 2kc and
  // 2kc+1 of a row, swapped on rows with bit 2 set) at pk_off = 0, one slab per chunk of 2
  // scale bytes per row at sc_off, the header at hdr_off. Tiles never cross
  // a 128-row block of the layout: each block is cut into tiles_per_block
  // tiles at multiples of rows_per_tile (a multiple of 8), the last one
  // shorter when rows_per_tile does not divide 128.
  int prep;
  int mtiles, nk;                // prepared: 128-row tiles per expert, K chunks
  int tiles_per_block;           // prepared: GEMV tiles per 128-row tile (the last may be short)
  uint32_t hdr_off, pk_off, sc_off;
  uint32_t prow;                 // stage bytes between a group's rows: 16 G, or 32
  uint32_t srow;                 // stage bytes between a scale's rows: G, or 2
  CUtensorMap pmap;              // prepared: packed slabs, box {4 rows_per_tile (8-byte), nk}
  CUtensorMap smap;              // prepared: scale slabs, box {2 rows_per_tile, nk}
};

// Written by the producer into each stage before its copies are issued.
struct StageHeader {
  int e;          // expert id
  int o0;         // first output row of the tile
  int rows;       // rows in the tile
  int scale_off;  // offset of the tile's first scale byte in the stage's
                  // scale area, or -1: read the scales from global memory
  int pad[28];    // keep the payload 128-byte aligned
};
static_assert(sizeof(StageHeader) == 128, "stage header is 128 bytes");

template <int N> struct Pow2Ceil { static constexpr int value = 2 * Pow2Ceil<(N + 1) / 2>::value; };
template <> struct Pow2Ceil<1> { static constexpr int value = 1; };

// ------------------------------------------------- self-routed mode -------
// For small batches each CTA builds, in shared memory, the part of the
// routing that it needs (the bucketer's lists, computed the same way): the
// per-expert counts and offsets, the ascending active list, its own
// cost-balanced unit range, the pair ids of its experts in (token, slot)
// order at their global positions, and the power-of-two scale of each of
// its tokens. This saves the bucketer's launch on the latency-bound path.
constexpr int kSelfMaxPairs = 1024;
constexpr int kSelfMaxExperts = 2048;
constexpr int kSelfMaxTokens = 1024;
static_assert(kSelfMaxExperts < 4096 && kSelfMaxPairs < (1 << 18),
              "the plan scans pairs and active experts packed in one int");
constexpr int kSigmaNeeded = -1000;            // token used by this CTA, scale pending
constexpr int kSelfPrefetchTokens = 64;        // token rows prefetched into L2 at start

struct SelfPlan {
  int* ids;      // [P]     the expert ids, as loaded (-1 for ids outside [0, E))
  int* off;      // [E + 1] segment offsets
  int* run;      // [E]     next free position while placing pairs
  int* active;   // [E]     ascending active experts
  int* list;     // [P]     pair ids of this CTA's experts, at their global positions
  int* sigma;    // [T]     token scale exponents (bf16 tokens)
  int* misc;     // [8]     0: active experts, 1: first unit, 2: end unit, 3: pairs,
                 //         4: first unit of the shared pool
};

__host__ __device__ inline uint32_t self_route_bytes(int E, int P, int T) {
  return (uint32_t)(((size_t)(E + 1) + 2 * (size_t)E + 2 * (size_t)P + (size_t)T + 8) * 4 +
                    127) /
         128 * 128;
}

__device__ __forceinline__ SelfPlan self_plan(unsigned char* area, int E, int P, int T) {
  SelfPlan sp;
  int* w = reinterpret_cast<int*>(area);
  sp.ids = w;
  sp.off = sp.ids + P;
  sp.run = sp.off + (E + 1);
  sp.active = sp.run + E;
  sp.list = sp.active + E;
  sp.sigma = sp.list + P;
  sp.misc = sp.sigma + T;
  return sp;
}

__device__ __forceinline__ long long load_id(const StreamArgs& a, int i) {
  return a.sel_i64 ? static_cast<const long long*>(a.sel)[i]
                   : (long long)static_cast<const int*>(a.sel)[i];
}

// First unit of CTA b of n under the cost-balanced split (unit (u, tile)
// costs fixed + tokens of active expert u); the same integer formula as the
// bucketer's table. Called by a whole warp: each lane tests one active
// expert of a 32-wide chunk (the cost prefix rises with u, so the experts
// that qualify form a prefix of the chunk) instead of one thread's binary
// search over dependent shared-memory loads.
__device__ __forceinline__ int split_begin_warp(const SelfPlan& sp, int na, int pairs, int64_t rt,
                                                int fixed, int64_t b, int64_t n, int lane) {
  if (b >= n) return (int)(na * rt);
  const int64_t C = rt * ((int64_t)fixed * na + pairs);   // cost of all units
  if (C == 0) return 0;
  auto cost_before = [&](int u) { return (int64_t)fixed * u + sp.off[sp.active[u]]; };
  // Largest u with rt * cost_before(u) * n <= b * C (u = 0 always qualifies).
  int u = 0;
  for (int base = 0; base < na; base += 32) {
    const int v = base + lane;
    const bool ok = v < na && rt * cost_before(v) * n <= b * C;
    const unsigned m = __ballot_sync(kFullMask, ok);
    if (m != 0u) u = base + 31 - __clz(m);
    if (m != kFullMask) break;
  }
  const int64_t e = sp.active[u];
  const int64_t cu = fixed + (sp.off[e + 1] - sp.off[e]);
  const int64_t lo_cost = rt * cost_before(u);
  const int64_t tile = (b * C - lo_cost * n + n * cu - 1) / (n * cu);
  return (int)(u * rt + tile);
}

// Barrier of the consumer warps only (the producer does not take part).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// The CTA's routing plan, by the whole block: counts, offsets, the active
// list and this CTA's unit range (what the producer needs).
__device__ void self_route_plan(const StreamArgs& a, const SelfPlan& sp) {
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, P = a.P, T = a.T;
  // The ids first: their loads are in flight while the counters are zeroed.
  constexpr int kIdsPerThread = (kSelfMaxPairs + kStreamThreads - 1) / kStreamThreads;
  long long id[kIdsPerThread];
#pragma unroll
  for (int j = 0; j < kIdsPerThread; ++j) {
    const int i = tid + j * nthr;
    id[j] = i < P ? load_id(a, i) : -1;
  }
  for (int e = tid; e < E; e += nthr) sp.off[e] = 0;
  for (int t = tid; t < T; t += nthr) sp.sigma[t] = 0;
  __syncthreads();
  // Counts (order does not matter here); the ids stay in shared memory.
  int bad = 0;
#pragma unroll
  for (int j = 0; j < kIdsPerThread; ++j) {
    const int i = tid + j * nthr;
    if (i >= P) continue;
    const long long e = id[j];
    const bool valid = e >= 0 && e < E;
    sp.ids[i] = valid ? (int)e : -1;
    if (valid) atomicAdd(&sp.off[e], 1);
    else ++bad;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) bad += __shfl_xor_sync(kFullMask, bad, o);
  if (lane == 0 && bad > 0 && blockIdx.x == 0)     // every CTA sees them; one counts
    atomicAdd(&a.status[kStatusBadPairs], (unsigned long long)bad);
  __syncthreads();
  // Offsets and the ascending active list, by warp 0 alone (lane l owns
  // experts [l*per, (l+1)*per)): one warp scan of pairs (from bit 12 up, at
  // most kSelfMaxPairs) and active experts (below, at most kSelfMaxExperts
  // < 4096) packed in one int.
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (sp.off[e] << 12) | (sp.off[e] > 0 ? 1 : 0);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(kFullMask, incl, 31);
    int off = (incl - mine) >> 12, act = (incl - mine) & 0xfff;
    for (int e = e0; e < e1; ++e) {
      const int c = sp.off[e];
      sp.off[e] = off;
      if (c > 0) sp.active[act++] = e;
      off += c;
    }
    if (lane == 0) {
      sp.off[E] = total >> 12;
      sp.misc[0] = total & 0xfff;
      sp.misc[3] = total >> 12;
    }
  }
  __syncthreads();
  // This CTA's static range and the start of the shared pool, one boundary
  // per warp: boundary b of n sits at b * static_permille / (1000 n) of the
  // cost.
  if (warp < 3) {
    const int64_t b = warp == 0 ? blockIdx.x : warp == 1 ? blockIdx.x + 1 : gridDim.x;
    const int v = split_begin_warp(sp, sp.misc[0], sp.misc[3], a.row_tiles, a.fixed_cost,
                                   b * a.static_permille, (int64_t)gridDim.x * 1000, lane);
    if (lane == 0) sp.misc[warp == 2 ? 4 : 1 + warp] = v;
  }
  __syncthreads();
}

// The rest, by the consumer warps while the producer starts its copies:
// the pair ids of the experts this CTA may meet (its own range and the
// shared pool) and the scales of their tokens.
__device__ void self_route_lists(const StreamArgs& a, const SelfPlan& sp, bool bf16_tokens) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int P = a.P, T = a.T;
  const int num_units = sp.misc[0] * a.row_tiles;
  const int ubeg = min(sp.misc[1], num_units), uend = min(sp.misc[2], num_units);
  const int pool_begin = min(sp.misc[4], num_units);
  if (ubeg >= uend && pool_begin >= num_units) return;
  // Expert ids e_lo .. e_hi (active slots ubeg/rt .. (uend-1)/rt) and, for
  // the pool, p_lo .. the last active expert (p_lo >= e_hi: the static
  // ranges lie before the pool); an empty range is 0 .. -1.
  int e_lo = 0, e_hi = -1, p_lo = 0, p_hi = -1;
  if (ubeg < uend) {
    e_lo = sp.active[ubeg / a.row_tiles];
    e_hi = sp.active[(uend - 1) / a.row_tiles];
  }
  if (pool_begin < num_units) {
    p_lo = sp.active[pool_begin / a.row_tiles];
    p_hi = sp.active[sp.misc[0] - 1];
  }
  // Their pair ids, placed in (token, slot) order by one warp.
  if (warp == 0) {
    for (int e = e_lo + lane; e <= e_hi; e += 32) sp.run[e] = sp.off[e];
    for (int e = max(p_lo, e_hi + 1) + lane; e <= p_hi; e += 32) sp.run[e] = sp.off[e];
    __syncwarp();
    const unsigned below = (1u << lane) - 1u;
    for (int base = 0; base < P; base += 32) {
      const int i = base + lane;
      const int e = i < P ? sp.ids[i] : -1;
      const bool mine = (e >= e_lo && e <= e_hi) || (e >= p_lo && e <= p_hi);
      const unsigned peers = __match_any_sync(kFullMask, mine ? e : -1);
      if (mine) {
        sp.list[sp.run[e] + __popc(peers & below)] = i;
        sp.sigma[i / a.K] = kSigmaNeeded;
      }
      __syncwarp();
      if (mine && (peers & below) == 0) sp.run[e] += __popc(peers);
      __syncwarp();
    }
  }
  consumers_sync();
  // Scale exponents of this CTA's bf16 tokens (as the token prep computes them).
  if (bf16_tokens) {
    for (int t = warp; t < T; t += kConsumerWarps) {
      if (sp.sigma[t] != kSigmaNeeded) continue;
      const uint4* row =
          reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)t * a.I);
      uint32_t m = 0;
      for (int i = lane; i < a.I / 8; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          m = max(m, (w[k] << 16) & 0x7fffffffu);
          m = max(m, w[k] & 0x7fff0000u);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(kFullMask, m, o));
      const int ex = (int)(m >> 23);
      int sg = 0;
      if (m != 0 && ex < 255) sg = min(126, 135 - ex);
      __syncwarp();
      if (lane == 0) sp.sigma[t] = sg;
    }
  }
  consumers_sync();
}

// One pass of one consumer warp over its RWS rows of a staged tile, for NTA
// tokens: lane = group g of the warp's column; each (row, token) gets one
// group partial per lane, summed across the warp and stored as the column's
// partial result. kScalesStaged: the tile's scale bytes are in shared memory
// (else they are read from global memory).
// The group partial v times 2^(s - 127 - sigma_t), exactly: the weight
// scale and the token's own power of two (bf16 tokens are pre-scaled by
// 2^sigma_t into f16; sigma_t = 0 for fp32 tokens) in one factor, so that no
// intermediate leaves float32's range when the result does not. The factor
// is a pair (f1, f2), applied as (v * f1) * f2, from a table in shared memory
// indexed by s + 126 - sigma_t (sigma_t is in [-119, 126], so 0..500);
// entry i stands for 2^e with e = i - 253:
//   -149 <= e <= 127: (2^e, 1)          one multiply by a float32 (2^e is
//                                       subnormal below -126): one rounding;
//   e > 127:          (2^127, 2^(e-127)) v * 2^127 is exact or overflows
//                                       only when v * 2^e does;
//   -165 <= e < -149: (2^-100, 2^(e+100)) for f16-token partials, which are
//                                       0 or at least 2^-24 in magnitude, so
//                                       v * 2^-100 is exact;
//   e < -165:         (0, 1)            |v| < 2^16 there, so v * 2^e rounds
//                                       to zero.
// fp32 tokens only reach -127 <= e <= 128.
__device__ __forceinline__ const float2* scale_lut() {
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  return reinterpret_cast<const float2*>(dyn_smem + kScaleLutOffset);
}
__device__ __forceinline__ float pow2f(int e) {          // exact 2^e, -149 <= e <= 127
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}
__device__ __forceinline__ void fill_scale_lut(float2* lut) {
  for (int i = threadIdx.x; i < kScaleLutEntries; i += blockDim.x) {
    const int e = i - 253;
    float2 f;
    if (e > 254) f = make_float2(pow2f(127), __uint_as_float(0x7f800000u));   // never indexed
    else if (e > 127) f = make_float2(pow2f(127), pow2f(e - 127));
    else if (e >= -149) f = make_float2(pow2f(e), 1.f);
    else if (e >= -165) f = make_float2(pow2f(-100), pow2f(e + 100));
    else f = make_float2(0.f, 1.f);
    lut[i] = f;
  }
}
// Table offset of a token's factors.
__device__ __forceinline__ int scale_offset(int sigma) { return 126 - sigma; }
__device__ __forceinline__ float apply_scale(float v, uint32_t s, const float2* lut_t) {
  const float2 f = lut_t[s];
  return (v * f.x) * f.y;
}

// kFull: all RWS rows of the warp lie inside the tile (no per-row test).
template <typename Elem, int RWS, int NTA, bool kScalesStaged, bool kFull>
__device__ __forceinline__ void stream_pass(const StreamArgs& a, const GroupToken<Elem> (&xt)[NTA],
                                            const int (&pair)[NTA], const int (&soff)[NTA],
                                            uint32_t sp_lane,
                                            uint32_t ss_lane, const uint8_t* gs_lane, int o0,
                                            int rows, int rbase, int c, int lane,
                                            uint32_t flip) {
  constexpr int V = Pow2Ceil<RWS * NTA>::value;
  constexpr int L = Log2<V>::value;
  const int G = a.G, O = a.O;
  const uint32_t prow = a.prow;                  // stage bytes between rows
  const float2* lut = scale_lut();
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  // Every lane runs the rows: lanes past the last group read group G-1's
  // weights against zeroed token values (see load_pass), so their partials
  // are zero without a branch or a select.
  uint32_t pa = sp_lane, sa = ss_lane;
  const uint8_t* ga = gs_lane;
#pragma unroll
  for (int r = 0; r < RWS; ++r) {
    if (kFull || rbase + r < rows) {
      uint32_t w[16];
      // Prepared weights: rows 4..7 of an 8-row group hold the row's 16-byte
      // halves in the other order (flip = +-16; 0 on the plain layout).
      decode_group(lds128(RWS == 8 && (r & 4) ? pa + flip : pa), w);
      const uint32_t sb = kScalesStaged ? lds_u8(sa) : (uint32_t)__ldg(ga);
#pragma unroll
      for (int j = 0; j < NTA; ++j) acc[r * NTA + j] = apply_scale(xt[j].dot(w), sb, lut + soff[j]);
    }
    pa += prow;
    sa += a.srow;
    if (!kScalesStaged) ga += G;
  }
  const float total = warp_reduce_scatter<V>(acc, lane);
  if ((lane & ((1 << (5 - L)) - 1)) == 0) {
    const int idx = (lane >> (5 - L)) & (V - 1);
    if (idx < RWS * NTA) {
      const int r = idx / NTA, j = idx - (idx / NTA) * NTA;
      if (kFull || rbase + r < rows) {
        int pj = pair[0];
#pragma unroll
        for (int q = 1; q < NTA; ++q) pj = (j == q) ? pair[q] : pj;
        a.part[((size_t)pj * a.ncol + c) * O + o0 + rbase + r] = total;
      }
    }
  }
}

// Both scale sources for one pass (the choice is uniform per tile); the
// global address of the lane's scale bytes is formed only when the tile's
// scales were not staged (expert e, group gc).
template <typename Elem, int RWS, int NTA>
__device__ __forceinline__ void stream_pass_any(const StreamArgs& a,
                                                const GroupToken<Elem> (&xt)[NTA],
                                                const int (&pair)[NTA],
                                                const int (&soff)[NTA], uint32_t sp_lane,
                                                uint32_t ss_lane, int e, int gc, bool staged,
                                                int o0, int rows, int rbase, int c, int lane,
                                                uint32_t flip) {
  if (staged && rbase + RWS <= rows) {
    stream_pass<Elem, RWS, NTA, true, true>(a, xt, pair, soff, sp_lane, ss_lane, nullptr, o0,
                                            rows, rbase, c, lane, flip);
  } else if (staged) {
    stream_pass<Elem, RWS, NTA, true, false>(a, xt, pair, soff, sp_lane, ss_lane, nullptr, o0,
                                             rows, rbase, c, lane, flip);
  } else {
    const uint8_t* gs_lane = a.scales + ((size_t)e * a.O + o0 + rbase) * a.G + gc;
    stream_pass<Elem, RWS, NTA, false, false>(a, xt, pair, soff, sp_lane, ss_lane, gs_lane,
                                              o0, rows, rbase, c, lane, flip);
  }
}

// Token operands (this lane's group) and pair ids of the pass starting at
// position `base` of an expert's segment [base, seg_end), and each token's
// offset into the scale-factor table (from its power of two; 0 for fp32
// tokens). Lanes past the last group (g >= G) get zeros.
template <typename Elem, int NT, bool kSelf>
__device__ __forceinline__ void load_pass(const StreamArgs& a, const SelfPlan& sp,
                                          GroupToken<Elem> (&xt)[NT], int (&pair)[NT],
                                          int (&soff)[NT], int base, int seg_end, int g) {
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int pos = base + min(j, seg_end - base - 1);
    pair[j] = kSelf ? sp.list[pos] : a.plan.pair_list[pos];
    const int t = pair[j] / a.K;
    if constexpr (kSelf && sizeof(Elem) == 2) {
      // bf16 tokens scaled on load by this CTA's own power of two.
      const int sg = sp.sigma[t];
      if (g < a.G)
        xt[j].load_scaled(static_cast<const __nv_bfloat16*>(a.x) + (size_t)t * a.I, g,
                          __uint_as_float((uint32_t)(sg + 127) << 23));
      else
        xt[j].zero();
      soff[j] = scale_offset(sg);
    } else {
      if (g < a.G) xt[j].load(static_cast<const Elem*>(a.x) + (size_t)t * a.I, g);
      else xt[j].zero();
      soff[j] = scale_offset(a.sigma != nullptr ? a.sigma[t] : 0);
    }
  }
}

template <typename Elem, int RWS, int NT, bool kSelf>
__global__ void __launch_bounds__(kStreamThreads, 1)
gemv_stream_kernel(const __grid_constant__ StreamArgs a) {
  static_assert(NT == 1 || NT == 2, "one or two tokens per pass");
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  unsigned char* route_area = smem + kStreamHeadBytes;
  unsigned char* stage_base = route_area + (kSelf ? a.route_bytes : 0u);
  // Prepared weights: stages start 1024-byte aligned (the launch adds the
  // slack), so every slab starts on a 128-byte line.
  if (a.prep) stage_base += (1024u - (smem_addr(stage_base) & 1023u)) & 1023u;
  const SelfPlan rp = self_plan(route_area, a.E, a.P, a.T);

  // A lane-0 shuffle makes the warp index provably warp-uniform, so that the
  // compiler keeps the warp's role and row arithmetic in uniform registers
  // (wide decode 286 -> 282 us).
  const int warp = __shfl_sync(kFullMask, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
  fill_scale_lut(reinterpret_cast<float2*>(smem + kScaleLutOffset));   // read after a barrier
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  // Self-routed: this is the call's first kernel, so it reads the ids and
  // tokens only after whatever ran before it on the stream has finished.
  // Otherwise: the bucketer's lists and the prepared tokens are ready.
  pdl_wait();
  // Only now may the combine start: it reads the call's other inputs before
  // waiting for this kernel, so everything before this kernel must be done.
  pdl_launch_dependents();
  // The pool counter starts at zero for this launch. A CTA that claims
  // before this reset gets a stale value: one past the pool ends its claims,
  // one inside the pool repeats a unit (the same values written twice). CTA
  // 0 claims only after its reset, so it keeps claiming until every pool
  // unit has been taken.
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.pool != nullptr) atomicExch(a.pool, 0);
  if constexpr (kSelf) {
    // Few tokens: start bringing their rows into L2 now; the CTA reads them
    // (scale, then operands) only after its routing plan is ready.
    if (warp == kConsumerWarps && a.T <= kSelfPrefetchTokens)
      for (int t = lane; t < a.T; t += 32)
        prefetch_l2(static_cast<const unsigned char*>(a.x) +
                        (size_t)t * a.I * (sizeof(Elem) == 2 ? 2 : 4),
                    (uint32_t)a.I * (sizeof(Elem) == 2 ? 2u : 4u));
    self_route_plan(a, rp);                // ends with a block barrier
    if (warp != kConsumerWarps) self_route_lists(a, rp, sizeof(Elem) == 2);
  } else {
    __syncthreads();
  }

  // Each CTA takes one contiguous range of units, so consecutive units are
  // consecutive row tiles of the same expert (and of consecutive memory).
  // The bucketer balances the ranges by cost (an expert's units cost more
  // the more tokens it has); without its table the ranges are equal.
  const int num_units = (kSelf ? rp.misc[0] : a.plan.meta[kMetaNumActive]) * a.row_tiles;
  int ubeg, uend, pool_begin = num_units;
  if (kSelf) {
    ubeg = min(rp.misc[1], num_units);
    uend = min(rp.misc[2], num_units);
    pool_begin = min(rp.misc[4], num_units);
  } else if (a.plan.unit_begin != nullptr) {
    ubeg = min(a.plan.unit_begin[blockIdx.x], num_units);
    uend = min(a.plan.unit_begin[blockIdx.x + 1], num_units);
    pool_begin = min(a.plan.unit_begin[gridDim.x], num_units);
  } else {
    const int per_cta = num_units / (int)gridDim.x;
    const int extra = num_units - per_cta * (int)gridDim.x;
    ubeg = (int)blockIdx.x * per_cta + min((int)blockIdx.x, extra);
    uend = ubeg + per_cta + ((int)blockIdx.x < extra ? 1 : 0);
  }
  const int G = a.G, O = a.O;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t policy = l2_evict_first_policy();
    int issued = 0;
    bool ok = true;
    int e = -1, cached_u = -1;
    // Units of the CTA's own range, then units claimed from the pool, then
    // an end marker: a stage whose header names no expert.
    int unit = ubeg;
    int st = 0;
    uint32_t round = 0;
    for (;; ++issued) {
      if (unit >= uend) {
        const int claim = pool_begin < num_units ? atomicAdd(a.pool, 1) : -1;
        unit = claim >= 0 && claim < num_units - pool_begin ? pool_begin + claim : -1;
      }
      if (unit < 0) {
        if (!mbar_wait(&empty[st], (round & 1u) ^ 1u)) { ok = false; break; }
        reinterpret_cast<StageHeader*>(stage_base + (size_t)st * a.stage_bytes + a.hdr_off)->e = -1;
        mbar_arrive(&full[st]);
        ++issued;
        break;
      }
      const int u = unit / a.row_tiles, tile = unit - u * a.row_tiles;
      if (u != cached_u) { e = kSelf ? rp.active[u] : a.plan.active[u]; cached_u = u; }
      int o0 = tile * a.rows_per_tile;
      int rows = min(a.rows_per_tile, O - o0);
      if (a.prep) {
        const int blk128 = tile / a.tiles_per_block, sub = tile - blk128 * a.tiles_per_block;
        o0 = blk128 * kPrepRows + sub * a.rows_per_tile;
        rows = min(min(a.rows_per_tile, kPrepRows - sub * a.rows_per_tile), O - o0);
      }
      if (rows <= 0) {              // a tile past the last row (prepared, O % 128 != 0)
        ++unit;
        --issued;
        continue;
      }
      if (a.prep) {
        // The tile's slabs: packed rows o0 % 128 .. of every K chunk of
        // 128-row tile o0 / 128 (one contiguous run of 32 bytes per row in
        // each block, the layout's half swap kept), and their scale bytes;
        // rows past the block read zeros.
        if (!mbar_wait(&empty[st], (round & 1u) ^ 1u)) { ok = false; break; }
        unsigned char* dst = stage_base + (size_t)st * a.stage_bytes;
        StageHeader* h = reinterpret_cast<StageHeader*>(dst + a.hdr_off);
        h->e = e;
        h->o0 = o0;
        h->rows = rows;
        h->scale_off = 0;
        const int blk = (e * a.mtiles + o0 / kPrepRows) * a.nk;
        const int r0 = o0 % kPrepRows;
        const uint32_t pbytes = (uint32_t)a.nk * (uint32_t)a.rows_per_tile * 32u;
        const uint32_t sbytes = (uint32_t)a.nk * (uint32_t)a.rows_per_tile * 2u;
        mbar_arrive_expect_tx(&full[st], pbytes + sbytes);     // releases the header
        tma_load_2d(dst + a.pk_off, &a.pmap, 4 * r0, blk, &full[st], policy);
        tma_load_2d(dst + a.sc_off, &a.smap, 2 * r0, blk, &full[st], policy);
      } else {
      const size_t row0 = (size_t)e * O + o0;
      const uint32_t pbytes = (uint32_t)rows * G * 16;
      // The tile's scale bytes: copy the 16-byte-aligned span that holds
      // them, unless that span would pass the end of the scales buffer.
      const uintptr_t s_lo = reinterpret_cast<uintptr_t>(a.scales + row0 * G);
      const uintptr_t s_hi = s_lo + (uintptr_t)rows * G;
      const uintptr_t c_lo = s_lo & ~(uintptr_t)15;
      const uintptr_t c_hi = (s_hi + 15) & ~(uintptr_t)15;
      const bool scale_copy = c_hi <= reinterpret_cast<uintptr_t>(a.scales_end);
      const uint32_t sbytes = scale_copy ? (uint32_t)(c_hi - c_lo) : 0u;
      if (!mbar_wait(&empty[st], (round & 1u) ^ 1u)) { ok = false; break; }
      unsigned char* dst = stage_base + (size_t)st * a.stage_bytes;
      StageHeader* h = reinterpret_cast<StageHeader*>(dst);
      h->e = e;
      h->o0 = o0;
      h->rows = rows;
      h->scale_off = scale_copy ? (int)(s_lo - c_lo) : -1;
      mbar_arrive_expect_tx(&full[st], pbytes + sbytes);     // releases the header
      bulk_copy_g2s(dst + sizeof(StageHeader), a.packed + row0 * G * 16, pbytes, &full[st],
                    policy);
      if (sbytes)
        bulk_copy_g2s(dst + sizeof(StageHeader) + a.packed_stage_bytes,
                      reinterpret_cast<const void*>(c_lo), sbytes, &full[st], policy);
      }
      ++unit;                       // past uend (pool units lie after every range): claim
      // Slow start: the first stage goes out alone and lands before the
      // rest of the ring is requested. With every CTA's whole ring
      // requested at once the first stages landed only after most of those
      // bytes (6 us after the request); the consumers, the bottleneck here,
      // now start about 1 us sooner (decode, measured).
      if (issued == 0 && !mbar_wait(&full[0], 0u)) { ok = false; break; }
      if (++st == a.stages) {
        st = 0;
        ++round;
      }
    }
    if (!ok) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
    // Do not leave copies in flight: wait (bounded) for the last round of
    // every stage this thread issued.
    for (int k = max(0, issued - a.stages); k < issued; ++k) {
      const int st = k % a.stages;
      if (!mbar_wait(&full[st], (uint32_t)(k / a.stages) & 1u)) {
        atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
        break;
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumers
  // Warp (c, s): group column c (groups 32c .. 32c+31), rows s*RWS .. +RWS-1.
  const bool working = warp < a.ncol * a.nsub;
  const int c = warp % a.ncol, sub = warp / a.ncol;
  const int g = c * 32 + lane;
  const int gc = min(g, a.G - 1);     // lanes past the last group shadow group G-1
  const int rbase = sub * RWS;
  int cached_e = -1, seg_beg = 0, seg_end = 0;
  // Token operands of the expert's first pass, kept across its tiles.
  GroupToken<Elem> x0[NT];
  int pair0[NT];
  int soff0[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) { pair0[j] = 0; soff0[j] = scale_offset(0); }

  // Self-routed: the first unit's expert is known from the plan, so its
  // tokens load while the first stage is still on its way.
  if (kSelf && working && ubeg < uend) {
    cached_e = rp.active[ubeg / a.row_tiles];
    seg_beg = rp.off[cached_e];
    seg_end = rp.off[cached_e + 1];
    load_pass<Elem, NT, kSelf>(a, rp, x0, pair0, soff0, seg_beg, seg_end, g);
  }
  // Stages in the producer's order until its end marker.
  int st = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait_suspend(&full[st], phase)) {
      if (lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
      return;
    }
    const unsigned char* hp = stage_base + (size_t)st * a.stage_bytes;
    // The header in one 16-byte load: expert, first row, rows, scale offset.
    const int4 hv = *reinterpret_cast<const int4*>(hp + a.hdr_off);
    const int e = hv.x;
    if (e < 0) break;
    const int o0 = hv.y, rows = hv.z, scale_off = hv.w;
    const unsigned char* sp = hp + a.pk_off;

    if (working && rbase < rows) {
      if (e != cached_e) {                    // new expert: its first pass
        cached_e = e;
        seg_beg = kSelf ? rp.off[e] : a.plan.offsets[e];
        seg_end = kSelf ? rp.off[e + 1] : a.plan.offsets[e + 1];
        load_pass<Elem, NT, kSelf>(a, rp, x0, pair0, soff0, seg_beg, seg_end, g);
      }
      // This lane's group in row rbase of the tile: packed bytes and scale
      // (prepared: in the slab of chunk gc / 2, half gc % 2 of the row, the
      // halves swapped on rows with bit 2 set; a tile starts at a multiple
      // of 8 rows of its 128-row block).
      const uint32_t rpt = (uint32_t)a.rows_per_tile;
      const uint32_t half = ((uint32_t)gc ^ ((uint32_t)rbase >> 2)) & 1u;
      const uint32_t flip = a.prep ? (half ? 0u - 16u : 16u) : 0u;
      const uint32_t sp_lane =
          a.prep ? smem_addr(sp) + ((uint32_t)gc >> 1) * rpt * 32u + (uint32_t)rbase * 32u +
                       half * 16u
                 : smem_addr(sp) + ((uint32_t)rbase * (uint32_t)G + (uint32_t)gc) * 16u;
      const uint32_t ss_lane =
          a.prep ? smem_addr(hp + a.sc_off) + ((uint32_t)gc >> 1) * rpt * 2u +
                       (uint32_t)rbase * 2u + ((uint32_t)gc & 1u)
                 : smem_addr(sp) + a.packed_stage_bytes + (uint32_t)(scale_off + rbase * G + gc);
      const bool staged = scale_off >= 0;
      for (int base = seg_beg;;) {
        if (seg_end - base >= NT) {
          stream_pass_any<Elem, RWS, NT>(a, x0, pair0, soff0, sp_lane, ss_lane, e, gc, staged,
                                         o0, rows, rbase, c, lane, flip);
        } else {                              // one token left (NT == 2)
          stream_pass_any<Elem, RWS, 1>(
              a, reinterpret_cast<const GroupToken<Elem>(&)[1]>(x0[0]),
              reinterpret_cast<const int(&)[1]>(pair0[0]),
              reinterpret_cast<const int(&)[1]>(soff0[0]), sp_lane, ss_lane, e, gc, staged,
              o0, rows, rbase, c, lane, flip);
        }
        base += NT;
        if (base >= seg_end) break;
        // More tokens: the cache now holds a later pass, so reload the first
        // one at the next tile.
        load_pass<Elem, NT, kSelf>(a, rp, x0, pair0, soff0, base, seg_end, g);
        cached_e = -1;
      }
    }
    fence_proxy_async_smem();           // stage read: the refill's bulk copies may land
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (++st == a.stages) {
      st = 0;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------- direct kernel -----
template <typename Tok, int R, int NT>
__global__ void __launch_bounds__(kDirectThreads, 2)
gemv_direct_kernel(const Tok* __restrict__ x, const uint8_t* __restrict__ packed,
                   const uint8_t* __restrict__ scales, RoutePlan plan,
                   float* __restrict__ part, int G, int O, int I, int K, int row_tiles) {
  constexpr int V = R * NT;
  constexpr int L = Log2<V>::value;
  pdl_wait();
  const int u = blockIdx.x / row_tiles;
  const int tile = blockIdx.x - u * row_tiles;
  if (u >= plan.meta[kMetaNumActive]) return;
  const int e = plan.active[u];
  const int seg_beg = plan.offsets[e], seg_end = plan.offsets[e + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int o0 = (tile * kDirectWarps + warp) * R;
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
    for (int j = 0; j < NT; ++j)
      xrow[j] = x + (size_t)(plan.pair_list[base + min(j, nt - 1)] / K) * I;
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    for (int g = lane; g < G; g += 32) {
      uint32_t w[R][16];
      E8M0 sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        decode_group(ld_stream_u4(wrow[r] + (size_t)g * 16), w[r]);
        sc[r] = e8m0(srow[r][g]);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if (j < nt) {
          float xf[32];
          TokenIO<Tok>::load32(xrow[j] + (size_t)g * 32, xf);
#pragma unroll
          for (int r = 0; r < R; ++r)
            acc[r * NT + j] = fmaf(dot_group_f32(w[r], xf) * sc[r].pre, sc[r].factor,
                                   acc[r * NT + j]);
        }
      }
    }
    const float total = warp_reduce_scatter<V>(acc, lane);
    if ((lane & ((1 << (5 - L)) - 1)) == 0) {
      const int idx = (lane >> (5 - L)) & (V - 1);
      const int r = idx / NT, j = idx - (idx / NT) * NT;
      if (j < nt && o0 + r < O)
        part[(size_t)plan.pair_list[base + j] * O + o0 + r] = total;
    }
  }
}

// ------------------------------------------------------------- launch ------
int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 152;
  }
  return cached[dev];
}

int64_t stream_grid(int64_t bound_units) { return std::min<int64_t>(num_sms(), bound_units); }

template <typename Elem, int RWS, bool kSelf>
cudaError_t launch_stream(StreamArgs a, size_t smem, int64_t bound_units, cudaStream_t stream) {
  // Two tokens per pass for f16 operands; fp32 operands take twice the
  // registers, so one.
  constexpr int NT = sizeof(Elem) == 2 ? 2 : 1;
  auto kern = gemv_stream_kernel<Elem, RWS, NT, kSelf>;
  static std::mutex mu;
  static size_t opted[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && opted[dev] < smem) {
      cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
      if (err != cudaSuccess) return err;
      opted[dev] = smem;
    }
  }
  const int64_t grid = stream_grid(bound_units);
  if (grid <= 0) return cudaSuccess;
  return launch_after_previous(kern, dim3((unsigned)grid), dim3(kStreamThreads), smem, stream, a);
}

template <typename Tok>
cudaError_t launch_direct(const Tok* x, const uint8_t* packed, const uint8_t* scales,
                          const RoutePlan& plan, float* part, int64_t T, int64_t E,
                          int64_t I, int64_t O, int64_t K, cudaStream_t stream) {
  constexpr int R = 4, NT = 4;
  const int64_t rows_per_cta = (int64_t)kDirectWarps * R;
  const int64_t row_tiles = (O + rows_per_cta - 1) / rows_per_cta;
  const int64_t blocks = std::min<int64_t>(E, T * K) * row_tiles;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_after_previous(gemv_direct_kernel<Tok, R, NT>, dim3((unsigned)blocks),
                               dim3(kDirectThreads), 0, stream, x, packed, scales, plan, part,
                               (int)(I / 32), (int)O, (int)I, (int)K, (int)row_tiles);
}

// Shape of the staged GEMV for a row width of G groups: group columns,
// consumer warps per column, rows per warp. rws == 0 when the rows are too
// wide to stage (the direct kernel runs instead).
struct StreamShape {
  int ncol = 0, nsub = 0, rws = 0;
};

size_t stage_bytes_for(size_t rows, int64_t G) {
  return 128 + rows * G * 16 + ((rows * G + 15) / 16) * 16 + 16;
}

// A stage of prepared weights: nk slabs of rows x 32 packed bytes, nk slabs
// of rows x 2 scale bytes, the header; 1024-byte multiples.
uint32_t prep_stage_bytes(size_t rows, int64_t nk, uint32_t* sc_off, uint32_t* hdr_off) {
  const size_t sc = (size_t)nk * rows * 32;
  const size_t hdr = (sc + (size_t)nk * rows * 2 + 127) / 128 * 128;
  if (sc_off) *sc_off = (uint32_t)sc;
  if (hdr_off) *hdr_off = (uint32_t)hdr;
  return (uint32_t)((hdr + sizeof(StageHeader) + 1023) / 1024 * 1024);
}

// Prepared weights: a tile's rows must start at a multiple of 8 inside a
// 128-row block of the layout (the consumers' undoing of the half swap and
// the scale slab's 16-byte units), so its height is a multiple of 8, and at
// most 64 (a box row of the packed copy holds at most 256 8-byte elements).
// The copies' boxes take at most 256 K chunks.
StreamShape stream_shape(int64_t G, bool prep = false) {
  StreamShape sh;
  const int64_t ncol = (G + 31) / 32;
  if (ncol > kConsumerWarps) return sh;
  sh.ncol = (int)ncol;
  sh.nsub = kConsumerWarps / sh.ncol;
  if (prep) {
    const int64_t nk = (G + 1) / 2;
    if (nk > 256) return sh;
    // All consumer warps if their tile height is a multiple of 8 (then the
    // 128-row blocks are cut into tiles at multiples of it), else the
    // largest power of two of warps per column.
    for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) {
        int n = 1;
        while (2 * n <= sh.nsub) n *= 2;
        sh.nsub = n;
      }
      for (int rws = 8; rws >= 1; rws /= 2) {
        const size_t rows = (size_t)sh.nsub * rws;
        if (rows % 8 == 0 && rows <= 64 &&
            prep_stage_bytes(rows, nk, nullptr, nullptr) <= kMaxStageBytes) {
          sh.rws = rws;
          return sh;
        }
      }
    }
    return sh;
  }
  for (int rws = 8; rws >= 1; rws /= 2) {
    if (stage_bytes_for((size_t)sh.nsub * rws, G) <= kMaxStageBytes) {
      sh.rws = rws;
      return sh;
    }
  }
  return sh;
}

// Units of the staged kernel: active experts (at most min(E, T*K)) times
// row tiles; the tile height follows from the stream shape.
int64_t stream_row_tiles(const StreamShape& sh, int64_t O, bool prep = false) {
  const int64_t rows = (int64_t)sh.nsub * sh.rws;
  if (prep) return (O + kPrepRows - 1) / kPrepRows * ((kPrepRows + rows - 1) / rows);
  return (O + rows - 1) / rows;
}

}  // namespace

// Cost of a unit beyond its tokens, in token passes. Measured on GB300: a
// unit's time grows with its expert's tokens; with the pool below, weighing
// tokens alone balances best.
#ifndef MXFP4EL_GEMV_FIXED_COST
#define MXFP4EL_GEMV_FIXED_COST 0
#endif
// Share of the cost, in thousandths, that the per-CTA ranges cover; the
// remaining units are claimed dynamically, so CTAs that stream faster or
// drew cheaper units than the cost model says take more of them. Measured
// on GB300: 900 takes the wide decode batch from 349 to 325 us and leaves
// the 8-token batch unchanged; 850 and 800 are slower on both.
#ifndef MXFP4EL_GEMV_STATIC_PERMILLE
#define MXFP4EL_GEMV_STATIC_PERMILLE 900
#endif

bool gemv_self_route(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, bool prep) {
  // Test knob: MXFP4EL_ROUTE=bucketer keeps the separate bucketer launch.
  if (const char* env = std::getenv("MXFP4EL_ROUTE"))
    if (std::strcmp(env, "bucketer") == 0) return false;
  const StreamShape sh = stream_shape(I / 32, prep);
  const int64_t P = T * K;
  if (sh.rws == 0 || P <= 0 || O <= 0 || P > kSelfMaxPairs || E > kSelfMaxExperts ||
      T > kSelfMaxTokens)
    return false;
  // The in-kernel split multiplies costs by the row tiles, 1000 and the
  // grid in int64.
  const int64_t max_cost = std::min<int64_t>(E, P) * MXFP4EL_GEMV_FIXED_COST + P;
  return stream_row_tiles(sh, O, prep) * max_cost <= ((int64_t)1 << 40);
}

UnitSplit gemv_unit_split(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, bool prep) {
  UnitSplit sp{0, 0, 0, 1000};
  const StreamShape sh = stream_shape(I / 32, prep);
  if (sh.rws == 0 || T * K == 0 || O == 0) return sp;
  const int64_t rt = stream_row_tiles(sh, O, prep);
  const int64_t bound_units = std::min<int64_t>(E, T * K) * rt;
  const int64_t ctas = stream_grid(bound_units);
  const int64_t fixed = MXFP4EL_GEMV_FIXED_COST;
  // The bucketer sums costs in int32 and multiplies them by rt, ctas and
  // 1000 in int64; beyond that the kernel keeps its even split.
  const int64_t max_cost = std::min<int64_t>(E, T * K) * fixed + T * K;
  if (ctas <= 0 || ctas > kMaxSplitCtas || bound_units > 0x7fffffff ||
      max_cost >= ((int64_t)1 << 31) || rt * max_cost > ((int64_t)1 << 40))
    return sp;
  sp.ctas = (int)ctas;
  sp.row_tiles = (int)rt;
  sp.fixed_cost = (int)fixed;
  sp.static_permille = MXFP4EL_GEMV_STATIC_PERMILLE;
  return sp;
}

int gemv_partial_columns(int64_t I) {
  const StreamShape sh = stream_shape(I / 32);
  return sh.rws > 0 ? sh.ncol : 1;
}

bool gemv_uses_stream(int64_t I, bool prep) { return stream_shape(I / 32, prep).rws > 0; }

cudaError_t launch_prep_tokens(const void* x, __half* x16, int* sigma, int64_t T, int64_t I,
                               cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_after_previous(prep_tokens_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0,
                               stream, static_cast<const __nv_bfloat16*>(x), x16, sigma, (int)T,
                               (int)I);
}

cudaError_t launch_gemv(const void* x, int token_dtype, const __half* x16, const int* sigma,
                        const void* sel, int index_dtype, const uint8_t* packed,
                        const uint8_t* scales, const RoutePlan& plan, float* part,
                        unsigned long long* status, int64_t T, int64_t E, int64_t I, int64_t O,
                        int64_t K, cudaStream_t stream, const PreparedView* prep) {
  const int64_t G = I / 32;
  const StreamShape sh = stream_shape(G, prep != nullptr);
  if (sh.rws == 0 && prep != nullptr) return cudaErrorInvalidValue;
  if (sh.rws == 0) {
    if (token_dtype == kTokenBF16)
      return launch_direct(static_cast<const __nv_bfloat16*>(x), packed, scales, plan, part,
                           T, E, I, O, K, stream);
    return launch_direct(static_cast<const float*>(x), packed, scales, plan, part, T, E, I,
                         O, K, stream);
  }
  const bool self = gemv_self_route(T, E, I, O, K, prep != nullptr);
  StreamArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = token_dtype == kTokenBF16 && !self ? static_cast<const void*>(x16) : x;
  a.sigma = token_dtype == kTokenBF16 && !self ? sigma : nullptr;
  a.sel = sel;
  a.sel_i64 = index_dtype == kIndexI64 ? 1 : 0;
  a.T = (int)T;
  a.E = (int)E;
  a.P = (int)(T * K);
  a.fixed_cost = MXFP4EL_GEMV_FIXED_COST;
  a.static_permille = MXFP4EL_GEMV_STATIC_PERMILLE;
  a.pool = plan.meta + kMetaPoolCounter;
  a.route_bytes = self ? self_route_bytes(a.E, a.P, a.T) : 0u;
  a.packed = packed;
  a.scales = scales;
  a.scales_end = scales + (size_t)E * O * G;
  a.plan = plan;
  a.part = part;
  a.status = status;
  a.G = (int)G;
  a.O = (int)O;
  a.I = (int)I;
  a.K = (int)K;
  a.ncol = sh.ncol;
  a.nsub = sh.nsub;
  a.rows_per_tile = sh.nsub * sh.rws;
  a.row_tiles = (int)stream_row_tiles(sh, O, prep != nullptr);
  // The bucketer wrote plan.unit_begin only if it was asked for a split.
  if (gemv_unit_split(T, E, I, O, K, prep != nullptr).ctas == 0) a.plan.unit_begin = nullptr;
  size_t slack = 0;
  if (prep != nullptr) {
    a.prep = 1;
    a.packed = nullptr;
    a.scales = nullptr;
    a.scales_end = nullptr;
    a.mtiles = (int)((O + kPrepRows - 1) / kPrepRows);
    a.nk = (int)((G + 1) / 2);
    a.tiles_per_block = (kPrepRows + a.rows_per_tile - 1) / a.rows_per_tile;
    a.pk_off = 0;
    a.stage_bytes = prep_stage_bytes(a.rows_per_tile, a.nk, &a.sc_off, &a.hdr_off);
    a.prow = 32;
    a.srow = 2;
    a.packed_stage_bytes = 0;
    slack = 1024;                 // stages start 1024-byte aligned
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t blocks = (cuuint64_t)E * (cuuint64_t)a.mtiles * (cuuint64_t)a.nk;
    // Packed bytes as 8-byte elements, so that a tile's rows of one block
    // (32 * rows contiguous bytes) are one box row: long contiguous reads.
    const cuuint64_t pdims[2] = {kPrepPackedBytes / 8, blocks};
    const cuuint64_t pstrides[1] = {kPrepBlockBytes};
    const cuuint32_t pbox[2] = {(cuuint32_t)(4 * a.rows_per_tile), (cuuint32_t)a.nk};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&a.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<unsigned char*>(prep->blocks),
            pdims, pstrides, pbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const cuuint64_t sdims[2] = {2 * kPrepRows, blocks};
    const cuuint64_t sstrides[1] = {kPrepBlockBytes};
    const cuuint32_t sbox[2] = {(cuuint32_t)(2 * a.rows_per_tile), (cuuint32_t)a.nk};
    if (enc(&a.smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<unsigned char*>(prep->blocks + kPrepPackedBytes), sdims, sstrides, sbox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    a.prep = 0;
    a.packed_stage_bytes = (uint32_t)((size_t)a.rows_per_tile * G * 16);
    a.stage_bytes = (uint32_t)((stage_bytes_for(a.rows_per_tile, G) + 127) / 128 * 128);
    a.hdr_off = 0;
    a.pk_off = sizeof(StageHeader);
    a.sc_off = sizeof(StageHeader) + a.packed_stage_bytes;
    a.prow = (uint32_t)G * 16u;
    a.srow = (uint32_t)G;
  }
  a.stages = (int)std::min<size_t>(
      kMaxStages, (kSmemBudget - kStreamHeadBytes - a.route_bytes - slack) / a.stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem =
      kStreamHeadBytes + a.route_bytes + slack + (size_t)a.stages * a.stage_bytes;
  const int64_t bound_units = std::min<int64_t>(E, T * K) * a.row_tiles;
  if (bound_units > 0x7fffffff) return cudaErrorInvalidConfiguration;
#define MXFP4EL_STREAM_CASES_SELF(ELEM, SELF)                                    \
  switch (sh.rws) {                                                               \
    case 8: return launch_stream<ELEM, 8, SELF>(a, smem, bound_units, stream);    \
    case 4: return launch_stream<ELEM, 4, SELF>(a, smem, bound_units, stream);    \
    case 2: return launch_stream<ELEM, 2, SELF>(a, smem, bound_units, stream);    \
    default: return launch_stream<ELEM, 1, SELF>(a, smem, bound_units, stream);   \
  }
#define MXFP4EL_STREAM_CASES(ELEM)                                     \
  if (self) { MXFP4EL_STREAM_CASES_SELF(ELEM, true) }                   \
  MXFP4EL_STREAM_CASES_SELF(ELEM, false)
  if (token_dtype == kTokenBF16) { MXFP4EL_STREAM_CASES(__half) }
  MXFP4EL_STREAM_CASES(float)
#undef MXFP4EL_STREAM_CASES
#undef MXFP4EL_STREAM_CASES_SELF
}

}  // namespace mxfp4el
