// gemm_tc.cu -- prefill-regime routed expert grouped GEMM on the 5th-gen
// tensor cores (tcgen05, TMEM, TMA).
//
// For every selected expert e and each block of its tokens it computes
// part[t*K+k, o] = sum_i W_e[o, i] x[t, i] for all output rows o, with W_e
// decoded from MXFP4 as in the problem statement ("MXFP4 Routed Expert
// Linear", Kimi K3): W_e[o, 32g+2j (+1)] = LUT[low (high) nibble of
// packed[e,o,g,j]] * 2^(scales[e,o,g] - 127).
//
// Shape ("swap AB"): M = 128 weight rows per tile, N = the tokens of one
// block (16..192, a multiple of 16), K = I in chunks of 64 (two groups).
//   * A (weights) is decoded exactly and written straight into tensor
//     memory: row m in TMEM lane m, two K elements per 32-bit column.
//   * B (tokens) is a copy of the token rows grouped by expert, written by
//     group_tokens_kernel in f16 scaled per row by a power of two; TMA loads
//     each 64-wide K chunk with the 128-byte swizzle that the K-major
//     shared-memory descriptor describes.
//   * tcgen05.mma kind::f16, fp32 accumulator in TMEM.
//
// Two exact operand modes, chosen per tile:
//   * f16: tokens pre-scaled per token by 2^sigma_t (max |x_t| 2^sigma_t in
//     [2^14, 2^15)), weights decoded by the hardware E2M1 -> f16x2
//     conversion and one f16x2 multiply by 2^(s - 127 - r_m), where r_m is a
//     per-row offset chosen so that every scaled weight of the row is a normal
//     f16 number; the epilogue multiplies by 2^(r_m - sigma_t). Possible when
//     every row's scale bytes span at most 26 binades. The mode of each tile
//     and the row offsets come from tile_scan_kernel, run before this kernel.
//   * bf16: weights decoded to their exact bf16 bit patterns (byte-permute
//     tables), any scale byte; the dequantizers convert the chunk's f16 token
//     rows to bf16 in shared memory (exact: they came from bf16 values) and
//     the epilogue multiplies by 2^-sigma_t.
// Products are exact in both modes and accumulate in fp32, so the modes give
// the same result up to the accumulation order inside the MMA.
//
// Warp roles in a CTA of 24 warps (one CTA per SM, persistent over units
// (expert, token block, 128-row tile), which CTAs take from a global counter
// as they go):
//   warp 0      producer of scales and packed weights (elected lane) and TMEM
//               allocation; takes each next unit from the counter and hands
//               its index to the other roles through a shared-memory ring
//   warp 1      MMA issuer (the whole warp waits for each chunk's readiness,
//               one elected lane issues)
//   warp 2      per-expert lists at start
//   warp 3      producer of token tiles (elected lane)
//   warps 4-19  dequantize, in four teams of 4 warps: team t takes chunks t,
//               t+4, ...; thread m decodes both groups of the chunk for
//               weight row m into TMEM A buffer (chunk mod 4), once the
//               chunk's token rows have landed and the buffer is free
//   warps 20-23 epilogue: TMEM -> registers (mode scaling) -> shared memory
//               (transposed) -> float32 partial results
// Every wait is bounded; a role whose wait gives up records it, stops, and
// the CTA still waits (bounded) for its own copies and MMAs before freeing
// TMEM.
//
// Gate/up tiles (gemm_tc_kernel<true, false>, the SwiGLU expert's stacked
// gate/up projection, 2F rows with the gate rows first): a tile's 128 rows
// are 64 gate rows f0.. and the matching 64 up rows F + f0.. (two 64-row TMA
// boxes into one stage, two scale spans), so the epilogue holds g and u of
// the same (pair, f) and writes h = silu(g) * u in bf16 instead of partial
// results, by pair or in the lists' grouped order; the down projection can
// then run as a second instance on the same lists (its own unit counter),
// its token rows being the grouped rows of h.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr int kTcThreads = 768;
constexpr int kBM = 128;                    // weight rows per tile
constexpr int kBK = 64;                     // K elements per chunk (two groups)
constexpr int kNMax = 192;                  // token columns per block (TMEM accumulator width)
constexpr int kABufs = 4;                   // TMEM A buffers: chunk c uses buffer c % kABufs
constexpr int kTeams = 4;                   // dequantizer teams: chunk c goes to team c % kTeams
constexpr int kStagesAMax = 16;             // packed-weight ring (from HBM)
constexpr int kStagesBMax = 8;              // token stages, as shared memory allows
constexpr uint32_t kStageA = kBM * 32;      // packed bytes of a chunk, 32 B per row
// A chunk block of the prepared layout: the chunk's packed bytes as the plain
// layout's stage holds them, then two scale bytes per row (rows in order).
constexpr uint32_t kStagePrep = kPrepBlockBytes;
static_assert(kPrepRows == kBM && kPrepPackedBytes == kStageA, "prepared blocks are tiles");
static_assert(kStageA % 1024 == 0, "stages keep 1024-byte alignment");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = 0;               // two accumulators of kNMax columns
constexpr uint32_t kACol = 2 * kNMax;       // kABufs A buffers of 32 columns
static_assert(kACol + kABufs * 32 <= kTmemCols, "TMEM budget");
// A chunk's A buffer is rewritten kABufs chunks later, once its MMAs are done;
// the MMAs of the kABufs - 1 chunks between cover the dequantizer's wake-up,
// TMEM stores and signal. (Measured: 192-column accumulators and 4 buffers
// beat 160 columns and 6 buffers, 525 against 535 us at the prefill shape.)
constexpr int kMaxExpertsTc = 512;          // per-expert lists kept in shared memory
constexpr uint32_t kEpiStage = 16 * 32 * 4; // epilogue staging per warp: 16 columns x 32 rows
constexpr int kUnitRing = 4;                // unit indices handed from producer A
constexpr int kListWarp = 2, kProdBWarp = 3;
constexpr int kNumLoads = kNMax / 16;       // token-box heights: 16, 32, ..., kNMax rows
__host__ __device__ constexpr int load_rows(int l) { return 16 * (l + 1); }
constexpr int kDequantWarp0 = 4, kDequantWarps = 16, kTeamWarps = 4, kEpiWarp0 = 20;
// Readers of the unit ring, one arrival each: the producer B warp, the MMA
// warp, the dequantizer warps and the epilogue warps.
constexpr int kUnitReaders = 2 + kDequantWarps + (kTcThreads / 32 - kEpiWarp0);
static_assert(kDequantWarps == kTeams * kTeamWarps, "four teams of four warps");
// The widest span of scale bytes within one row that f16 operands hold
// exactly: LUT values 0.5..6 times 2^d are normal f16 numbers for
// -13 <= d <= 13.
constexpr int kF16Span = 26;

struct TcArgs {
  RoutePlan plan;
  const uint8_t* scales;
  const uint8_t* scales_end;
  float* part;                   // [T*K, O]
  unsigned long long* status;
  const int* sigma;              // per grouped row: the power of two of its f16 copy
  int G, O, K;
  int mtiles;                    // ceil(O / 128) (or ceil(F / 64) for gate/up tiles)
  int stages_a;                  // packed-weight ring depth
  int stages_b;                  // token ring depth (4 .. kStagesBMax)
  uint32_t stage_a;              // bytes per packed-weight stage (kStageA, or kStagePrep)
  const unsigned char* prep;     // prepared chunk blocks [E][mtiles][G/2], or null
  int nmax;                      // token columns per block (<= kNMax)
  uint32_t stage_b;              // bytes per token stage: nmax rows x 128 B
  uint32_t scale_cap;            // bytes per scale buffer
  int b_f16;                      // the grouped rows are f16 copies scaled by 2^sigma
                                 // (else plain bf16 rows: every tile takes the bf16 mode)
  int f16_tiles;                  // tiles may take the f16 mode (b_f16, unless a test
                                 // keeps every tile in bf16)
  const uint8_t* tile_mode;      // [E][mtiles]: 1 = the tile's rows fit f16 operands
  const int16_t* row_off;        // [E*O]: row offset r of every weight row (f16 mode)
  // Gate/up tiles of the SwiGLU expert (F > 0; the matrix has 2F rows, gate
  // rows first): tile rows 0..63 are gate rows f0.., rows 64..127 the
  // matching up rows F + f0..; the epilogue writes h = silu(gate) * up in
  // bf16 and the pairs' expert ids instead of the partial results.
  int F;
  __nv_bfloat16* h;              // (P, F), row = pair (or position in the lists: h_grouped)
  int32_t* sel2;                 // (P): expert of each pair (zeroed by the token prep), or null
  int h_grouped;
  int counter_word;              // plan.meta word this kernel takes its units from
};

struct TcMaps {
  CUtensorMap a;                 // packed weights as uint8 [E*O, G*16], box {32, 128}, 32B swizzle
  CUtensorMap a_half;            // packed weights, box {32, 64} (gate/up tiles)
  CUtensorMap b[kNumLoads];      // grouped token rows [P, I], box {64, rows}, 128B swizzle
};

struct __align__(16) TcShared {
  uint64_t full_a[kStagesAMax], empty_a[kStagesAMax];
  // Chunk c uses token stage c % SB and TMEM A buffer c % kABufs.
  uint64_t b_full[kStagesBMax];  // the chunk's token rows have landed
  uint64_t done[kStagesBMax];    // the chunk's MMAs finished: its stage and A buffer free
  uint64_t d_full[2], d_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t drain;
  uint64_t u_full[kUnitRing], u_empty[kUnitRing];
  int unit_ring[kUnitRing];      // unit indices in the order this CTA takes them; -1 ends
  // Per A buffer: completes once the team's kTeamWarps warps have stored the
  // chunk's A columns and seen its token rows land (and, for bf16 tiles on
  // f16 token rows, converted them). One wait per chunk for the MMA warp,
  // which suspends in the barrier: polling a counter instead kept 32 lanes
  // spinning beside the dequantizer and epilogue warps of its sub-partition
  // and measured 6 to 8 % slower.
  uint64_t a_full[kABufs];
  uint32_t tmem_base;
  int scale_off[2];              // per scale buffer: offset of the tile's first byte, or -1
  int scale_off_up[2];           // per scale buffer: offset of the up rows' first byte
  int num_units;
  int num_active;
  // Per active expert u: id, first position in the grouped list, tokens,
  // and the prefix of token blocks (unit_prefix[num_active] = all blocks).
  int ex_id[kMaxExpertsTc];
  int ex_beg[kMaxExpertsTc];
  int ex_cnt[kMaxExpertsTc];
  int unit_prefix[kMaxExpertsTc + 1];
  uint64_t epi_bar;              // the four epilogue warps (gate/up tiles)
};

// Position in a ring of n slots: slot index and the parity of its use.
struct RingPos {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// One unit of work, derived identically by every role from its index.
struct Unit {
  int e;          // expert id
  int m0;         // first weight row
  int rows;       // weight rows in the tile (<= 128)
  int tok0;       // first position of the block in the grouped token list
  int ntok;       // tokens in the block
  int nmma;       // MMA N: ntok rounded up to 16
  int load;       // token box: load_rows(load) >= nmma
  int mt;         // row tile index
  int nblk;       // the expert's token blocks: its tiles are read once per block
};

template <bool kSplit>
__device__ __forceinline__ Unit unit_at(const TcArgs& a, const TcShared& sh, int idx) {
  // Binary search the expert whose block range holds idx / mtiles.
  const int blk = idx / a.mtiles;
  const int mt = idx - blk * a.mtiles;
  int lo = 0, hi = sh.num_active;         // unit_prefix[u] <= blk < unit_prefix[u + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.unit_prefix[mid] <= blk) lo = mid;
    else hi = mid;
  }
  const int u = lo;
  const int j = blk - sh.unit_prefix[u];
  const int nblk = sh.unit_prefix[u + 1] - sh.unit_prefix[u];
  Unit w;
  w.e = sh.ex_id[u];
  const int beg = sh.ex_beg[u], cnt = sh.ex_cnt[u];
  // Equal blocks, each a multiple of 16 tokens except the last.
  const int bsz = (((cnt + nblk - 1) / nblk) + 15) / 16 * 16;
  w.tok0 = beg + j * bsz;
  w.ntok = min(bsz, cnt - j * bsz);
  w.nmma = (w.ntok + 15) / 16 * 16;
  w.load = w.nmma / 16 - 1;
  // Gate/up tiles: m0 is the first gate row f0, rows the valid rows of each half.
  constexpr int tm = kSplit ? kBM / 2 : kBM;
  w.mt = mt;
  w.nblk = nblk;
  w.m0 = mt * tm;
  w.rows = min(tm, (kSplit ? a.F : a.O) - w.m0);
  return w;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B both f16
// or both bf16, both K-major, shape M x N.
__device__ __forceinline__ uint32_t mma_idesc(int m, int n, bool f16) {
  const uint32_t ab = f16 ? 0u : 1u;     // operand format: 0 f16, 1 bf16
  return (1u << 4)                       // D format: fp32
         | (ab << 7)                     // A format
         | (ab << 10)                    // B format
         | ((uint32_t)(n >> 3) << 17)    // N / 8
         | ((uint32_t)(m >> 4) << 24);   // M / 16
}

// Shared-memory descriptor of a K-major tile with the 128-byte swizzle:
// 128-byte rows, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu)    // start address
         | ((uint64_t)1 << 16)                // leading byte offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows
         | ((uint64_t)1 << 46)                // descriptor version
         | ((uint64_t)2 << 61);               // layout: 128-byte swizzle
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The bf16 bit patterns of the eight magnitudes LUT[j] * 2^(s - 127),
// j = 0..7 (0, 0.5, 1, 1.5, 2, 3, 4, 6), as byte tables for prmt: h0/h1 hold
// the high bytes of j = 0..3 / 4..7, l0/l1 the low bytes.
struct MagnitudeTable {
  uint32_t h0, h1, l0, l1;
};

__device__ __forceinline__ MagnitudeTable magnitude_table(uint32_t s) {
  uint32_t v01, v23, v45, v67;   // (v_j | v_{j+1} << 16)
  if (s - 2u <= 250u) {
    // 2 <= s <= 252: every nonzero magnitude times 2^(s - 127) is a normal
    // bf16 with exponent field s - 1, s, s, s + 1, s + 1, s + 2, s + 2 and
    // mantissa 0 or 0x40 (the factor 1.5).
    const uint32_t t = s * 0x00800080u;            // s << 7 in both halves
    v01 = (s - 1u) << 23;                          // 0 | 0.5
    v23 = t + 0x00400000u;                         // 1 | 1.5
    v45 = t + 0x00C00080u;                         // 2 | 3
    v67 = t + 0x01400100u;                         // 4 | 6
  } else {
    // Subnormal or overflowing results: the exact float32 product (the two
    // factors of e8m0_split are finite for every byte), rounded to bf16.
    const float2 f = e8m0_split(s);
    auto bits = [&](float m) {
      return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((m * f.x) * f.y));
    };
    v01 = bits(0.5f) << 16;
    v23 = bits(1.0f) | (bits(1.5f) << 16);
    v45 = bits(2.0f) | (bits(3.0f) << 16);
    v67 = bits(4.0f) | (bits(6.0f) << 16);
  }
  return {prmt(v01, v23, 0x7531u), prmt(v45, v67, 0x7531u), prmt(v01, v23, 0x6420u),
          prmt(v45, v67, 0x6420u)};
}

// Eight E2M1 codes (one packed word, low nibble first) -> four bf16x2 words,
// w[i] = (value of code 2i, value of code 2i+1). The low three bits of each
// code index the tables; prmt's sign-replicate selectors turn the code's
// sign bit into a byte of all ones, whose top bit becomes the bf16 sign.
__device__ __forceinline__ void decode_word(uint32_t q, const MagnitudeTable& t, uint32_t* w) {
  const uint32_t sel_lo = q & 0x77777777u, sel_hi = sel_lo >> 16;
  const uint32_t y = q << 4;     // byte k of y: sign of code 2k in bit 7; of q: code 2k+1
  const uint32_t h03 = prmt(t.h0, t.h1, sel_lo) | (prmt(y, q, 0xD9C8u) & 0x80808080u);
  const uint32_t h47 = prmt(t.h0, t.h1, sel_hi) | (prmt(y, q, 0xFBEAu) & 0x80808080u);
  const uint32_t l03 = prmt(t.l0, t.l1, sel_lo), l47 = prmt(t.l0, t.l1, sel_hi);
  w[0] = prmt(l03, h03, 0x5140u);
  w[1] = prmt(l03, h03, 0x7362u);
  w[2] = prmt(l47, h47, 0x5140u);
  w[3] = prmt(l47, h47, 0x7362u);
}

// 16 packed bytes (32 codes) of one group and its scale byte -> 16 bf16x2
// words, exactly LUT[code] * 2^(s - 127) wherever that is a bf16 number.
__device__ __forceinline__ void dequant_group_bf16(const uint4& q, uint32_t s, uint32_t (&w)[16]) {
  const MagnitudeTable t = magnitude_table(s);
  decode_word(q.x, t, w);
  decode_word(q.y, t, w + 4);
  decode_word(q.z, t, w + 8);
  decode_word(q.w, t, w + 12);
}

// The same group as 16 f16x2 words LUT[code] * 2^(s - 127 - r): the hardware
// conversion gives LUT[code] in f16 (exact), one f16x2 multiply applies the
// power of two. Exact when -13 <= s - 127 - r <= 13 (then every nonzero
// product lies in [2^-14, 49152], the normal f16 range).
__device__ __forceinline__ void dequant_group_f16(const uint4& q, uint32_t s, int r,
                                                  uint32_t (&w)[16]) {
  const uint32_t f = (uint32_t)((int)s - 112 - r) * 0x04000400u;   // f16x2 2^(s-127-r)
  const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(qq[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[4 * i + j] = hmul2(h[j], f);
  }
}

// The tile's operand mode (1: f16) and, for weight row `row` of expert e,
// its offset r.
__device__ __forceinline__ bool tile_f16(const TcArgs& a, const Unit& w) {
  return a.f16_tiles && a.tile_mode[(size_t)w.e * a.mtiles + w.mt] != 0;
}

// A 16-byte global store with an L2 eviction policy.
__device__ __forceinline__ void st_f4_policy(float* p, const float4& v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

// v * 2^e for any integer e, exact unless the result itself leaves the
// float32 range: one multiply by a normal power of two when |e| allows it,
// else several.
__device__ __forceinline__ float scale_pow2(float v, int e) {
  if (e >= -126 && e <= 127) return v * __uint_as_float((uint32_t)(e + 127) << 23);
  while (e > 127) {
    v *= __uint_as_float(254u << 23);     // 2^127
    e -= 127;
  }
  while (e < -126) {
    v *= __uint_as_float(1u << 23);       // 2^-126
    e += 126;
  }
  return v * __uint_as_float((uint32_t)(e + 127) << 23);
}

// One lane of a fully converged warp (elect.sync; the elected lane may
// differ from call to call).
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " .reg .b32 r;\n"
      " elect.sync r|p, 0xffffffff;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(e));
  return e != 0;
}

// The dequantizer's chunk loop for one tile whose chunks have global indices
// base .. base+nk-1: thread m of team t decodes groups 2kc and 2kc+1 of row m
// into A buffer (base + kc) % kABufs for each of the team's chunks kc (those
// with base + kc = t mod kTeams; `next` is the team's next global chunk).
// Chunk c's packed bytes are in weight stage c % stages_a with the 32-byte
// swizzle: the two 16-byte halves of row m are exchanged when bit 2 of m is
// set, so eight consecutive rows read eight different bank groups. Scale
// bytes: kPrep, the two after the packed bytes of the stage (row m at byte
// kStageA + 2m); else scale(g), the row's scale byte of group g. f16 selects
// the f16 decode with row offset r; convert: the chunk's token rows are f16
// and this tile runs on bf16 operands. Returns false if a wait gave up.
template <bool kPrep, typename ScaleFn>
__device__ __forceinline__ bool dequant_tile(TcShared& sh, const unsigned char* ring_a,
                                             uint32_t stage_a, int stages_a,
                                             unsigned char* ring_b, uint32_t stage_b, int SB,
                                             uint32_t tmem, uint32_t lane_base, int m, int lane,
                                             int tid, int base, int nk, int nmma, int& next,
                                             ScaleFn scale, bool f16, int r, bool convert) {
  const uint32_t sw = (uint32_t)(m >> 2) & 1u;
  const uint32_t off0 = (uint32_t)m * 32u + sw * 16u, off1 = (uint32_t)m * 32u + (sw ^ 1u) * 16u;
  const uint32_t a_cols = tmem + lane_base + kACol;
  // The wait that frees this chunk's A buffer and token stage (see below).
  const int back = min(SB, kABufs);
  for (; next < base + nk; next += kTeams) {
    const int kc = next - base;
    const int sa = next % stages_a;
    if (!mbar_wait_warp(&sh.full_a[sa], (uint32_t)(next / stages_a) & 1u)) return false;
    const unsigned char* stage = ring_a + (size_t)sa * stage_a;
    const uint4 pk0 = *reinterpret_cast<const uint4*>(stage + off0);
    const uint4 pk1 = *reinterpret_cast<const uint4*>(stage + off1);
    uint32_t s0, s1;
    if constexpr (kPrep) {
      const uint32_t s01 = *reinterpret_cast<const uint16_t*>(stage + kStageA + 2 * m);
      s0 = s01 & 0xffu;
      s1 = s01 >> 8;
    } else {
      s0 = scale(2 * kc);
      s1 = scale(2 * kc + 1);
    }
    fence_proxy_async_smem();                             // before the refill's copy lands
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty_a[sa]);         // packed bytes consumed
    uint32_t v0[16], v1[16];
    if (f16) {
      dequant_group_f16(pk0, s0, r, v0);
      dequant_group_f16(pk1, s1, r, v1);
    } else {
      dequant_group_bf16(pk0, s0, v0);
      dequant_group_bf16(pk1, s1, v1);
    }
    // Wait for the MMAs of chunk pc = next - min(SB, kABufs). In-order MMA
    // completion makes that cover what this chunk needs before its A columns
    // may be written: A buffer next % kABufs was last used by chunk
    // next - kABufs <= pc; chunk next - SB <= pc, which used this chunk's
    // token stage, had its token rows landed, so the stage's barrier is now
    // on this chunk's phase (a parity wait cannot tell that phase from an
    // unfinished earlier one); and the barrier of pc's stage cannot have
    // moved two phases past pc (its next use, pc + SB >= next, needs this
    // chunk). The MMAs of the chunks in between cover the rest of this path.
    // Then this chunk's token rows must have landed before the team reports
    // it ready. bf16 tiles on f16 token rows: convert them in place, each of
    // the team's 128 threads a share of the 16-byte pieces (f16 -> bf16 is
    // exact for these values, which came from bf16), and make the writes
    // visible to the tensor cores' reads.
    if (next >= back) {
      const int pc = next - back;
      if (!mbar_wait_warp(&sh.done[pc % SB], (uint32_t)(pc / SB) & 1u)) return false;
    }
    const int st = next % SB;
    if (!mbar_wait_warp(&sh.b_full[st], (uint32_t)(next / SB) & 1u)) return false;
    if (convert) {
      uint4* sb_base = reinterpret_cast<uint4*>(ring_b + (size_t)st * stage_b);
      for (int i = tid; i < nmma * 8; i += kTeamWarps * 32) {
        uint4 v = sb_base[i];
        uint32_t* wv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = f16x2_to_f32x2(wv[k]);
          const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
          wv[k] = *reinterpret_cast<const uint32_t*>(&b);
        }
        sb_base[i] = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    const uint32_t buf = (uint32_t)(next % kABufs);
    const uint32_t a_col = a_cols + buf * 32;
    tc_fence_after_sync();
    tmem_st16(a_col, v0);
    tmem_st16(a_col + 16, v1);
    tmem_wait_st();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.a_full[buf]);
  }
  return true;
}

// The next unit index from the ring. kWarp: called by a whole warp, whose
// lane 0 arrives once all lanes have read it; else by one thread. Returns
// false if the wait gave up; *idx < 0 means no more units.
template <bool kWarp>
__device__ __forceinline__ bool pop_unit(TcShared& sh, RingPos& pu, int lane, int* idx) {
  if (kWarp ? !mbar_wait_warp(&sh.u_full[pu.idx], pu.phase)
            : !mbar_wait(&sh.u_full[pu.idx], pu.phase))
    return false;
  *idx = sh.unit_ring[pu.idx];
  if (kWarp) __syncwarp();
  if (lane == 0) mbar_arrive(&sh.u_empty[pu.idx]);
  pu.next(kUnitRing);
  return true;
}

// Barrier of the four epilogue warps, on an mbarrier of four arrivals so
// that the wait is bounded like every other; false if it gave up.
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& phase, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool done = mbar_wait_warp(bar, phase);
  phase ^= 1u;
  return done;
}

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Epilogue of a gate/up tile: 16 token columns at a time, each epilogue warp
// moves its 32 accumulator rows into shared memory (column-major, all four
// warps' rows side by side), scaled back from the f16 operands' powers of
// two in f16 mode; then thread (cq, rp) forms h = silu(gate) * up for gate
// rows 2rp, 2rp+1 of the tile (their up rows sit 64 rows further, two warps
// on) and token columns 4cq..4cq+3, in float32, and stores each pair of rows
// as one bf16x2. The tile of the first rows of a token block also writes its
// pairs' expert for the down projection. Returns false if a wait gave up.
__device__ bool swiglu_epilogue(const TcArgs& a, const Unit& w, uint32_t d_cols,
                                uint32_t lane_base, float* epi_all, int q, int lane,
                                uint64_t* bar, uint32_t& phase, int roff) {
  float* mine = epi_all + q * (kEpiStage / 4);
  const int et = 32 * q + lane;
  const int rp = et & 31, cq = et >> 5;
  const int r0 = 2 * rp;
  const float* gsrc = epi_all + (r0 >> 5) * (kEpiStage / 4) + (r0 & 31);
  const float* usrc = gsrc + 2 * (kEpiStage / 4);
  const bool row_ok = r0 < w.rows;             // rows is even: r0 + 1 too
  for (int c0 = 0; c0 < w.nmma; c0 += 16) {
    // sigma of the grouped rows of these 16 columns: one load per lane, then broadcast.
    int my_sig = 0;
    if (a.b_f16 && lane < 16 && c0 + lane < w.ntok) my_sig = a.sigma[w.tok0 + c0 + lane];
    uint32_t v[16];
    __syncwarp();
    tmem_ld16(d_cols + lane_base + (uint32_t)c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int sg = __shfl_sync(kFullMask, my_sig, i);
      const float x = __uint_as_float(v[i]);
      mine[i * 32 + lane] = a.b_f16 ? scale_pow2(x, roff - sg) : x;
    }
    if (!epi_sync(bar, phase, lane)) return false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 4 * cq + j;
      if (row_ok && c0 + c < w.ntok) {
        const int pos = w.tok0 + c0 + c;
        const int row = a.h_grouped ? pos : a.plan.pair_list[pos];
        const float h0 = silu_times(gsrc[c * 32], usrc[c * 32]);
        const float h1 = silu_times(gsrc[c * 32 + 1], usrc[c * 32 + 1]);
        *reinterpret_cast<__nv_bfloat162*>(a.h + (size_t)row * a.F + w.m0 + r0) =
            __floats2bfloat162_rn(h0, h1);
      }
    }
    if (!epi_sync(bar, phase, lane)) return false;
  }
  if (w.m0 == 0 && a.sel2 != nullptr)
    for (int c = et; c < w.ntok; c += 128) a.sel2[a.plan.pair_list[w.tok0 + c]] = w.e;
  return true;
}

// kSplit: gate/up tiles of the SwiGLU expert (see TcArgs::F). kPrep: the
// weights come as prepared chunk blocks (TcArgs::prep), one bulk copy per
// chunk with the chunk's scale bytes inside, instead of tiled loads of the
// packed rows and a copy of each tile's scale bytes.
template <bool kSplit, bool kPrep>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  static_assert(!(kSplit && kPrep), "gate/up tiles read the plain layout");
  const int SB = a.stages_b;     // token ring depth, kTeams .. kStagesBMax (checked by the host)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Token stages need 1024-byte alignment (128-byte swizzle atoms).
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* ring_b = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* ring_a = ring_b + (size_t)SB * a.stage_b;
  unsigned char* scale_buf = ring_a + (size_t)a.stages_a * a.stage_a;
  TcShared& sh = *reinterpret_cast<TcShared*>(scale_buf + 2 * a.scale_cap);
  float* epi_stage = reinterpret_cast<float*>(&sh + 1);   // 16-byte aligned (TcShared is)

  // Values that feed tcgen05 and TMA operands (TMEM and shared-memory
  // addresses, instruction descriptors) go through a lane-0 shuffle, which
  // the compiler knows to be warp-uniform. Otherwise it has to uniformise
  // them at every issue, and that happens inside the MMA thread's per-chunk
  // loop, whose gaps set the tensor pipe's idle time (same bits; prefill GEMM
  // 1031 -> 1170 TFLOP/s).
  const int warp = __shfl_sync(kFullMask, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages_a; ++s) {
      mbar_init(&sh.full_a[s], 1);
      mbar_init(&sh.empty_a[s], kTeamWarps);
    }
    for (int r = 0; r < SB; ++r) {
      mbar_init(&sh.b_full[r], 1);               // producer B (bytes)
      mbar_init(&sh.done[r], 1);
    }
    for (int r = 0; r < kABufs; ++r) mbar_init(&sh.a_full[r], kTeamWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], 4);
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_empty[b], kDequantWarps);
    }
    mbar_init(&sh.drain, 32);                    // every lane of the MMA warp
    if (kSplit) mbar_init(&sh.epi_bar, 4);
    for (int r = 0; r < kUnitRing; ++r) {
      mbar_init(&sh.u_full[r], 1);
      mbar_init(&sh.u_empty[r], kUnitReaders);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();                    // routing lists and prepared tokens are ready
  if (warp == kListWarp) {
    // Per active expert: id, segment and token-block count (ceil(cnt / nmax));
    // units are (expert, token block, 128-row tile).
    const int na = a.plan.meta[kMetaNumActive];
    int run = 0;
    for (int base = 0; base < na; base += 32) {
      const int u = base + lane;
      int nb = 0;
      if (u < na) {
        const int e = a.plan.active[u];
        const int beg = a.plan.offsets[e];
        const int cnt = a.plan.offsets[e + 1] - beg;
        sh.ex_id[u] = e;
        sh.ex_beg[u] = beg;
        sh.ex_cnt[u] = cnt;
        nb = (cnt + a.nmax - 1) / a.nmax;
      }
      int incl = nb;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += v;
      }
      if (u < na) sh.unit_prefix[u] = run + incl - nb;
      run += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) {
      sh.unit_prefix[na] = run;
      sh.num_active = na;
      sh.num_units = run * a.mtiles;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = __shfl_sync(kFullMask, sh.tmem_base, 0);
  const int num_units = sh.num_units;
  const int G = a.G, O = a.O;
  const int nk = G / 2;                              // chunks of 64 = two groups
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------- producer A: scales + weights
    // The whole warp runs the loop and its waits; lane 0 takes the units,
    // and one elected lane issues each copy. (Issuing copies from a loop
    // that lane 0 runs alone measured 3 % slower per plain-layout prefill
    // step, like the MMA issue: code under elect.sync issues better.)
    {
      // Weights: evict-first when the expert has one token block (each
      // tile read once); with several blocks every tile is read again for
      // each block, a wave or so later, so those keep the normal priority
      // and are not re-read from DRAM (skewed prefill 1 % faster).
      const uint64_t pol_once = l2_evict_first_policy();
      const uint64_t pol_reuse = l2_evict_normal_policy();
      int it = 0, issued = 0;
      RingPos pa, pu;
      int* counter = &a.plan.meta[a.counter_word];
      int next = 0;
      if (lane == 0) next = atomicAdd(counter, 1);       // one unit ahead
      next = __shfl_sync(kFullMask, next, 0);
      for (;; ++it) {
        const int idx = next < num_units ? next : -1;
        if (!mbar_wait_warp(&sh.u_empty[pu.idx], pu.phase ^ 1u)) { ok = false; break; }
        if (lane == 0) {
          sh.unit_ring[pu.idx] = idx;
          mbar_arrive(&sh.u_full[pu.idx]);               // releases the index
        }
        pu.next(kUnitRing);
        if (idx < 0) break;
        if (lane == 0) next = atomicAdd(counter, 1);
        next = __shfl_sync(kFullMask, next, 0);
        const Unit w = unit_at<kSplit>(a, sh, idx);
        if (w.ntok <= 0) { --it; continue; }
        const uint64_t pol = w.nblk > 1 ? pol_reuse : pol_once;
        if constexpr (kPrep) {
          // The tile's chunk blocks are consecutive: one bulk copy each.
          const unsigned char* blk =
              a.prep + ((size_t)w.e * a.mtiles + w.mt) * (size_t)nk * kStagePrep;
          for (int kc = 0; kc < nk; ++kc, ++issued) {
            if (!mbar_wait_warp(&sh.empty_a[pa.idx], pa.phase ^ 1u)) {
              ok = false;
              break;
            }
            if (elect_one()) {
              mbar_arrive_expect_tx(&sh.full_a[pa.idx], kStagePrep);
              bulk_copy_g2s(ring_a + (size_t)pa.idx * kStagePrep, blk + (size_t)kc * kStagePrep,
                            kStagePrep, &sh.full_a[pa.idx], pol);
            }
            pa.next(a.stages_a);
          }
          if (!ok) break;
          continue;
        }
        // The tile's scale bytes, by one bulk copy of the aligned span that
        // holds them when it stays inside the scales buffer.
        const int sb = it & 1;
        if (!mbar_wait_warp(&sh.s_empty[sb], ((uint32_t)(it >> 1) & 1u) ^ 1u)) { ok = false; break; }
        const size_t row0 = (size_t)w.e * O + w.m0;
        const uintptr_t s_lo = reinterpret_cast<uintptr_t>(a.scales + row0 * G);
        const uintptr_t s_hi = s_lo + (uintptr_t)w.rows * G;
        const uintptr_t c_lo = s_lo & ~(uintptr_t)15, c_hi = (s_hi + 15) & ~(uintptr_t)15;
        const uintptr_t end = reinterpret_cast<uintptr_t>(a.scales_end);
        // Gate/up tiles: the up rows' scale bytes are a second span, copied
        // right after the first.
        const uintptr_t u_lo = s_lo + (uintptr_t)a.F * G, u_hi = u_lo + (uintptr_t)w.rows * G;
        const uintptr_t d_lo = u_lo & ~(uintptr_t)15, d_hi = (u_hi + 15) & ~(uintptr_t)15;
        const uint32_t bytes1 = (uint32_t)(c_hi - c_lo);
        const uint32_t bytes2 = kSplit ? (uint32_t)(d_hi - d_lo) : 0u;
        const bool copy = c_hi <= end && (!kSplit || d_hi <= end) &&
                          (size_t)bytes1 + bytes2 <= a.scale_cap;
        if (elect_one()) {
          sh.scale_off[sb] = copy ? (int)(s_lo - c_lo) : -1;
          if constexpr (kSplit) sh.scale_off_up[sb] = copy ? (int)(bytes1 + (u_lo - d_lo)) : -1;
          if (copy) {
            unsigned char* dst = scale_buf + (size_t)sb * a.scale_cap;
            mbar_arrive_expect_tx(&sh.s_full[sb], bytes1 + bytes2);
            bulk_copy_g2s(dst, reinterpret_cast<const void*>(c_lo), bytes1, &sh.s_full[sb], pol);
            if (bytes2)
              bulk_copy_g2s(dst + bytes1, reinterpret_cast<const void*>(d_lo), bytes2,
                            &sh.s_full[sb], pol);
          } else {
            mbar_arrive(&sh.s_full[sb]);
          }
        }
        for (int kc = 0; kc < nk; ++kc, ++issued) {
          if (!mbar_wait_warp(&sh.empty_a[pa.idx], pa.phase ^ 1u)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&sh.full_a[pa.idx], kStageA);
            unsigned char* stage = ring_a + (size_t)pa.idx * kStageA;
            if constexpr (kSplit) {
              // 64 gate rows, then the 64 matching up rows (same swizzle
              // phase: the second box starts 2048 bytes in).
              tma_load_2d(stage, &maps.a_half, kc * 32, (int)row0, &sh.full_a[pa.idx], pol);
              tma_load_2d(stage + kStageA / 2, &maps.a_half, kc * 32, (int)(row0 + a.F),
                          &sh.full_a[pa.idx], pol);
            } else {
              tma_load_2d(stage, &maps.a, kc * 32, (int)row0, &sh.full_a[pa.idx], pol);
            }
          }
          pa.next(a.stages_a);
        }
      }
      if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
      // Wait (bounded) until the copies the warp issued have landed: the
      // last min(issued, stages) uses of the ring, walking back from pa.
      if (lane == 0) {
        for (int k = 0; k < min(issued, a.stages_a); ++k) {
          int idx = pa.idx - 1 - k;
          uint32_t ph = pa.phase;
          if (idx < 0) { idx += a.stages_a; ph ^= 1u; }
          if (!mbar_wait(&sh.full_a[idx], ph)) break;
        }
        if constexpr (!kPrep)
          for (int k = max(0, it - 2); k < it; ++k)
            if (!mbar_wait(&sh.s_full[k & 1], (uint32_t)(k >> 1) & 1u)) break;
      }
    }
    __syncwarp();
  } else if (warp == kProdBWarp) {
    // ------------------------------------------------------ producer B: tokens
    // Like producer A: the whole warp waits, one elected lane issues.
    {
      const uint64_t pol = l2_evict_last_policy();      // tokens: reread per tile
      int issued = 0, idx;
      RingPos pr, pu;
      while (ok) {
        if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
        if (idx < 0) break;
        const Unit w = unit_at<kSplit>(a, sh, idx);
        if (w.ntok <= 0) continue;
        const uint32_t box = (uint32_t)load_rows(w.load) * 128u;
        for (int kc = 0; kc < nk; ++kc, ++issued) {
          if (!mbar_wait_warp(&sh.done[pr.idx], pr.phase ^ 1u)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&sh.b_full[pr.idx], box);
            tma_load_2d(ring_b + (size_t)pr.idx * a.stage_b, &maps.b[w.load], kc * kBK, w.tok0,
                        &sh.b_full[pr.idx], pol);
          }
          pr.next(SB);
        }
      }
      if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
      if (lane == 0) {
        for (int k = 0; k < min(issued, SB); ++k) {
          int ridx = pr.idx - 1 - k;
          uint32_t ph = pr.phase;
          if (ridx < 0) { ridx += SB; ph ^= 1u; }
          if (!mbar_wait(&sh.b_full[ridx], ph)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues a
    // chunk's MMAs and, in the same block, the commits that depend on them
    // (a commit tracks only the MMAs of the thread that issues it). elect.sync
    // need not pick the same lane each time, and MMAs into one accumulator
    // from different threads are ordered only across a thread
    // synchronisation bracketed by the tcgen05 fences: the issuing lane
    // fences before the warp synchronises, every lane after its waits.
    int it = 0, idx;
    uint32_t chunk = 0;               // chunks issued so far: chunk c uses A buffer c % kABufs
    RingPos pb, pu;                   // token stage, unit ring
    for (; ok; ++it) {
      if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
      if (idx < 0) break;
      const Unit w = unit_at<kSplit>(a, sh, idx);
      if (w.ntok <= 0) { --it; continue; }
      const int db = it & 1;
      if (!mbar_wait_warp(&sh.d_empty[db], ((uint32_t)(it >> 1) & 1u) ^ 1u)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem + kDCol + (uint32_t)db * kNMax;
      const uint32_t idesc = __shfl_sync(kFullMask, mma_idesc(kBM, w.nmma, tile_f16(a, w)), 0);
      for (int kc = 0; kc < nk; ++kc) {
        // Ready once all kTeamWarps warps of the team arrived for this
        // chunk: a warp arrives for its next chunk in this buffer only after
        // these MMAs finished, so the barrier cannot run a phase ahead.
        // (Every lane gives up together, so that the warp stays converged
        // for the shuffle and elect.sync below.)
        const uint32_t buf = chunk % kABufs;
        if (!mbar_wait_warp(&sh.a_full[buf], (chunk / kABufs) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t b_addr =
            __shfl_sync(kFullMask, smem_addr(ring_b + (size_t)pb.idx * a.stage_b), 0);
        const uint32_t a_tmem = tmem + kACol + buf * 32;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128(b_addr + kk * 32), idesc,
                      (kc > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sh.done[pb.idx]);     // token stage and A buffer free once these finish
          if (kc == nk - 1) tc_commit(&sh.d_full[db]);   // accumulator complete
          tc_fence_before_sync();
        }
        __syncwarp();
        ++chunk;
        pb.next(SB);
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
    // Do not free TMEM under running MMAs: every lane commits (whichever
    // lanes issued MMAs), and the drain completes when all of them have.
    tc_commit(&sh.drain);
    mbar_wait(&sh.drain, 0);
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + kDequantWarps) {
    // -------------------------------------------------------- dequantizers
    const int sub = warp - kDequantWarp0;
    const int team = sub / kTeamWarps;
    const int q = warp & 3;                          // TMEM lane quarter
    const int m = 32 * q + lane;                     // weight row in the tile
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int next = team;                                 // chunk `team` is the team's first
    int it = 0, base = 0, idx;
    RingPos pu;
    for (; ok; ++it) {
      if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
      if (idx < 0) break;
      const Unit w = unit_at<kSplit>(a, sh, idx);
      if (w.ntok <= 0) { --it; continue; }
      const int sb = it & 1;
      if (!kPrep && !mbar_wait_warp(&sh.s_full[sb], (uint32_t)(it >> 1) & 1u)) {
        ok = false;
        break;
      }
      // Row m's place in its span: gate/up tiles hold two spans of rows
      // (m < 64: gate row f0 + m; else up row F + f0 + m - 64).
      const bool up = kSplit && m >= kBM / 2;
      const int hrow = min(kSplit ? (m & (kBM / 2 - 1)) : m, w.rows - 1);
      const bool f16 = tile_f16(a, w);
      const int r = f16 ? a.row_off[(size_t)w.e * O + (up ? a.F : 0) + w.m0 + hrow] : 0;
      const bool convert = !f16 && a.b_f16 != 0;     // bf16 tile on f16 token rows
      const int tid = (sub % kTeamWarps) * 32 + lane;
      if constexpr (kPrep) {
        ok = dequant_tile<true>(sh, ring_a, a.stage_a, a.stages_a, ring_b, a.stage_b, SB, tmem,
                                lane_base, m, lane, tid, base, nk, w.nmma, next,
                                [](int) { return 0u; }, f16, r, convert);
      } else {
        // The choice of scale source is the same for the whole tile: take it
        // once, so the chunk loop holds no global load.
        const int soff = up ? sh.scale_off_up[sb] : sh.scale_off[sb];
        if (soff >= 0) {
          const unsigned char* srow =
              scale_buf + (size_t)sb * a.scale_cap + soff + (size_t)hrow * G;
          ok = dequant_tile<false>(sh, ring_a, a.stage_a, a.stages_a, ring_b, a.stage_b, SB, tmem,
                                   lane_base, m, lane, tid, base, nk, w.nmma, next,
                                   [&](int g) { return (uint32_t)srow[g]; }, f16, r, convert);
        } else {
          const uint8_t* grow =
              a.scales + ((size_t)w.e * O + (up ? a.F : 0) + w.m0 + hrow) * G;
          ok = dequant_tile<false>(sh, ring_a, a.stage_a, a.stages_a, ring_b, a.stage_b, SB, tmem,
                                   lane_base, m, lane, tid, base, nk, w.nmma, next,
                                   [&](int g) { return (uint32_t)__ldg(grow + g); }, f16, r,
                                   convert);
        }
      }
      base += nk;
      if (!ok) break;
      if constexpr (!kPrep) {
        fence_proxy_async_smem();                    // scale bytes read: the next copy may land
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_empty[sb]);
      }
    }
    if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    float* stage = epi_stage + (size_t)(warp - kEpiWarp0) * (kEpiStage / 4);
    const int m = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int it = 0, idx;
    uint32_t epi_phase = 0;
    RingPos pu;
    for (; ok; ++it) {
      if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
      if (idx < 0) break;
      const Unit w = unit_at<kSplit>(a, sh, idx);
      if (w.ntok <= 0) { --it; continue; }
      const int db = it & 1;
      // The accumulator holds 2^(sigma - r) times the result for f16 token
      // rows (r = 0 in bf16 mode).
      int roff = 0;
      if (tile_f16(a, w)) {
        const bool up = kSplit && m >= kBM / 2;
        const int hrow = min(kSplit ? (m & (kBM / 2 - 1)) : m, w.rows - 1);
        roff = a.row_off[(size_t)w.e * O + (up ? a.F : 0) + w.m0 + hrow];
      }
      if constexpr (kSplit) {
        if (!mbar_wait_warp(&sh.d_full[db], (uint32_t)(it >> 1) & 1u)) { ok = false; break; }
        tc_fence_after_sync();
        if (!swiglu_epilogue(a, w, tmem + kDCol + (uint32_t)db * kNMax, lane_base, epi_stage, q,
                             lane, &sh.epi_bar, epi_phase, roff)) {
          ok = false;
          break;
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.d_empty[db]);
        continue;
      }
      const bool row_ok = m < w.rows;
      float* out_col = a.part + w.m0 + m;

      // Four consecutive rows per store: this warp's 32 rows x 16 columns go
      // through shared memory (column-major), then lane (c, j) of each round
      // stores rows 4j..4j+3 of column c. Needs whole 4-row groups inside
      // the tile and 16-byte aligned part rows.
      const bool vec = (O & 3) == 0 && 32 * q + 32 <= w.rows;
      const int jr = lane & 7;                       // 4-row group of the lane
      float* part_rows = a.part + w.m0 + 32 * q + 4 * jr;
      // Partial results are written once and read once by the combine: keep
      // them from evicting the token rows, which every row tile rereads.
      const uint64_t st_pol = l2_evict_first_policy();
      if (!mbar_wait_warp(&sh.d_full[db], (uint32_t)(it >> 1) & 1u)) { ok = false; break; }
      tc_fence_after_sync();
      for (int c0 = 0; c0 < w.nmma; c0 += 16) {
        // Pair ids (and for f16 rows the powers of two) of these 16 columns:
        // one load per lane, then broadcast.
        int my_pair = 0, my_sig = 0;
        if (lane < 16 && c0 + lane < w.ntok) {
          my_pair = a.plan.pair_list[w.tok0 + c0 + lane];
          if (a.b_f16) my_sig = a.sigma[w.tok0 + c0 + lane];
        }
        uint32_t v[16];
        __syncwarp();
        tmem_ld16(tmem + lane_base + kDCol + (uint32_t)db * kNMax + (uint32_t)c0, v);
        tmem_wait_ld();
        if (a.b_f16) {
          // One multiply by 2^(r - sigma) per element; the range check once
          // per 16 columns (the smallest and largest sigma of the group).
          int smin = lane < 16 && c0 + lane < w.ntok ? my_sig : 1 << 20;
          int smax = lane < 16 && c0 + lane < w.ntok ? my_sig : -(1 << 20);
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) {
            smin = min(smin, __shfl_xor_sync(kFullMask, smin, o));
            smax = max(smax, __shfl_xor_sync(kFullMask, smax, o));
          }
          smin = __shfl_sync(kFullMask, smin, 0);
          smax = __shfl_sync(kFullMask, smax, 0);
          if (roff - smax >= -126 && roff - smin <= 127) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int e = roff - __shfl_sync(kFullMask, my_sig, i) + 127;
              v[i] = __float_as_uint(__uint_as_float(v[i]) * __uint_as_float((uint32_t)e << 23));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int sg = __shfl_sync(kFullMask, my_sig, i);
              v[i] = __float_as_uint(scale_pow2(__uint_as_float(v[i]), roff - sg));
            }
          }
        }
        if (vec) {
#pragma unroll
          for (int i = 0; i < 16; ++i) stage[i * 32 + lane] = __uint_as_float(v[i]);
          __syncwarp();
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int c = 4 * r + (lane >> 3);
            const int pair = __shfl_sync(kFullMask, my_pair, c);
            if (c0 + c < w.ntok)
              st_f4_policy(part_rows + (size_t)pair * O,
                           *reinterpret_cast<const float4*>(stage + c * 32 + 4 * jr), st_pol);
          }
          __syncwarp();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int pair = __shfl_sync(kFullMask, my_pair, i);
            if (row_ok && c0 + i < w.ntok) out_col[(size_t)pair * O] = __uint_as_float(v[i]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty[db]);
    }
    if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Token rows grouped by expert for the tensor-core kernel: row p of xg is
// token t = pair_list[p] / K as f16(x[t] 2^sigma) with max |x_t| 2^sigma in
// [2^14, 2^15), sigma[p] its power of two (the computation of prep_token
// with top = 14). One warp per token: it reads and converts the token's row
// once and writes it to the positions of its valid pairs (pos_of_pair), so
// a token picked by K experts costs one conversion and K row stores. Also
// resets the kernel's unit counters and, for gate/up tiles, the down
// projection's ids.
__global__ void __launch_bounds__(256)
group_tokens_kernel(const __nv_bfloat16* __restrict__ x, __half* __restrict__ xg,
                    int* __restrict__ sigma, RoutePlan plan, int T, int I, int K,
                    int32_t* __restrict__ zero_ids, int64_t nzero) {
  pdl_launch_dependents();
  pdl_wait();                    // the bucketer's lists are ready
  // The tensor-core kernel after this one takes its units from this counter.
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    plan.meta[kMetaUnitCounter] = 0;
    plan.meta[kMetaUnitCounter2] = 0;      // a second tensor-core kernel on these lists
  }
  // Gate/up tiles: the down projection's ids start at expert 0 (the kernel
  // after this one writes the valid pairs' experts).
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nzero;
       i += (int64_t)gridDim.x * blockDim.x)
    zero_ids[i] = 0;
  constexpr int kSlots = 8;                        // pair positions held per pass
  const int lane = threadIdx.x & 31, warps = blockDim.x / 32, nvec = I / 8;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * I);
    int s = -1;                                    // computed once, on the first valid slot
    float up = 0.f;
    for (int k0 = 0; k0 < K; k0 += kSlots) {
      int pos[kSlots];
      bool any = false;
#pragma unroll
      for (int j = 0; j < kSlots; ++j) {
        pos[j] = k0 + j < K ? plan.pos_of_pair[(size_t)t * K + k0 + j] : -1;
        any |= pos[j] >= 0;
      }
      if (!any) continue;
      if (s < 0) {
        uint32_t m = 0;                            // max |x| as float32 bits
        for (int i = lane; i < nvec; i += 32) {
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
        s = 0;
        if (m != 0 && ex < 255) s = min(126, 127 + 14 - ex);
        up = __uint_as_float((uint32_t)(s + 127) << 23);
      }
      for (int i = lane; i < nvec; i += 32) {
        const uint4 v = __ldg(row + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 p = __floats2half2_rn(__uint_as_float(w[k] << 16) * up,
                                              __uint_as_float(w[k] & 0xffff0000u) * up);
          h[k] = *reinterpret_cast<const uint32_t*>(&p);
        }
        const uint4 hv = make_uint4(h[0], h[1], h[2], h[3]);
#pragma unroll
        for (int j = 0; j < kSlots; ++j)
          if (pos[j] >= 0) reinterpret_cast<uint4*>(xg + (size_t)pos[j] * I)[i] = hv;
      }
#pragma unroll
      for (int j = 0; j < kSlots; ++j)
        if (lane == j && pos[j] >= 0) sigma[pos[j]] = s;
    }
  }
}

// Operand modes of the tensor-core kernel's tiles: for tile mt of expert e
// (128 rows, or for gate/up tiles 64 gate rows and their 64 up rows), every
// row's smallest and largest scale byte; tile_mode = 1 when every row spans
// at most kF16Span binades, row_off[row] = largest - 140 (so that the row's
// largest scaled weight is 6 * 2^13). One block of 128 threads per tile: the
// tile's scale bytes (one or two contiguous spans of rows) are copied into
// shared memory with consecutive threads on consecutive bytes, then thread m
// scans row m. It reads only the weights' scale bytes before it waits for the
// previous kernel, and writes its outputs only after that wait.
template <bool kSplit>
__global__ void __launch_bounds__(128)
tile_scan_kernel(const uint8_t* __restrict__ scales, int G, int O, int F, int mtiles,
                 uint8_t* __restrict__ tile_mode, int16_t* __restrict__ row_off) {
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t span[];   // kBM * G + 64 bytes
  const int mt = blockIdx.x, e = blockIdx.y, m = threadIdx.x;
  // Rows of each span: [r0, r0 + n) of expert e's matrix, stored at span
  // offset base.
  constexpr int kSpans = kSplit ? 2 : 1;
  constexpr int kSpanRows = kBM / kSpans;
  // Each span through the 16-byte aligned window that holds it (a 16-byte
  // aligned block never crosses a page, so the window's extra bytes are
  // always readable); row j of span h then starts at off[h] + j * G.
  __shared__ int off[kSpans];
  for (int h = 0; h < kSpans; ++h) {
    const int first = kSplit ? mt * kSpanRows : mt * kBM;
    const int limit = kSplit ? F : O;
    const int n = max(0, min(kSpanRows, limit - first));
    const int r0 = (kSplit && h == 1 ? F : 0) + first;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(scales + ((size_t)e * O + r0) * G);
    const uintptr_t w0 = lo & ~(uintptr_t)15, w1 = (lo + (uintptr_t)n * G + 15) & ~(uintptr_t)15;
    uint4* dst = reinterpret_cast<uint4*>(span + (size_t)h * (kSpanRows * G + 32));
    const uint4* src = reinterpret_cast<const uint4*>(w0);
    // Eight loads in flight per thread before their stores.
    const int nv = (int)((w1 - w0) / 16), step = blockDim.x;
    int i = m;
    for (; i + 7 * step < nv; i += 8 * step) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldg(src + i + j * step);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[i + j * step] = v[j];
    }
    for (; i < nv; i += step) dst[i] = __ldg(src + i);
    if (m == 0) off[h] = h * (kSpanRows * G + 32) + (int)(lo - w0);
  }
  __syncthreads();
  int row = -1;
  if (kSplit) {
    const int f = mt * kSpanRows + (m & (kSpanRows - 1));
    if (f < F) row = (m >= kSpanRows ? F : 0) + f;
  } else if (mt * kBM + m < O) {
    row = mt * kBM + m;
  }
  bool fits = true;
  uint32_t lo = 255, hi = 0;
  if (row >= 0) {
    const uint8_t* p = span + off[kSplit && m >= kSpanRows ? 1 : 0] + (size_t)(m % kSpanRows) * G;
    // Rows are G bytes apart: each thread starts at its own byte m mod G,
    // so that a warp's reads spread over the banks instead of piling onto
    // the few that G-byte strides hit.
    int g = m % G;
#pragma unroll 8
    for (int n = 0; n < G; ++n) {
      const uint32_t v = p[g];
      lo = min(lo, v);
      hi = max(hi, v);
      g = g + 1 == G ? 0 : g + 1;
    }
    fits = (int)(hi - lo) <= kF16Span;
  }
  const int all = __syncthreads_and(fits ? 1 : 0);
  // The outputs live in the call's scratch, which earlier kernels on the
  // stream may still be using: write them only once those have finished.
  pdl_wait();
  if (row >= 0) row_off[(size_t)e * O + row] = (int16_t)((int)hi - 140);
  if (m == 0) tile_mode[(size_t)e * mtiles + mt] = all ? 1 : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int num_sms_tc() {
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

size_t tc_shared_bytes(int stages_a, uint32_t stage_a, int stages_b, uint32_t stage_b,
                       uint32_t scale_cap) {
  return 1024 + (size_t)stages_b * stage_b + (size_t)stages_a * stage_a + 2 * (size_t)scale_cap +
         sizeof(TcShared) + (kTcThreads / 32 - kEpiWarp0) * (size_t)kEpiStage;
}

constexpr size_t kSmemLimit = 227 * 1024;

// Ring sizes and block width for one launch: as many token stages (up to
// kStagesBMax, at least kTeams) of the widest block (kNMax, else 128 token
// columns) as fit beside eight packed-weight stages of stage_a bytes, then as
// deep a packed-weight ring as shared memory allows (a multiple of kTeams:
// each dequantizer team keeps to its own stages, so the last use of a stage
// is always its own). Token refills wait for the MMAs of the chunk SB back,
// so the token ring's depth is what hides their latency. Returns false if
// nothing fits.
struct TcConfig {
  int nmax;
  int stages_b;
  int stages_a;
  uint32_t stage_b;
};
bool tc_config(uint32_t scale_cap, uint32_t stage_a, TcConfig* c) {
  for (int nmax : {kNMax, 128}) {
    const uint32_t sbytes = (uint32_t)nmax * 128u;
    for (int sb = kStagesBMax; sb >= kTeams; --sb) {
      if (tc_shared_bytes(2 * kTeams, stage_a, sb, sbytes, scale_cap) > kSmemLimit) continue;
      int sa = kStagesAMax;
      while (sa > kTeams && tc_shared_bytes(sa, stage_a, sb, sbytes, scale_cap) > kSmemLimit)
        sa -= kTeams;
      *c = TcConfig{nmax, sb, sa, sbytes};
      return true;
    }
  }
  return false;
}

template <bool kSplit, bool kPrep>
cudaError_t launch_tc(const TcMaps& maps, const TcArgs& args, size_t smem, cudaStream_t stream) {
  static std::mutex mu;
  static size_t opted[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && opted[dev] < smem) {
      cudaError_t err = cudaFuncSetAttribute(gemm_tc_kernel<kSplit, kPrep>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      opted[dev] = smem;
    }
  }
  return launch_after_previous(gemm_tc_kernel<kSplit, kPrep>, dim3((unsigned)num_sms_tc()),
                               dim3(kTcThreads), smem, stream, maps, args);
}

}  // namespace

void* tensor_map_encoder() { return reinterpret_cast<void*>(encode_fn()); }

cudaError_t launch_group_tokens(const void* x, const RoutePlan& plan, __half* xg, int* sigma,
                                int64_t T, int64_t I, int64_t K, int32_t* zero_ids,
                                cudaStream_t stream) {
  if (plan.pos_of_pair == nullptr) return cudaErrorInvalidValue;
  const int64_t P = T * K;
  const int64_t blocks = std::min<int64_t>((T + 7) / 8, (int64_t)num_sms_tc() * 8);
  return launch_after_previous(group_tokens_kernel, dim3((unsigned)std::max<int64_t>(blocks, 1)),
                               dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x), xg,
                               sigma, plan, (int)T, (int)I, (int)K, zero_ids,
                               zero_ids != nullptr ? P : (int64_t)0);
}

size_t gemm_tc_grouped_bytes(int64_t T, int64_t K, int64_t I) {
  return (size_t)T * K * I * sizeof(__half);
}

int64_t gemm_tc_row_tiles(int64_t O, int64_t F) {
  return F > 0 ? (F + kBM / 2 - 1) / (kBM / 2) : (O + kBM - 1) / kBM;
}

bool tile_scan_fits(int64_t I) { return (size_t)kBM * (I / 32) + 64 <= 48 * 1024; }

cudaError_t launch_tile_scan(const uint8_t* scales, int64_t E, int64_t I, int64_t O, int64_t F,
                             uint8_t* tile_mode, int16_t* row_off, cudaStream_t stream) {
  const int64_t mtiles = gemm_tc_row_tiles(O, F);
  if (E <= 0 || mtiles <= 0) return cudaSuccess;
  const dim3 grid((unsigned)mtiles, (unsigned)E);
  const size_t smem = (size_t)kBM * (I / 32) + 64;   // a tile's scale bytes, two windows
  if (!tile_scan_fits(I)) return cudaErrorInvalidValue;
  if (F > 0)
    return launch_after_previous(tile_scan_kernel<true>, grid, dim3(128), smem, stream, scales,
                                 (int)(I / 32), (int)O, (int)F, (int)mtiles, tile_mode, row_off);
  return launch_after_previous(tile_scan_kernel<false>, grid, dim3(128), smem, stream, scales,
                               (int)(I / 32), (int)O, 0, (int)mtiles, tile_mode, row_off);
}

// Bytes per scale buffer: one tile's span, or the two spans of a gate/up tile.
uint32_t tc_scale_cap(int64_t G, bool halves) {
  const uint32_t whole = (uint32_t)((kBM * G + 31) / 16 * 16);
  const uint32_t two = 2u * (uint32_t)(((kBM / 2) * G + 31) / 16 * 16);
  return halves ? std::max(whole, two) : whole;
}

bool gemm_tc_supported(int64_t E, int64_t I, int64_t O) {
  const int64_t G = I / 32;
  if (G % 2 != 0) return false;                    // chunks of whole group pairs
  if (E > kMaxExpertsTc || E * O > 0x7fffffff) return false;
  TcConfig c;
  return tc_config(tc_scale_cap(G, false), kStageA, &c) && tc_config(0u, kStagePrep, &c);
}

bool gemm_tc_swiglu_supported(int64_t E, int64_t I, int64_t F) {
  TcConfig c;
  return F > 0 && F % 32 == 0 && gemm_tc_supported(E, I, 2 * F) &&
         tc_config(tc_scale_cap(I / 32, true), kStageA, &c);
}

cudaError_t launch_gemm_tc(const TcTokens& tok, const TcTileModes& modes, const uint8_t* packed,
                           const uint8_t* scales, const RoutePlan& plan, float* part,
                           unsigned long long* status, int64_t E, int64_t I, int64_t O,
                           int64_t K, const SwigluTiles& swiglu, cudaStream_t stream,
                           int counter_word, const uint8_t* prepared) {
  if (swiglu.F > 0 && (O != 2 * swiglu.F || !gemm_tc_swiglu_supported(E, I, swiglu.F)))
    return cudaErrorInvalidValue;
  const bool prep = prepared != nullptr;
  if (prep && swiglu.F > 0) return cudaErrorInvalidValue;
  const int64_t G = I / 32;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  TcConfig cfg;
  const uint32_t scale_cap = prep ? 0u : tc_scale_cap(G, swiglu.F > 0);
  const uint32_t stage_a = prep ? kStagePrep : kStageA;
  if (!tc_config(scale_cap, stage_a, &cfg)) return cudaErrorInvalidValue;

  // Tensor maps (the prepared layout needs none for the weights).
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!prep) {
    const cuuint64_t dims[2] = {(cuuint64_t)(G * 16), (cuuint64_t)(E * O)};
    const cuuint64_t strides[1] = {(cuuint64_t)(G * 16)};
    const cuuint32_t box[2] = {32, (cuuint32_t)kBM};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const cuuint32_t half_box[2] = {32, (cuuint32_t)(kBM / 2)};
    if (enc(&maps.a_half, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), dims,
            strides, half_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int l = 0; l < kNumLoads; ++l) {
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)std::max<int64_t>(tok.nrows, 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)(I * 2)};
    const cuuint32_t box[2] = {64, (cuuint32_t)load_rows(l)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&maps.b[l], tok.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
            2, const_cast<void*>(tok.rows), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  TcArgs args;
  args.plan = plan;
  args.scales = prep ? nullptr : scales;
  args.scales_end = prep ? nullptr : scales + (size_t)E * O * G;
  args.prep = prepared;
  args.stage_a = stage_a;
  args.part = part;
  args.status = status;
  args.sigma = tok.sigma;
  args.G = (int)G;
  args.O = (int)O;
  args.K = (int)K;
  args.F = (int)swiglu.F;
  args.h = static_cast<__nv_bfloat16*>(swiglu.h);
  args.sel2 = swiglu.sel2;
  args.h_grouped = swiglu.grouped ? 1 : 0;
  args.counter_word = counter_word;
  args.mtiles = (int)gemm_tc_row_tiles(O, swiglu.F);
  args.scale_cap = scale_cap;
  args.b_f16 = tok.f16 && tok.sigma != nullptr ? 1 : 0;
  args.f16_tiles = args.b_f16 && modes.tile_mode != nullptr && modes.row_off != nullptr ? 1 : 0;
  args.tile_mode = modes.tile_mode;
  args.row_off = modes.row_off;
  // Test knob: MXFP4EL_TC_MODE=bf16 keeps every tile in the bf16 operand mode.
  if (const char* env = std::getenv("MXFP4EL_TC_MODE"))
    if (std::strcmp(env, "bf16") == 0) args.f16_tiles = 0;
  args.nmax = cfg.nmax;
  args.stage_b = cfg.stage_b;
  args.stages_a = cfg.stages_a;
  args.stages_b = cfg.stages_b;
  const size_t smem =
      tc_shared_bytes(cfg.stages_a, stage_a, cfg.stages_b, cfg.stage_b, scale_cap);
  if (prep) return launch_tc<false, true>(maps, args, smem, stream);
  return swiglu.F > 0 ? launch_tc<true, false>(maps, args, smem, stream)
                      : launch_tc<false, false>(maps, args, smem, stream);
}

}  // namespace mxfp4el
