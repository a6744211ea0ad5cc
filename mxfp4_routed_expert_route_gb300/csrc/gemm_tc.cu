// gemm_tc.cu -- prefill-regime routed expert grouped GEMM on the 5th-gen
// tensor cores (tcgen05, TMEM, TMA).
//
// For every selected expert e and each block of up to 192 of its tokens it
// computes part[t*K+k, o] = sum_i W_e[o, i] x[t, i] for all output rows o,
// with W_e decoded from MXFP4 as in the problem statement ("MXFP4 Routed
// Expert Linear", Kimi K3): W_e[o, 32g+2j (+1)] = LUT[low (high) nibble of
// packed[e,o,g,j]] * 2^(scales[e,o,g] - 127).
//
// Shape ("swap AB"): M = 128 weight rows per tile, N = the tokens of one
// block (16..192, a multiple of 16), K = I in chunks of 64 (two groups).
//   * A (weights) is decoded exactly to bf16 -- every E2M1 value times a
//     power of two is a bf16 number while it stays in bf16's range -- and
//     written straight into tensor memory: row m in TMEM lane m, two K
//     elements per 32-bit column.
//   * B (tokens) is a copy of x with the rows grouped by expert (written by
//     gather_tokens_kernel); TMA loads 64-wide K chunks with the 128-byte
//     swizzle that the K-major shared-memory descriptor describes.
//   * tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), accumulator in TMEM.
//
// Warp roles in a CTA of 24 warps (one CTA per SM, persistent over units
// (expert, token block, 128-row tile), which CTAs take from a global counter
// as they go, so the cost differences between units even out):
//   warp 0      producer of scales and packed weights (lane 0; a deep ring
//               of 4 KB stages covers HBM latency) and TMEM allocation; it
//               takes each next unit from the counter and hands its index to
//               the other roles through a small shared-memory ring
//   warp 1      MMA issuer (the whole warp waits, one elected lane issues)
//   warp 2      per-expert lists in shared memory at start
//   warp 3      producer of token tiles (lane 0)
//   warps 4-19  dequantize, in four teams of 4 warps: team t owns A buffer t
//               and takes chunks t, t+4, t+8, ..., so the teams' decode,
//               waits and stores interleave; in a team thread m (one weight
//               row) decodes both groups of the chunk into 32 TMEM columns
//   warps 20-23 epilogue: TMEM -> registers -> shared memory (transposed) ->
//               float32 partial results, four consecutive rows per store
// Four A buffers and two accumulators in TMEM, and a ring of four to six
// token stages in shared memory (a stage is refilled only after its chunk's
// MMAs finish, so its TMA latency needs several chunks of cover), let the
// loads, dequantize, MMA and epilogue of consecutive chunks and units
// overlap. Every wait is bounded;
// a role whose wait gives up records it, stops, and the CTA still waits
// (bounded) for its own copies and MMAs before freeing TMEM.
//
// Gate/up tiles (gemm_tc_kernel<SB, true>, the SwiGLU expert's stacked
// gate/up projection, 2F rows with the gate rows first): a tile's 128 rows
// are 64 gate rows f0.. and the matching 64 up rows F + f0.. (two 64-row TMA
// boxes into one stage, two scale spans), so the epilogue holds g and u of
// the same (pair, f) and writes h = silu(g) * u in bf16 instead of partial
// results, by pair or in the lists' grouped order; the down projection can
// then run as a second instance on the same lists (its own unit counter).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr int kTcThreads = 768;
constexpr int kBM = 128;                    // weight rows per tile
constexpr int kBK = 64;                     // K elements per stage
constexpr int kNMax = 192;                  // tokens per block
constexpr int kStagesAMax = 16;            // packed-weight ring (from HBM)
constexpr int kRing = 4;                   // TMEM A buffers (one per dequantizer team)
constexpr int kStagesBMax = 6;             // token stages, as shared memory allows
constexpr uint32_t kStageB = kNMax * 128;   // token tile, 128 B per row
constexpr uint32_t kStageA = kBM * 32;      // packed bytes, 32 B per row
static_assert(kStageB % 1024 == 0 && kStageA % 1024 == 0, "stages keep 1024-byte alignment");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = 0;               // two accumulators of kNMax columns
constexpr uint32_t kACol = 2 * kNMax;       // kRing A buffers of 32 columns
static_assert(kACol + kRing * 32 <= kTmemCols, "TMEM budget");
constexpr int kMaxExpertsTc = 512;          // per-expert lists kept in shared memory
constexpr uint32_t kEpiStage = 16 * 32 * 4; // epilogue staging per warp: 16 columns x 32 rows
constexpr int kUnitRing = 4;                // unit indices handed from producer A
constexpr int kDequantWarp0 = 4, kDequantWarps = 16, kTeamWarps = 4, kEpiWarp0 = 20;
// Readers of the unit ring, one arrival each: producer B, the MMA warp, the
// dequantizer warps and the epilogue warps.
constexpr int kUnitReaders = 2 + kDequantWarps + (kTcThreads / 32 - kEpiWarp0);
static_assert(kDequantWarps == kRing * kTeamWarps, "one team per A buffer");
constexpr int kNumLoads = 5;                // token-box heights
__host__ __device__ constexpr int load_rows(int l) {
  return l == 0 ? 16 : l == 1 ? 32 : l == 2 ? 64 : l == 3 ? 128 : 192;
}

struct TcArgs {
  RoutePlan plan;
  const uint8_t* scales;
  const uint8_t* scales_end;
  float* part;                   // [T*K, O]
  unsigned long long* status;
  int G, O, K;
  int mtiles;                    // ceil(O / 128)
  int stages_a;
  uint32_t scale_cap;            // bytes per scale buffer
  // Gate/up tiles of the SwiGLU expert (F > 0; the matrix has 2F rows, gate
  // rows first): tile rows 0..63 are gate rows f0.., rows 64..127 the
  // matching up rows F + f0..; the epilogue writes h = silu(gate) * up in
  // bf16 and the pairs' expert ids instead of the partial results.
  int F;
  __nv_bfloat16* h;              // (P, F), row = pair (or position in the lists: h_grouped)
  int32_t* sel2;                 // (P): expert of each pair (zeroed by the gather), or null
  int h_grouped;
  int counter_word;              // plan.meta word this kernel takes its units from
};

struct TcMaps {
  CUtensorMap a;                 // packed weights as uint8 [E*O, G*16], box {32, 128}
  CUtensorMap b[kNumLoads];      // grouped tokens bf16 [P, I], box {64, rows}, 128B swizzle
  CUtensorMap a_half;            // packed weights, box {32, 64} (gate/up tiles)
};

struct __align__(16) TcShared {
  uint64_t full_a[kStagesAMax], empty_a[kStagesAMax];
  // Chunk c uses token stage c % SB and TMEM A buffer c % kRing.
  uint64_t full_b[kStagesBMax];  // tokens landed (TMA)
  uint64_t done[kStagesBMax];    // the chunk's MMAs finished: its stage and A buffer free
  uint64_t a_full[kRing];        // A buffer written (dequantizers)
  uint64_t d_full[2], d_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t drain;
  uint64_t u_full[kUnitRing], u_empty[kUnitRing];
  int unit_ring[kUnitRing];      // unit indices in the order this CTA takes them; -1 ends
  uint32_t tmem_base;
  int scale_off[2];              // per scale buffer: offset of the tile's first byte, or -1
  int num_units;
  int num_active;
  // Per active expert u: id, first position in the grouped list, tokens,
  // and the prefix of token blocks (unit_prefix[num_active] = all blocks).
  int ex_id[kMaxExpertsTc];
  int ex_beg[kMaxExpertsTc];
  int ex_cnt[kMaxExpertsTc];
  int unit_prefix[kMaxExpertsTc + 1];
  // Gate/up tiles only.
  int scale_off_up[2];           // per scale buffer: offset of the up rows' first byte
  uint64_t epi_bar;              // the four epilogue warps
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
  w.load = 0;
  while (load_rows(w.load) < w.nmma) ++w.load;
  // Gate/up tiles: m0 is the first gate row f0, rows the valid rows of each half.
  constexpr int tm = kSplit ? kBM / 2 : kBM;
  w.m0 = mt * tm;
  w.rows = min(tm, (kSplit ? a.F : a.O) - w.m0);
  return w;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B bf16,
// both K-major, shape M x N.
__device__ __forceinline__ uint32_t mma_idesc(int m, int n) {
  return (1u << 4)                       // D format: fp32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
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

// A dequantizer team's place in the chunk sequence of its CTA: the global
// index of its next chunk (chunks of earlier tiles included), that chunk's
// packed stage and phase, and the use parity of the team's A buffer.
struct TeamPos {
  int next;
  int stage;
  uint32_t stage_phase;
  uint32_t buf_phase;
};

// The dequantizer's chunk loop for one tile whose chunks have global indices
// base .. base+nk-1: thread m of team t decodes groups 2kc and 2kc+1 of row
// m into A buffer t for each of the team's chunks kc. The packed tile
// arrives with the 32-byte swizzle: the two 16-byte halves of row m are
// exchanged when bit 2 of m is set, so eight consecutive rows read eight
// different bank groups. scale(g) returns the row's scale byte of group g.
// Returns false if a wait gave up.
template <int SB, typename ScaleFn>
__device__ __forceinline__ bool dequant_tile(TcShared& sh, const unsigned char* ring_a,
                                             int stages_a, uint32_t tmem, uint32_t lane_base,
                                             int team, int m, int lane, int base, int nk,
                                             TeamPos& tp, ScaleFn scale) {
  const uint32_t sw = (uint32_t)(m >> 2) & 1u;
  const uint32_t off0 = (uint32_t)m * 32u + sw * 16u, off1 = (uint32_t)m * 32u + (sw ^ 1u) * 16u;
  const uint32_t a_col = tmem + lane_base + kACol + (uint32_t)team * 32;
  for (; tp.next < base + nk; tp.next += kRing) {
    const int kc = tp.next - base;
    if (!mbar_wait(&sh.full_a[tp.stage], tp.stage_phase)) return false;
    const unsigned char* stage = ring_a + (size_t)tp.stage * kStageA;
    const uint4 pk0 = *reinterpret_cast<const uint4*>(stage + off0);
    const uint4 pk1 = *reinterpret_cast<const uint4*>(stage + off1);
    const uint32_t s0 = scale(2 * kc), s1 = scale(2 * kc + 1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty_a[tp.stage]);   // packed bytes consumed
    tp.stage += kRing;                                    // stages_a is a multiple of kRing
    if (tp.stage >= stages_a) {
      tp.stage -= stages_a;
      tp.stage_phase ^= 1u;
    }
    uint32_t v0[16], v1[16];
    dequant_group_bf16(pk0, s0, v0);
    dequant_group_bf16(pk1, s1, v1);
    // The buffer is free once the MMAs of this team's previous chunk finished
    // (chunk next - kRing, whose token stage is (next - kRing) % SB).
    if (tp.next >= kRing) {
      const int pc = tp.next - kRing;
      if (!mbar_wait(&sh.done[pc % SB], (uint32_t)(pc / SB) & 1u)) return false;
    }
    tc_fence_after_sync();
    tmem_st16(a_col, v0);
    tmem_st16(a_col + 16, v1);
    tmem_wait_st();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.a_full[team]);
    tp.buf_phase ^= 1u;
  }
  return true;
}

// The next unit index from the ring. kWarp: called by a whole warp, whose
// lane 0 arrives once all lanes have read it; else by one thread. Returns
// false if the wait gave up; *idx < 0 means no more units.
template <bool kWarp>
__device__ __forceinline__ bool pop_unit(TcShared& sh, RingPos& pu, int lane, int* idx) {
  if (!mbar_wait(&sh.u_full[pu.idx], pu.phase)) return false;
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
  const bool done = mbar_wait(bar, phase);
  phase ^= 1u;
  return done;
}

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Epilogue of a gate/up tile: 16 token columns at a time, each epilogue warp
// moves its 32 accumulator rows into shared memory (column-major, all four
// warps' rows side by side); then thread (cq, rp) forms h = silu(gate) * up
// for gate rows 2rp, 2rp+1 of the tile (their up rows sit 64 rows further,
// two warps on) and token columns 4cq..4cq+3, in float32, and stores each
// pair of rows as one bf16x2. The tile of the first rows of a token block
// also writes its pairs' expert for the down projection. Returns false if a
// wait gave up.
__device__ bool swiglu_epilogue(const TcArgs& a, const Unit& w, uint32_t d_cols,
                                uint32_t lane_base, float* epi_all, int q, int lane,
                                uint64_t* bar, uint32_t& phase) {
  float* mine = epi_all + q * (kEpiStage / 4);
  const int et = 32 * q + lane;
  const int rp = et & 31, cq = et >> 5;
  const int r0 = 2 * rp;
  const float* gsrc = epi_all + (r0 >> 5) * (kEpiStage / 4) + (r0 & 31);
  const float* usrc = gsrc + 2 * (kEpiStage / 4);
  const bool row_ok = r0 < w.rows;             // rows is even: r0 + 1 too
  for (int c0 = 0; c0 < w.nmma; c0 += 16) {
    uint32_t v[16];
    tmem_ld16(d_cols + lane_base + (uint32_t)c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) mine[i * 32 + lane] = __uint_as_float(v[i]);
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

// kSplit: gate/up tiles of the SwiGLU expert (see TcArgs::F).
template <int SB, bool kSplit>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  static_assert(SB >= kRing && SB <= kStagesBMax, "token ring depth");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Token stages need 1024-byte alignment (128-byte swizzle atoms).
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* ring_b = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* ring_a = ring_b + (size_t)SB * kStageB;
  unsigned char* scale_buf = ring_a + (size_t)a.stages_a * kStageA;
  TcShared& sh = *reinterpret_cast<TcShared*>(scale_buf + 2 * a.scale_cap);
  float* epi_stage = reinterpret_cast<float*>(&sh + 1);   // 16-byte aligned (TcShared is)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages_a; ++s) {
      mbar_init(&sh.full_a[s], 1);
      mbar_init(&sh.empty_a[s], kTeamWarps);
    }
    for (int r = 0; r < SB; ++r) {
      mbar_init(&sh.full_b[r], 1);
      mbar_init(&sh.done[r], 1);
    }
    for (int r = 0; r < kRing; ++r) mbar_init(&sh.a_full[r], kTeamWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], 4);
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_empty[b], kDequantWarps);
    }
    mbar_init(&sh.drain, 1);
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
  pdl_wait();                    // routing lists and grouped tokens are ready
  if (warp == 2) {
    // Per active expert: id, segment and token-block count (ceil(cnt / 192));
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
        nb = (cnt + kNMax - 1) / kNMax;
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
  const uint32_t tmem = sh.tmem_base;
  const int num_units = sh.num_units;
  const int G = a.G, O = a.O;
  const int nk = G / 2;                              // chunks of 64 = 2 groups
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------- producer A: scales + weights
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();     // weights: read once
      int it = 0, issued = 0;
      RingPos pa, pu;
      int* counter = &a.plan.meta[a.counter_word];
      int next = atomicAdd(counter, 1);                  // one unit ahead
      for (;; ++it) {
        const int idx = next < num_units ? next : -1;
        if (!mbar_wait(&sh.u_empty[pu.idx], pu.phase ^ 1u)) { ok = false; break; }
        sh.unit_ring[pu.idx] = idx;
        mbar_arrive(&sh.u_full[pu.idx]);                 // releases the index
        pu.next(kUnitRing);
        if (idx < 0) break;
        next = atomicAdd(counter, 1);
        const Unit w = unit_at<kSplit>(a, sh, idx);
        if (w.ntok <= 0) { --it; continue; }
        // The tile's scale bytes, by one bulk copy of the aligned span that
        // holds them when it stays inside the scales buffer.
        const int sb = it & 1;
        if (!mbar_wait(&sh.s_empty[sb], ((uint32_t)(it >> 1) & 1u) ^ 1u)) { ok = false; break; }
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
        for (int kc = 0; kc < nk; ++kc, ++issued) {
          if (!mbar_wait(&sh.empty_a[pa.idx], pa.phase ^ 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full_a[pa.idx], kStageA);
          unsigned char* stage = ring_a + (size_t)pa.idx * kStageA;
          if constexpr (kSplit) {
            // 64 gate rows, then the 64 matching up rows (same swizzle phase:
            // the second box starts 2048 bytes in).
            tma_load_2d(stage, &maps.a_half, kc * 32, (int)row0, &sh.full_a[pa.idx], pol);
            tma_load_2d(stage + kStageA / 2, &maps.a_half, kc * 32, (int)(row0 + a.F),
                        &sh.full_a[pa.idx], pol);
          } else {
            tma_load_2d(stage, &maps.a, kc * 32, (int)row0, &sh.full_a[pa.idx], pol);
          }
          pa.next(a.stages_a);
        }
      }
      if (!ok) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
      // Wait (bounded) until the copies this thread issued have landed: the
      // last min(issued, stages) uses of the ring, walking back from pa.
      for (int k = 0; k < min(issued, a.stages_a); ++k) {
        int idx = pa.idx - 1 - k;
        uint32_t ph = pa.phase;
        if (idx < 0) { idx += a.stages_a; ph ^= 1u; }
        if (!mbar_wait(&sh.full_a[idx], ph)) break;
      }
      for (int k = max(0, it - 2); k < it; ++k)
        if (!mbar_wait(&sh.s_full[k & 1], (uint32_t)(k >> 1) & 1u)) break;
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------ producer B: tokens
    if (lane == 0) {
      const uint64_t pol = l2_evict_last_policy();      // tokens: reread per tile
      int issued = 0, idx;
      RingPos pr, pu;
      while (ok) {
        if (!pop_unit<false>(sh, pu, 0, &idx)) { ok = false; break; }
        if (idx < 0) break;
        const Unit w = unit_at<kSplit>(a, sh, idx);
        if (w.ntok <= 0) continue;
        const uint32_t tx = (uint32_t)load_rows(w.load) * 128u;
        for (int kc = 0; kc < nk; ++kc, ++issued) {
          if (!mbar_wait(&sh.done[pr.idx], pr.phase ^ 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full_b[pr.idx], tx);
          tma_load_2d(ring_b + (size_t)pr.idx * kStageB, &maps.b[w.load], kc * kBK, w.tok0,
                      &sh.full_b[pr.idx], pol);
          pr.next(SB);
        }
      }
      if (!ok) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
      for (int k = 0; k < min(issued, SB); ++k) {
        int idx = pr.idx - 1 - k;
        uint32_t ph = pr.phase;
        if (idx < 0) { idx += SB; ph ^= 1u; }
        if (!mbar_wait(&sh.full_b[idx], ph)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and waits; one elected lane (always the
    // same one, so its commits track its own MMAs) issues.
    int it = 0, idx;
    RingPos pr, pb, pu;               // A buffer, token stage, unit ring
    for (; ok; ++it) {
      if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
      if (idx < 0) break;
      const Unit w = unit_at<kSplit>(a, sh, idx);
      if (w.ntok <= 0) { --it; continue; }
      const int db = it & 1;
      if (!mbar_wait(&sh.d_empty[db], ((uint32_t)(it >> 1) & 1u) ^ 1u)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t idesc = mma_idesc(kBM, w.nmma);
      const uint32_t d_tmem = tmem + kDCol + (uint32_t)db * kNMax;
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait(&sh.full_b[pb.idx], pb.phase) ||
            !mbar_wait(&sh.a_full[pr.idx], pr.phase)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t b_addr = smem_addr(ring_b + (size_t)pb.idx * kStageB);
        const uint32_t a_tmem = tmem + kACol + (uint32_t)pr.idx * 32;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128(b_addr + kk * 32), idesc,
                      (kc > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sh.done[pb.idx]);     // token stage and A buffer free once these finish
        }
        __syncwarp();
        pr.next(kRing);
        pb.next(SB);
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&sh.d_full[db]);   // accumulator complete
      __syncwarp();
    }
    if (!ok && lane == 0) atomicAdd(&a.status[kStatusWaitTimeouts], 1ull);
    // Do not free TMEM under running MMAs: wait (bounded) for all of them.
    if (elect_one()) tc_commit(&sh.drain);
    __syncwarp();
    mbar_wait(&sh.drain, 0);
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + kDequantWarps) {
    // -------------------------------------------------------- dequantizers
    const int team = (warp - kDequantWarp0) / kTeamWarps;
    const int q = warp & 3;                          // TMEM lane quarter
    const int m = 32 * q + lane;                     // weight row in the tile
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    TeamPos tp{team, team, 0u, 0u};                  // chunk `team` is the team's first
    int it = 0, base = 0, idx;
    RingPos pu;
    for (; ok; ++it) {
      if (!pop_unit<true>(sh, pu, lane, &idx)) { ok = false; break; }
      if (idx < 0) break;
      const Unit w = unit_at<kSplit>(a, sh, idx);
      if (w.ntok <= 0) { --it; continue; }
      const int sb = it & 1;
      if (!mbar_wait(&sh.s_full[sb], (uint32_t)(it >> 1) & 1u)) { ok = false; break; }
      // Row m's place in its span: gate/up tiles hold two spans of rows
      // (m < 64: gate row f0 + m; else up row F + f0 + m - 64).
      const bool up = kSplit && m >= kBM / 2;
      const int hrow = min(kSplit ? (m & (kBM / 2 - 1)) : m, w.rows - 1);
      const int soff = up ? sh.scale_off_up[sb] : sh.scale_off[sb];
      // The choice of scale source is the same for the whole tile: take it
      // once, so the chunk loop holds no global load.
      if (soff >= 0) {
        const unsigned char* srow =
            scale_buf + (size_t)sb * a.scale_cap + soff + (size_t)hrow * G;
        ok = dequant_tile<SB>(sh, ring_a, a.stages_a, tmem, lane_base, team, m, lane, base, nk,
                              tp, [&](int g) { return (uint32_t)srow[g]; });
      } else {
        const uint8_t* grow =
            a.scales + ((size_t)w.e * O + (up ? a.F : 0) + w.m0 + hrow) * G;
        ok = dequant_tile<SB>(sh, ring_a, a.stages_a, tmem, lane_base, team, m, lane, base, nk,
                              tp, [&](int g) { return (uint32_t)__ldg(grow + g); });
      }
      base += nk;
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_empty[sb]);
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
      if (!mbar_wait(&sh.d_full[db], (uint32_t)(it >> 1) & 1u)) { ok = false; break; }
      tc_fence_after_sync();
      if constexpr (kSplit) {
        if (!swiglu_epilogue(a, w, tmem + kDCol + (uint32_t)db * kNMax, lane_base, epi_stage, q,
                             lane, &sh.epi_bar, epi_phase)) {
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
      for (int c0 = 0; c0 < w.nmma; c0 += 16) {
        // Pair ids of these 16 columns: one load per lane, then broadcast.
        const int my_pair = (lane < 16 && c0 + lane < w.ntok)
                                ? a.plan.pair_list[w.tok0 + c0 + lane] : 0;
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + kDCol + (uint32_t)db * kNMax + (uint32_t)c0, v);
        tmem_wait_ld();
        if (vec) {
#pragma unroll
          for (int i = 0; i < 16; ++i) stage[i * 32 + lane] = __uint_as_float(v[i]);
          __syncwarp();
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int c = 4 * r + (lane >> 3);
            const int pair = __shfl_sync(kFullMask, my_pair, c);
            if (c0 + c < w.ntok)
              *reinterpret_cast<float4*>(part_rows + (size_t)pair * O) =
                  *reinterpret_cast<const float4*>(stage + c * 32 + 4 * jr);
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

// x rows grouped by expert: xg[pos, :] = x[pair_list[pos] / K, :].
__global__ void __launch_bounds__(256)
gather_tokens_kernel(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ xg,
                     RoutePlan plan, int I, int K, int32_t* __restrict__ zero_ids,
                     int64_t nzero) {
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
  const int npairs = plan.meta[kMetaNumPairs];
  const int vec_per_row = I / 8;
  const int warps = blockDim.x / 32;
  for (int pos = blockIdx.x * warps + (threadIdx.x >> 5); pos < npairs; pos += gridDim.x * warps) {
    const int t = plan.pair_list[pos] / K;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * I);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)pos * I);
    for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
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

size_t tc_shared_bytes(int stages_a, int stages_b, uint32_t scale_cap) {
  return 1024 + (size_t)stages_b * kStageB + (size_t)stages_a * kStageA + 2 * (size_t)scale_cap +
         sizeof(TcShared) + (kTcThreads / 32 - kEpiWarp0) * (size_t)kEpiStage;
}

constexpr size_t kSmemLimit = 227 * 1024;

template <int SB, bool kSplit>
cudaError_t launch_tc(const TcMaps& maps, const TcArgs& args, size_t smem, cudaStream_t stream) {
  static std::mutex mu;
  static size_t opted[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && opted[dev] < smem) {
      cudaError_t err = cudaFuncSetAttribute(gemm_tc_kernel<SB, kSplit>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      opted[dev] = smem;
    }
  }
  return launch_after_previous(gemm_tc_kernel<SB, kSplit>, dim3((unsigned)num_sms_tc()), dim3(kTcThreads),
                               smem, stream, maps, args);
}

}  // namespace

cudaError_t launch_gather_tokens(const void* x, const RoutePlan& plan, void* grouped,
                                 int64_t T, int64_t I, int64_t K, int32_t* zero_ids,
                                 cudaStream_t stream) {
  const int64_t P = T * K;
  const int64_t blocks = std::min<int64_t>((P + 7) / 8, (int64_t)num_sms_tc() * 8);
  return launch_after_previous(gather_tokens_kernel, dim3((unsigned)std::max<int64_t>(blocks, 1)),
                               dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x),
                               static_cast<__nv_bfloat16*>(grouped), plan, (int)I, (int)K,
                               zero_ids, zero_ids != nullptr ? P : (int64_t)0);
}

// Bytes per scale buffer: one tile's span, or the two spans of a gate/up tile.
uint32_t tc_scale_cap(int64_t G, bool halves) {
  const uint32_t whole = (uint32_t)((kBM * G + 31) / 16 * 16);
  const uint32_t two = 2u * (uint32_t)(((kBM / 2) * G + 31) / 16 * 16);
  return halves ? std::max(whole, two) : whole;
}

bool gemm_tc_supported(int64_t E, int64_t I, int64_t O) {
  const int64_t G = I / 32;
  if (G % 2 != 0) return false;                    // K chunks of 64
  if (E > kMaxExpertsTc || E * O > 0x7fffffff) return false;
  return tc_shared_bytes(kRing, kRing, tc_scale_cap(G, false)) <= kSmemLimit;
}

bool gemm_tc_swiglu_supported(int64_t E, int64_t I, int64_t F) {
  return F > 0 && F % 32 == 0 && gemm_tc_supported(E, I, 2 * F) &&
         tc_shared_bytes(kRing, kRing, tc_scale_cap(I / 32, true)) <= kSmemLimit;
}

size_t gemm_tc_grouped_bytes(int64_t T, int64_t K, int64_t I) {
  return (size_t)T * K * I * sizeof(__nv_bfloat16);
}

cudaError_t launch_gemm_tc(const void* x, const uint8_t* packed, const uint8_t* scales,
                           const RoutePlan& plan, void* grouped, float* part,
                           unsigned long long* status, int64_t T, int64_t E, int64_t I,
                           int64_t O, int64_t K, const SwigluTiles& swiglu,
                           cudaStream_t stream, int counter_word) {
  if (swiglu.F > 0 && (O != 2 * swiglu.F || !gemm_tc_swiglu_supported(E, I, swiglu.F)))
    return cudaErrorInvalidValue;
  const int64_t G = I / 32, P = T * K;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;

  (void)x;
  // Tensor maps.
  TcMaps maps;
  {
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
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)std::max<int64_t>(P, 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)(I * 2)};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)load_rows(l)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&maps.b[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, grouped, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  TcArgs args;
  args.plan = plan;
  args.scales = scales;
  args.scales_end = scales + (size_t)E * O * G;
  args.part = part;
  args.status = status;
  args.G = (int)G;
  args.O = (int)O;
  args.K = (int)K;
  args.F = (int)swiglu.F;
  args.h = static_cast<__nv_bfloat16*>(swiglu.h);
  args.sel2 = swiglu.sel2;
  args.h_grouped = swiglu.grouped ? 1 : 0;
  args.counter_word = counter_word;
  args.mtiles = swiglu.F > 0 ? (int)((swiglu.F + kBM / 2 - 1) / (kBM / 2))
                             : (int)((O + kBM - 1) / kBM);
  args.scale_cap = tc_scale_cap(G, swiglu.F > 0);
  // As many token stages as fit next to 8 packed-weight stages (their
  // refill latency is what the MMAs wait on), then as deep a packed-weight
  // ring as shared memory allows, a multiple of kRing so that each
  // dequantizer team keeps to its own stages.
  int sb = kRing;
  while (sb < kStagesBMax && tc_shared_bytes(2 * kRing, sb + 1, args.scale_cap) <= kSmemLimit) ++sb;
  int sa = kStagesAMax;
  while (sa > kRing && tc_shared_bytes(sa, sb, args.scale_cap) > kSmemLimit) sa -= kRing;
  args.stages_a = sa;
  const size_t smem = tc_shared_bytes(sa, sb, args.scale_cap);
  switch (sb) {
    case 6:
      return swiglu.F > 0 ? launch_tc<6, true>(maps, args, smem, stream)
                          : launch_tc<6, false>(maps, args, smem, stream);
    case 5:
      return swiglu.F > 0 ? launch_tc<5, true>(maps, args, smem, stream)
                          : launch_tc<5, false>(maps, args, smem, stream);
    default:
      return swiglu.F > 0 ? launch_tc<4, true>(maps, args, smem, stream)
                          : launch_tc<4, false>(maps, args, smem, stream);
  }
}

}  // namespace mxfp4el
