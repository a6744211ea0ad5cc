// common.cuh -- device helpers shared by the kernels of the MXFP4 routed
// expert linear (problem statement "MXFP4 Routed Expert Linear", Kimi K3).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace mxfp4el {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------- loads ----
// Packed weights are read exactly once per call: stream them past L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Token rows are re-read by every output row: keep the default caching.
__device__ __forceinline__ uint4 ld_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ------------------------------------------------------------ E2M1 codes ---
// One packed byte holds two E2M1 codes: input position 2j in the low nibble
// and 2j+1 in the high nibble ("What is stored in one group"). The hardware
// conversion turns the low nibble into the low half of an f16x2 and the high
// nibble into the high half; every E2M1 value is exact in f16 and in f32.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t word, uint32_t (&h)[4]) {
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(word));
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
  float2 r;
  asm("{\n"
      " .reg .f16 lo, hi;\n"
      " mov.b32 {lo, hi}, %2;\n"
      " cvt.f32.f16 %0, lo;\n"
      " cvt.f32.f16 %1, hi;\n"
      "}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(h));
  return r;
}

// d = a * b + c on two float32 lanes at once (Blackwell packed FMA).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n"
      " .reg .b64 ra, rb, rc, rd;\n"
      " mov.b64 ra, {%2, %3};\n"
      " mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n"
      " mov.b64 {%0, %1}, rd;\n"
      "}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// a * b on two float32 lanes at once.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n"
      " .reg .b64 ra, rb, rd;\n"
      " mov.b64 ra, {%2, %3};\n"
      " mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n"
      "}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// ------------------------------------------------------------ E8M0 scale ---
// The group factor 2^(s-127) ("Apply the shared group scale"), applied to a
// float32 partial sum so that the product is exact for every byte s:
// s = 1..254 is the normal float 2^(s-127); s = 0 is the subnormal 2^-127;
// s = 255 (2^128, beyond float32) is applied as 2^127 after doubling the
// partial. The caller multiplies the partial by `pre` and then by `factor`.
struct E8M0 {
  float factor;
  float pre;
};

__device__ __forceinline__ E8M0 e8m0(uint32_t s) {
  E8M0 r;
  r.factor = __uint_as_float(min(s, 254u) << 23);
  r.pre = 1.0f;
  if (s == 0u) r.factor = __uint_as_float(0x00400000u);   // 2^-127
  if (s == 255u) r.pre = 2.0f;
  return r;
}

// The same factor as two normal float32 powers of two whose product is
// 2^(s-127) for every byte s: 2^(floor(s/2) - 63) * 2^(ceil(s/2) - 64).
// Multiplying a partial by both in turn is exact (barring overflow or
// underflow of the product itself) and needs no case analysis.
__device__ __forceinline__ float2 e8m0_split(uint32_t s) {
  const uint32_t lo = s >> 1, hi = s - lo;
  return make_float2(__uint_as_float((lo + 64u) << 23), __uint_as_float((hi + 63u) << 23));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// ------------------------------------------------------------- tokens ------
template <typename Tok> struct TokenIO;

template <> struct TokenIO<float> {
  // 32 consecutive token values (one group) as float32.
  static __device__ __forceinline__ void load32(const float* p, float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 v = ld_u4(p + 4 * q);
      x[4 * q + 0] = __uint_as_float(v.x);
      x[4 * q + 1] = __uint_as_float(v.y);
      x[4 * q + 2] = __uint_as_float(v.z);
      x[4 * q + 3] = __uint_as_float(v.w);
    }
  }
  static __device__ __forceinline__ float to_f32(float v) { return v; }
  static __device__ __forceinline__ float from_f32(float v) { return v; }
};

template <> struct TokenIO<__nv_bfloat16> {
  // bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits.
  static __device__ __forceinline__ void load32(const __nv_bfloat16* p, float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 v = ld_u4(p + 8 * q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        x[8 * q + 2 * m + 0] = __uint_as_float(w[m] << 16);
        x[8 * q + 2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
      }
    }
  }
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// ------------------------------------------------------ f16 arithmetic ----
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ------------------------------------------- mbarriers and bulk copies -----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait on another warp or on a copy gives up after this long; the
// kernel then records the timeout and returns instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Waits until the mbarrier phase with `parity` has completed. Returns false
// if that did not happen within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// mbar_wait by a whole warp: every lane waits, then the lanes vote, so the
// result is the same in every lane and the warp is converged on return (as
// the .sync.aligned tcgen05 instructions that often follow require: lanes
// leave a spin loop at different times and need not reconverge by
// themselves before the next instruction).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}

// As mbar_wait, but each test may suspend the thread in hardware until the
// phase completes (or about 20 us pass) instead of spinning on issue slots
// that other warps of the SM need.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_suspend(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Asks the TMA engine to bring `bytes` (a multiple of 16) at the 16-byte
// aligned `src` into L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One contiguous global -> shared copy on the TMA engine; completion is
// signalled on `bar` as `bytes` transaction bytes. Both addresses must be
// 16-byte aligned and `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Orders this thread's earlier shared-memory accesses through the generic
// proxy (ordinary loads and stores) before later accesses through the async
// proxy (TMA and bulk copies, tensor-core operand reads). A consumer that read
// a staging buffer with ordinary loads calls it before it releases the buffer
// to a producer that refills it by copy: the release alone does not order the
// two proxies, and a refill can then overwrite bytes that a load still in
// flight reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy for data read exactly once (the packed weights and scales).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------ tensor memory (tcgen05) --
// TMEM addresses: bits 31..16 lane, bits 15..0 column (32-bit cells).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] x B[smem], one instruction of the current kind::f16 shape.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// This thread's TMEM lane, 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------- TMA tensor loads --
// 2D tiled load of a box at element coordinates (x innermost, y); x times
// the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same for a 3-D tensor map: box origin (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialization may start while
// its predecessor in the stream is still running; pdl_wait() blocks until
// the predecessor has completed and its memory is visible. Both are no-ops
// for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------- token prep -----
// Prepared bf16 tokens: per token t a power of two 2^sigma_t and
// x16[t, i] = f16(x[t, i] 2^sigma_t). One warp per token: sigma_t from
// max|x_t|, then x16[t] = f16(x_t 2^sigma_t) with max|x_t| 2^sigma_t in
// [2^top, 2^(top+1)): top = 8 for the GEMV, whose f16 partial sums of 8
// products must not overflow, and 14 for the tensor cores, which only need
// the operands themselves in range. A bf16 value keeps its 8 significant
// bits in f16 wherever the scaled value is a normal f16 number.
__device__ __forceinline__ void prep_token(const __nv_bfloat16* __restrict__ x,
                                           __half* __restrict__ x16,
                                           int* __restrict__ sigma, int t, int I, int lane,
                                           int top = 8) {
  const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * I);
  const int nvec = I / 8;
  uint32_t m = 0;                                // max |x| as float32 bits
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
  const int ex = (int)(m >> 23);                 // biased exponent of max|x|
  int s = 0;
  if (m != 0 && ex < 255) s = min(126, 127 + top - ex);   // max|x| 2^s in [2^top, 2^(top+1))
  const float up = __uint_as_float((uint32_t)(s + 127) << 23);
  uint4* out = reinterpret_cast<uint4*>(x16 + (size_t)t * I);
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
    out[i] = make_uint4(h[0], h[1], h[2], h[3]);
  }
  if (lane == 0) sigma[t] = s;
}

// ------------------------------------------------------ warp reductions ----
// Sums V = 2^L values over the 32 lanes of a warp with 2^L - 1 + (5 - L)
// shuffles instead of 5 V: each level hands half of the remaining values to
// the partner lane. On return every lane holds the full sum of value index
// (lane >> (5 - L)) & (V - 1).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be 2^L <= 32");
  int off = 16;
#pragma unroll
  for (int half = V / 2; half >= 1; half /= 2, off /= 2) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
    }
  }
#pragma unroll
  for (; off >= 1; off /= 2) v[0] += __shfl_xor_sync(kFullMask, v[0], off);
  return v[0];
}

}  // namespace mxfp4el
