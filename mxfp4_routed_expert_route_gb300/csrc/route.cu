// route.cu -- the routing bucketer.
//
// Groups the T*K (token, slot) pairs by selected expert so that every expert
// some token picked is read once, for all of its tokens, and no other expert
// is read at all ("Decode only selected experts", problem statement "MXFP4
// Routed Expert Linear", Kimi K3). It is a stable counting sort in one CTA:
//   A. each warp owns a contiguous chunk of pairs and counts, per expert, the
//      pairs of its chunk (warp-local counters, no atomics);
//   B. per-expert totals, an exclusive prefix sum over experts (segment
//      offsets), the compact ascending list of experts with at least one pair,
//      and each warp's starting position inside every expert segment;
//   C. each warp walks its chunk again and scatters pair ids into place.
// Inside a segment the pairs keep their (token, slot) order. Pairs whose
// expert id lies outside [0, E) are skipped and counted on the device.
// Large batches (at least 8192 pairs) run the same sort over many CTAs in
// three kernels (count, scan, scatter); small ones keep the single launch.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxfp4el {

// Status words of this device: counts the host reads and resets.
__device__ unsigned long long g_status[kStatusWords];

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Exclusive block-wide prefix sum of one int per thread; returns the prefix
// and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(kFullMask, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) warp_buf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_buf[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(kFullMask, wi, off);
      if (lane >= off) wi += n;
    }
    warp_buf[lane] = wi - w;          // exclusive prefix of warp totals
    if (lane == 31) warp_buf[32] = wi;
  }
  __syncthreads();
  const int r = warp_buf[warp] + incl - v;
  *total = warp_buf[32];
  __syncthreads();
  return r;
}

// Cost-balanced GEMV split, by the whole block after the counts and the
// active list are known. The calling thread owns experts [e0, e1), whose
// active ones are the consecutive active slots act0, act0+1, ...; their cost
// prefix comes from one more scan. Every CTA boundary b < ctas lies in
// exactly one expert's cost interval, and that expert's thread writes it.
__device__ void write_unit_split(const RoutePlan& plan, const UnitSplit& split, int e0, int e1,
                                 int act0, int total_active, int* warp_buf) {
  if (split.ctas <= 0) return;
  int my_cost = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = plan.counts[e];
    if (c > 0) my_cost += split.fixed_cost + c;
  }
  int total_cost;
  int cost = block_exclusive_scan(my_cost, warp_buf, &total_cost);
  const int64_t rt = split.row_tiles, n = split.ctas;
  const int64_t C = rt * (int64_t)total_cost;        // total cost of all units
  if (C == 0) {
    for (int b = threadIdx.x; b <= split.ctas; b += blockDim.x) plan.unit_begin[b] = 0;
    return;
  }
  // Boundary b of n (b = n: the pool's start) sits at cost b*S*C/N with
  // S = static_permille and N = 1000 n.
  const int64_t S = split.static_permille, N = 1000 * n;
  int slot = act0;
  for (int e = e0; e < e1; ++e) {
    const int c = plan.counts[e];
    if (c == 0) continue;
    const int64_t cu = split.fixed_cost + c;
    const int64_t lo = rt * cost, hi = rt * (cost + cu);   // [lo, hi) in cost units
    // Boundaries b with b*S*C/N in [lo, hi).
    for (int64_t b = (lo * N + S * C - 1) / (S * C); b <= n && b * S * C < hi * N; ++b) {
      const int64_t tile = (b * S * C - lo * N + N * cu - 1) / (N * cu);
      plan.unit_begin[b] = (int)(slot * rt + tile);
    }
    cost += (int)cu;
    ++slot;
  }
  // With S = 1000 boundary n is the end of the last expert's units.
  if (threadIdx.x == 0 && S >= 1000)
    plan.unit_begin[split.ctas] = (int)((int64_t)total_active * rt);
}

template <typename Idx>
__global__ void __launch_bounds__(kRouteThreads, 1)
route_kernel(const Idx* __restrict__ sel, int64_t P, int E, int* wc_global,
             RoutePlan plan, int T, TokenPrep prep, UnitSplit split) {
  pdl_launch_dependents();
  extern __shared__ int smem_wc[];
  __shared__ int warp_buf[33];
  int* wc = wc_global != nullptr ? wc_global : smem_wc;   // [warp][expert]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lanes_below = (1u << lane) - 1u;

  for (int i = threadIdx.x; i < kRouteWarps * E; i += kRouteThreads) wc[i] = 0;
  __syncthreads();

  const int64_t chunk = (P + kRouteWarps - 1) / kRouteWarps;
  const int64_t pbeg = min(P, (int64_t)warp * chunk);
  const int64_t pend = min(P, pbeg + chunk);
  int* my_wc = wc + (size_t)warp * E;

  // A. per-warp counts.
  int bad = 0;
  for (int64_t base = pbeg; base < pend; base += 32) {
    const int64_t i = base + lane;
    const bool in = i < pend;
    const long long e = in ? (long long)sel[i] : -1;
    const bool valid = in && e >= 0 && e < E;
    bad += (in && !valid) ? 1 : 0;
    const unsigned peers = __match_any_sync(kFullMask, valid ? (int)e : -1);
    if (valid && (peers & lanes_below) == 0) my_wc[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();

  // B. totals, offsets, active list, per-warp segment starts.
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
  int my_pairs = 0, my_active = 0;
  for (int e = e0; e < e1; ++e) {
    int c = 0;
    for (int w = 0; w < kRouteWarps; ++w) c += wc[w * E + e];
    plan.counts[e] = c;
    my_pairs += c;
    my_active += c > 0 ? 1 : 0;
  }
  int total_pairs, total_active;
  int off = block_exclusive_scan(my_pairs, warp_buf, &total_pairs);
  int act = block_exclusive_scan(my_active, warp_buf, &total_active);
  const int act0 = act;
  for (int e = e0; e < e1; ++e) {
    const int c = plan.counts[e];
    plan.offsets[e] = off;
    if (c > 0) plan.active[act++] = e;
    int run = off;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int cw = wc[w * E + e];
      wc[w * E + e] = run;
      run += cw;
    }
    off += c;
  }
  if (threadIdx.x == 0) {
    plan.offsets[E] = total_pairs;
    plan.meta[kMetaNumActive] = total_active;
    plan.meta[kMetaNumPairs] = total_pairs;
  }

  // B'. Cost-balanced GEMV split.
  write_unit_split(plan, split, e0, e1, act0, total_active, warp_buf);
  __syncthreads();

  // C. stable scatter of pair ids.
  for (int64_t base = pbeg; base < pend; base += 32) {
    const int64_t i = base + lane;
    const bool in = i < pend;
    const long long e = in ? (long long)sel[i] : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(kFullMask, valid ? (int)e : -1);
    int start = 0;
    if (valid) start = my_wc[e];
    __syncwarp();
    if (valid) {
      plan.pair_list[start + __popc(peers & lanes_below)] = (int)i;
      if ((peers & lanes_below) == 0) my_wc[e] = start + __popc(peers);
    }
    if (in && plan.pos_of_pair != nullptr)
      plan.pos_of_pair[i] = valid ? start + __popc(peers & lanes_below) : -1;
    __syncwarp();
  }

  // Invalid ids: count them for mxfp4el_device_errors().
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) bad += __shfl_xor_sync(kFullMask, bad, o);
  if (lane == 0 && bad > 0) atomicAdd(&g_status[kStatusBadPairs], (unsigned long long)bad);

  // Token prep for the staged GEMV, one warp per token.
  if (prep.x != nullptr)
    for (int t = warp; t < T; t += kRouteWarps)
      prep_token(static_cast<const __nv_bfloat16*>(prep.x), prep.x16, prep.sigma, t,
                 (int)prep.I, lane);
}

// ---------------------------------------------------------------------------
// Multi-CTA bucketer for many pairs: the same stable counting sort in three
// kernels. CTA c owns pairs [c*kMultiChunk, (c+1)*kMultiChunk), its warps
// contiguous sub-chunks of it.
//   count:   per-CTA, per-expert counts -> cta_counts[e][c]
//   scan:    one CTA: per-expert totals, exclusive prefix of cta_counts over
//            CTAs (each CTA's first position inside every expert segment),
//            offsets, active list, meta, GEMV split
//   scatter: each CTA counts its chunk again per warp and scatters pair ids
constexpr int kMultiThreads = 256;
constexpr int kMultiWarps = kMultiThreads / 32;
constexpr int kMultiChunk = 512;                 // pairs per CTA
constexpr int kMultiPerWarp = kMultiChunk / kMultiWarps;
constexpr int64_t kMultiMinPairs = 8192;         // below this one CTA is faster
constexpr int kMultiMaxExperts = 1024;           // per-warp counters in shared memory

// Per-warp counts of this CTA's chunk into wc[warp][E]; returns the warp's
// number of invalid ids.
template <typename Idx>
__device__ __forceinline__ int count_chunk(const Idx* __restrict__ sel, int64_t P, int E,
                                           int* wc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lanes_below = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < kMultiWarps * E; i += kMultiThreads) wc[i] = 0;
  __syncthreads();
  const int64_t pbeg = min(P, (int64_t)blockIdx.x * kMultiChunk + (int64_t)warp * kMultiPerWarp);
  const int64_t pend = min(P, pbeg + kMultiPerWarp);
  int* my_wc = wc + (size_t)warp * E;
  int bad = 0;
  for (int64_t base = pbeg; base < pend; base += 32) {
    const int64_t i = base + lane;
    const bool in = i < pend;
    const long long e = in ? (long long)sel[i] : -1;
    const bool valid = in && e >= 0 && e < E;
    bad += (in && !valid) ? 1 : 0;
    const unsigned peers = __match_any_sync(kFullMask, valid ? (int)e : -1);
    if (valid && (peers & lanes_below) == 0) my_wc[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  return bad;
}

template <typename Idx>
__global__ void __launch_bounds__(kMultiThreads)
route_count_kernel(const Idx* __restrict__ sel, int64_t P, int E, int* __restrict__ cta_counts) {
  pdl_launch_dependents();
  extern __shared__ int wc[];                    // [kMultiWarps][E]
  int bad = count_chunk(sel, P, E, wc);
  const int nctas = gridDim.x;
  for (int e = threadIdx.x; e < E; e += kMultiThreads) {
    int c = 0;
    for (int w = 0; w < kMultiWarps; ++w) c += wc[w * E + e];
    cta_counts[(size_t)e * nctas + blockIdx.x] = c;
  }
  // Invalid ids: count them for mxfp4el_device_errors().
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) bad += __shfl_xor_sync(kFullMask, bad, o);
  if ((threadIdx.x & 31) == 0 && bad > 0)
    atomicAdd(&g_status[kStatusBadPairs], (unsigned long long)bad);
}

__global__ void __launch_bounds__(kRouteThreads, 1)
route_scan_kernel(int* __restrict__ cta_counts, int nctas, int E, RoutePlan plan,
                  UnitSplit split) {
  pdl_launch_dependents();
  pdl_wait();                                    // the counts are complete
  __shared__ int warp_buf[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Per expert (one warp each): exclusive prefix over CTAs, in place. The
  // counts of 128 CTAs are loaded before any is scanned, so that a warp
  // waits for one load per 128 CTAs instead of one per 32.
  constexpr int kBatch = 4;
  for (int e = warp; e < E; e += kRouteWarps) {
    int* row = cta_counts + (size_t)e * nctas;
    int run = 0;
    for (int c0 = 0; c0 < nctas; c0 += 32 * kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = c0 + 32 * j + lane;
        v[j] = c < nctas ? row[c] : 0;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int c = c0 + 32 * j + lane;
        int incl = v[j];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int n = __shfl_up_sync(kFullMask, incl, off);
          if (lane >= off) incl += n;
        }
        if (c < nctas) row[c] = run + incl - v[j];
        run += __shfl_sync(kFullMask, incl, 31);
      }
    }
    if (lane == 0) plan.counts[e] = run;
  }
  __syncthreads();
  // Totals -> offsets, active list, meta (as phase B of route_kernel).
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
  int my_pairs = 0, my_active = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = plan.counts[e];
    my_pairs += c;
    my_active += c > 0 ? 1 : 0;
  }
  int total_pairs, total_active;
  int off = block_exclusive_scan(my_pairs, warp_buf, &total_pairs);
  int act = block_exclusive_scan(my_active, warp_buf, &total_active);
  const int act0 = act;
  for (int e = e0; e < e1; ++e) {
    const int c = plan.counts[e];
    plan.offsets[e] = off;
    if (c > 0) plan.active[act++] = e;
    off += c;
  }
  if (threadIdx.x == 0) {
    plan.offsets[E] = total_pairs;
    plan.meta[kMetaNumActive] = total_active;
    plan.meta[kMetaNumPairs] = total_pairs;
  }
  write_unit_split(plan, split, e0, e1, act0, total_active, warp_buf);
}

template <typename Idx>
__global__ void __launch_bounds__(kMultiThreads)
route_scatter_kernel(const Idx* __restrict__ sel, int64_t P, int E,
                     const int* __restrict__ cta_bases, RoutePlan plan) {
  pdl_launch_dependents();
  extern __shared__ int wc[];                    // [kMultiWarps][E]
  count_chunk(sel, P, E, wc);                    // reads only the ids
  pdl_wait();                                    // offsets and CTA bases are ready
  const int nctas = gridDim.x;
  for (int e = threadIdx.x; e < E; e += kMultiThreads) {
    int run = plan.offsets[e] + cta_bases[(size_t)e * nctas + blockIdx.x];
    for (int w = 0; w < kMultiWarps; ++w) {
      const int cw = wc[w * E + e];
      wc[w * E + e] = run;
      run += cw;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lanes_below = (1u << lane) - 1u;
  const int64_t pbeg = min(P, (int64_t)blockIdx.x * kMultiChunk + (int64_t)warp * kMultiPerWarp);
  const int64_t pend = min(P, pbeg + kMultiPerWarp);
  int* my_wc = wc + (size_t)warp * E;
  for (int64_t base = pbeg; base < pend; base += 32) {
    const int64_t i = base + lane;
    const bool in = i < pend;
    const long long e = in ? (long long)sel[i] : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(kFullMask, valid ? (int)e : -1);
    int start = 0;
    if (valid) start = my_wc[e];
    __syncwarp();
    if (valid) {
      plan.pair_list[start + __popc(peers & lanes_below)] = (int)i;
      if ((peers & lanes_below) == 0) my_wc[e] = start + __popc(peers);
    }
    if (in && plan.pos_of_pair != nullptr)
      plan.pos_of_pair[i] = valid ? start + __popc(peers & lanes_below) : -1;
    __syncwarp();
  }
}

int multi_ctas(int64_t P, int64_t E, bool prep) {
  if (prep || P < kMultiMinPairs || E == 0 || E > kMultiMaxExperts) return 0;
  const int64_t n = (P + kMultiChunk - 1) / kMultiChunk;
  return n <= 0x7fffffff ? (int)n : 0;
}

template <typename Idx>
cudaError_t launch_multi(const Idx* sel, int64_t P, int64_t E, int nctas, int* cta_counts,
                         const RoutePlan& plan, const UnitSplit& split, cudaStream_t stream) {
  const size_t smem = (size_t)kMultiWarps * E * sizeof(int);
  route_count_kernel<Idx><<<nctas, kMultiThreads, smem, stream>>>(sel, P, (int)E, cta_counts);
  note_launch();
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  err = launch_after_previous(route_scan_kernel, dim3(1), dim3(kRouteThreads), 0, stream,
                              cta_counts, nctas, (int)E, plan, split);
  if (err != cudaSuccess) return err;
  return launch_after_previous(route_scatter_kernel<Idx>, dim3((unsigned)nctas),
                               dim3(kMultiThreads), smem, stream, sel, P, (int)E,
                               static_cast<const int*>(cta_counts), plan);
}

}  // namespace

size_t route_global_counter_words(int64_t T, int64_t K, int64_t E, bool prep_in_route) {
  const int nctas = multi_ctas(T * K, E, prep_in_route);
  if (nctas > 0) return (size_t)nctas * (size_t)E;
  return kRouteWarps * (size_t)E * sizeof(int) > kRouteSmemLimit
             ? (size_t)kRouteWarps * (size_t)E : 0;
}

bool prep_fits_route(int64_t T, int64_t I) { return T <= 64 && T * I <= ((int64_t)1 << 20); }

cudaError_t launch_route(const void* sel, int index_dtype, int64_t T, int64_t K,
                         int64_t E, int* wc_global, const RoutePlan& plan,
                         const TokenPrep& prep, const UnitSplit& split, cudaStream_t stream) {
  const int64_t P = T * K;
  const int nctas = multi_ctas(P, E, prep.x != nullptr);
  if (nctas > 0) {
    if (index_dtype == kIndexI64)
      return launch_multi(static_cast<const int64_t*>(sel), P, E, nctas, wc_global, plan, split,
                          stream);
    return launch_multi(static_cast<const int32_t*>(sel), P, E, nctas, wc_global, plan, split,
                        stream);
  }
  const size_t smem = wc_global ? 0 : kRouteWarps * (size_t)E * sizeof(int);
  // Dynamic plus static shared memory above 48 KiB needs the opt-in.
  if (smem > 40 * 1024) {
    cudaError_t err;
    if (index_dtype == kIndexI64)
      err = cudaFuncSetAttribute(route_kernel<int64_t>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    else
      err = cudaFuncSetAttribute(route_kernel<int32_t>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  if (index_dtype == kIndexI64)
    route_kernel<int64_t><<<1, kRouteThreads, smem, stream>>>(
        static_cast<const int64_t*>(sel), P, (int)E, wc_global, plan, (int)T, prep, split);
  else
    route_kernel<int32_t><<<1, kRouteThreads, smem, stream>>>(
        static_cast<const int32_t*>(sel), P, (int)E, wc_global, plan, (int)T, prep, split);
  note_launch();
  return cudaGetLastError();
}

unsigned long long* device_status_words() {
  static std::mutex mu;
  static unsigned long long* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned long long*>(p);
  }
  return addr[dev];
}

cudaError_t read_and_reset_status(cudaStream_t stream, int word, int64_t* out) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  unsigned long long v = 0;
  const size_t off = (size_t)word * sizeof(unsigned long long);
  err = cudaMemcpyFromSymbol(&v, g_status, sizeof(v), off);
  if (err != cudaSuccess) return err;
  const unsigned long long zero = 0;
  err = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero), off);
  *out = (int64_t)v;
  return err;
}

}  // namespace mxfp4el
