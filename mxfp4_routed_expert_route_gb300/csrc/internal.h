// internal.h -- declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxfp4el {

constexpr int kTokenF32 = 0;
constexpr int kTokenBF16 = 1;
constexpr int kIndexI32 = 0;
constexpr int kIndexI64 = 1;

// Per-warp expert counters live in shared memory up to this many bytes and
// in the workspace beyond it.
constexpr size_t kRouteSmemLimit = 96 * 1024;

// Slots of RoutePlan::meta.
constexpr int kMetaNumActive = 0;   // experts with at least one valid pair
constexpr int kMetaNumPairs = 1;    // valid pairs
constexpr int kMetaWords = 64;

// Routing lists written by the bucketer, all in device memory.
struct RoutePlan {
  int* meta;        // [kMetaWords]
  int* counts;      // [E]     pairs per expert
  int* offsets;     // [E + 1] start of each expert's segment in pair_list
  int* active;      // [E]     ascending ids of experts with count > 0
  int* pair_list;   // [T*K]   pair ids t*K + k grouped by expert, stable
};

// Workspace layout for one call.
struct Workspace {
  RoutePlan plan;
  int* wc_global;   // per-warp counters when they do not fit in shared memory
  float* part;      // [T*K, O] float32 routed result of every pair
  size_t bytes;     // total
};

// Offsets of every region for the given sizes; base == nullptr only sizes.
bool carve_workspace(void* base, int64_t T, int64_t E, int64_t O, int64_t K,
                     Workspace* ws);

size_t route_global_counter_words(int64_t E);

cudaError_t launch_route(const void* sel, int index_dtype, int64_t T,
                         int64_t K, int64_t E, int* wc_global,
                         const RoutePlan& plan, cudaStream_t stream);

cudaError_t launch_gemv(const void* x, int token_dtype, const uint8_t* packed,
                        const uint8_t* scales, const RoutePlan& plan,
                        float* part, int64_t T, int64_t E, int64_t I,
                        int64_t O, int64_t K, cudaStream_t stream);

cudaError_t launch_combine(const void* y_shared, const void* sel,
                           int index_dtype, const float* p, const float* part,
                           void* out, int token_dtype, int64_t T, int64_t E,
                           int64_t O, int64_t K, cudaStream_t stream);

cudaError_t read_and_reset_bad_pairs(cudaStream_t stream, int64_t* out);

// Counts kernel launches made by the library (process-wide).
void note_launch();

}  // namespace mxfp4el
