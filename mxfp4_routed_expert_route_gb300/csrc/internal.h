// internal.h -- declarations shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace mxfp4el {

constexpr int kTokenF32 = 0;
constexpr int kTokenBF16 = 1;
constexpr int kIndexI32 = 0;
constexpr int kIndexI64 = 1;

// Per-warp expert counters live in shared memory up to this many bytes and
// in the workspace beyond it.
constexpr size_t kRouteSmemLimit = 96 * 1024;

// Device status words (one array per device, see device_status_words()).
constexpr int kStatusBadPairs = 0;      // (t, k) pairs with an out-of-range id
constexpr int kStatusWaitTimeouts = 1;  // kernel waits that hit their time limit
constexpr int kStatusWords = 4;

// Slots of RoutePlan::meta.
constexpr int kMetaNumActive = 0;   // experts with at least one valid pair
constexpr int kMetaNumPairs = 1;    // valid pairs
constexpr int kMetaUnitCounter = 2; // next unit of the tensor-core kernel (reset by the gather)
constexpr int kMetaPoolCounter = 3; // next pool unit of the staged GEMV (reset by the GEMV)
constexpr int kMetaUnitCounter2 = 4; // next unit of a second tensor-core kernel on the same
                                     // lists (the SwiGLU down projection; reset by the gather)
constexpr int kMetaWords = 64;

// Routing lists written by the bucketer, all in device memory.
struct RoutePlan {
  int* meta;        // [kMetaWords]
  int* counts;      // [E]     pairs per expert
  int* offsets;     // [E + 1] start of each expert's segment in pair_list
  int* active;      // [E]     ascending ids of experts with count > 0
  int* pair_list;   // [T*K]   pair ids t*K + k grouped by expert, stable
  int* pos_of_pair; // [T*K] or null: each pair's position in pair_list, -1 for an
                    // out-of-range id (written by the bucketer when not null)
  int* unit_begin;  // [kMaxSplitCtas + 1] first GEMV unit of each CTA, when
                    // the bucketer was asked for a cost-balanced split
};

// Cost-balanced split of the staged GEMV's units (active expert, row tile)
// over its CTAs, computed by the bucketer: unit (u, tile) costs
// fixed_cost + (tokens of expert u), CTA b starts at the first unit whose
// cost prefix reaches b * static_permille / (1000 ctas) of the total; entry
// ctas is the first unit of the pool that the CTAs share after their own
// ranges. With equal unit counts per CTA, the CTAs that drew experts with
// several tokens finished last and the others idled. ctas == 0: no split.
constexpr int kMaxSplitCtas = 1024;
struct UnitSplit {
  int ctas;
  int row_tiles;
  int fixed_cost;
  int static_permille;
};

// Workspace layout for one call.
struct Workspace {
  RoutePlan plan;
  int* wc_global;   // per-warp counters when they do not fit in shared memory
  __half* x16;      // [T, I] tokens scaled by 2^sigma_t in f16 (staged GEMV, bf16 tokens)
  int* sigma;       // [T] the power of two of each token (staged GEMV, bf16 tokens)
  __half* grouped;  // [T*K, I] f16 token rows grouped by expert (tensor-core path)
  int* gsigma;      // [T*K] the power of two of each grouped row
  uint8_t* tile_mode;  // [E][row tiles] operand mode of each tile (tensor-core path)
  int16_t* row_off;    // [E*O] row offsets (tensor-core path)
  float* part;      // [T*K, ncol, O] float32 partial results of every pair
  size_t bytes;     // total
};

// Offsets of every region for the given sizes; base == nullptr only sizes.
// with_part = false: no partial-result buffer (ws->part = nullptr), for a
// linear whose kernel writes something else (gate/up tiles).
// tiles_F > 0: the tensor-core path runs gate/up tiles of F gate rows (the
// tile modes then cover 64-row halves).
bool carve_workspace(void* base, int64_t T, int64_t E, int64_t I, int64_t O,
                     int64_t K, int token_dtype, Workspace* ws, bool with_part = true,
                     int64_t tiles_F = 0, bool prepared = false);

// Partial results per (pair, row) that the chosen linear kernel writes.
int linear_partial_columns(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                           int token_dtype);

// Workspace words the bucketer needs for its counters: per-warp counters
// when they do not fit in shared memory (single CTA), or per-CTA counts
// (many pairs, several CTAs). prep_in_route: the bucketer also prepares
// the tokens (then it runs as one CTA).
size_t route_global_counter_words(int64_t T, int64_t K, int64_t E, bool prep_in_route);

// Tokens prepared for the staged GEMV (bf16 tokens): x16 = f16(x 2^sigma).
struct TokenPrep {
  const void* x;    // bf16 tokens (T, I), or nullptr: nothing to prepare
  __half* x16;
  int* sigma;
  int64_t I;
};

// Bucketer; also prepares the tokens in the same launch when `prep.x` is
// set, and writes plan.unit_begin when `split.ctas` > 0.
cudaError_t launch_route(const void* sel, int index_dtype, int64_t T,
                         int64_t K, int64_t E, int* wc_global,
                         const RoutePlan& plan, const TokenPrep& prep,
                         const UnitSplit& split, cudaStream_t stream);

// True when token prep for these sizes fits in the bucketer's launch.
bool prep_fits_route(int64_t T, int64_t I);


// True when the rows of width I fit the staged (bulk-copy) GEMV; bf16
// tokens then need launch_prep_tokens first.
bool gemv_uses_stream(int64_t I, bool prep = false);

// The split the staged GEMV wants for these sizes (ctas == 0: none, the
// kernel then splits its units evenly).
UnitSplit gemv_unit_split(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                          bool prep = false);

// Partial results per (pair, output row) that the GEMV writes for width I:
// one per group column of the staged kernel, 1 for the direct kernel. The
// combine adds them in column order.
int gemv_partial_columns(int64_t I);

cudaError_t launch_prep_tokens(const void* x, __half* x16, int* sigma, int64_t T,
                               int64_t I, cudaStream_t stream);

// True when the staged GEMV routes for itself: few enough pairs that each
// CTA derives the routing lists and token scales it needs from the ids, and
// neither the bucketer nor the token prep runs.
bool gemv_self_route(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                     bool prep = false);

struct PreparedView;
// prep: the weights as prepared blocks (packed and scales unused), or null.
cudaError_t launch_gemv(const void* x, int token_dtype, const __half* x16,
                        const int* sigma, const void* sel, int index_dtype,
                        const uint8_t* packed, const uint8_t* scales,
                        const RoutePlan& plan, float* part,
                        unsigned long long* status, int64_t T, int64_t E,
                        int64_t I, int64_t O, int64_t K, cudaStream_t stream,
                        const PreparedView* prep = nullptr);

// Prefill-regime grouped GEMM on the tensor cores (bf16 tokens).
bool gemm_tc_supported(int64_t E, int64_t I, int64_t O);

// Gate/up tiles for the SwiGLU expert (F > 0): the tensor-core kernel runs
// the stacked gate/up projection (O = 2F rows, gate rows first) in tiles of
// 64 gate rows plus the matching 64 up rows and writes h = silu(gate) * up
// (bf16, (P, F)) and each pair's expert (sel2) instead of partial results.
struct SwigluTiles {
  int64_t F = 0;
  void* h = nullptr;
  int32_t* sel2 = nullptr;   // or nullptr: not needed
  bool grouped = false;      // h rows in the lists' (expert-grouped) order, not by pair
};
bool gemm_tc_swiglu_supported(int64_t E, int64_t I, int64_t F);

// The B operand rows of the tensor-core kernel, in the routing lists'
// (expert-grouped) order: f16 copies scaled per row by 2^sigma
// (launch_group_tokens; tiles may then take the f16 operand mode), or plain
// bf16 rows (every tile takes the bf16 mode).
struct TcTokens {
  const void* rows = nullptr;     // [nrows, I]
  const int* sigma = nullptr;     // [nrows] (f16 rows)
  bool f16 = false;
  int64_t nrows = 0;
};
size_t gemm_tc_grouped_bytes(int64_t T, int64_t K, int64_t I);

// xg[p] = f16(x[t] 2^sigma) for t = pair_list[p] / K (max |x_t| 2^sigma in
// [2^14, 2^15)), sigma[p] its power of two, one warp per token through
// plan.pos_of_pair (required: cudaErrorInvalidValue without it); also resets
// the tensor-core kernel's unit counters; zero_ids (T*K ints) or nullptr:
// also set to 0 (gate/up tiles).
cudaError_t launch_group_tokens(const void* x, const RoutePlan& plan, __half* xg, int* sigma,
                                int64_t T, int64_t I, int64_t K, int32_t* zero_ids,
                                cudaStream_t stream);
// Operand modes of the tensor-core kernel's row tiles (launch_tile_scan):
// tile_mode [E][gemm_tc_row_tiles(O, F)] (1: f16 operands hold every weight
// of the tile exactly) and row_off [E*O] (each weight row's offset r). With
// null pointers every tile takes the bf16 mode.
struct TcTileModes {
  const uint8_t* tile_mode = nullptr;
  const int16_t* row_off = nullptr;
};
int64_t gemm_tc_row_tiles(int64_t O, int64_t F);
cudaError_t launch_tile_scan(const uint8_t* scales, int64_t E, int64_t I, int64_t O, int64_t F,
                             uint8_t* tile_mode, int16_t* row_off, cudaStream_t stream);
cudaError_t launch_gemm_tc(const TcTokens& tokens, const TcTileModes& modes, const uint8_t* packed,
                           const uint8_t* scales, const RoutePlan& plan, float* part,
                           unsigned long long* status, int64_t E, int64_t I, int64_t O,
                           int64_t K, const SwigluTiles& swiglu, cudaStream_t stream,
                           int counter_word = kMetaUnitCounter,
                           const uint8_t* prepared = nullptr);

// Prepared weights (prepare.cu): one block per (expert, 128-row tile, 64-wide
// K chunk) of the chunk's packed bytes (32 per row, 16-byte halves swapped
// when bit 2 of the row is set) and then its scale bytes (2 per row); after
// the blocks, the tensor-core kernel's f16 row offsets and tile modes.
constexpr int kPrepRows = 128;
constexpr uint32_t kPrepPackedBytes = kPrepRows * 32;
constexpr uint32_t kPrepBlockBytes = kPrepPackedBytes + 2 * kPrepRows;
struct PreparedView {
  const unsigned char* blocks = nullptr;   // [E][ceil(O/128)][ceil(G/2)] blocks
  const int16_t* row_off = nullptr;        // [E][O]
  const uint8_t* tile_mode = nullptr;      // [E][ceil(O/128)]
};
size_t prepared_bytes(int64_t E, int64_t I, int64_t O);
PreparedView prepared_view(const void* base, int64_t E, int64_t I, int64_t O);
cudaError_t launch_prepare(const uint8_t* packed, const uint8_t* scales, int64_t E, int64_t I,
                           int64_t O, void* prepared, cudaStream_t stream);
// cuTensorMapEncodeTiled from the driver (PFN_cuTensorMapEncodeTiled_v12000),
// or null.
void* tensor_map_encoder();
// Whether the per-tile scan of f16 operand modes handles rows of width I.
bool tile_scan_fits(int64_t I);

// Argument checks shared by every routed-linear entry point (api.cu):
// MXFP4EL_OK or the first error, in the order the public header documents.
int validate_linear(const void* x, const uint8_t* packed, const uint8_t* scales,
                    const void* sel, const float* p, const void* ys, void* out,
                    int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                    int token_dtype, int index_dtype);

// Which kernel computes the routed linear for these sizes.
enum class LinearPath { kGemv, kGemm };
LinearPath choose_path(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, int token_dtype);

// after_linear: the previous kernel on `stream` is the library's linear
// kernel (which releases its dependents only after everything before it has
// finished); the combine then reads y_shared, the ids and the weights before
// waiting for the partial results.
cudaError_t launch_combine(const void* y_shared, const void* sel,
                           int index_dtype, const float* p, const float* part,
                           int ncol, void* out, int token_dtype, int64_t T,
                           int64_t E, int64_t O, int64_t K, bool after_linear,
                           cudaStream_t stream);

// Sigmoid top-K router (router.cu): one warp per token, the warp's raw,
// choice and chosen scores in shared memory.
constexpr int kRouterThreads = 256;
constexpr int64_t kRouterSmemLimit = 48 * 1024;
// Warps per block whose shared memory fits (0: 2E + K too large).
int router_warps_per_block(int64_t E, int64_t K);
cudaError_t launch_router(const float* logits, const float* bias, int64_t T, int64_t E,
                          int64_t K, float scaling, int32_t* sel, float* p,
                          cudaStream_t stream);

// SwiGLU between the two projections of the SwiGLU expert (swiglu.cu): from
// the gate/up projection's partial results `part` (P pairs x ncol columns x
// 2F rows, gate rows first) h[pair, f] = silu(gate) * up in float32, rounded
// to the token dtype, and sel2[pair] = the pair's expert, or 0 (with h = 0)
// for an id outside [0, E).
cudaError_t launch_swiglu(const float* part, int ncol, const void* sel, int index_dtype,
                          int64_t E, int64_t P, int64_t F, int token_dtype, void* h,
                          int32_t* sel2, cudaStream_t stream);

// Device address of the status words on the current device.
unsigned long long* device_status_words();

// Synchronises `stream`, reads one status word and resets it to zero.
cudaError_t read_and_reset_status(cudaStream_t stream, int word, int64_t* out);

// Counts kernel launches made by the library (process-wide).
void note_launch();

// Launches `kernel` so that it may start before the previous kernel on
// `stream` finishes (programmatic stream serialization); the kernel must call
// pdl_wait() before it reads anything that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace mxfp4el
