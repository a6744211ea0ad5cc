// api.cu -- the C ABI (include/mxfp4_expert_linear.h): argument checks,
// workspace, and the launch sequences on one stream: route -> linear (GEMV or
// GEMM) -> combine; router -> that; and for the SwiGLU expert gate/up linear
// -> SwiGLU -> down linear -> combine.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/mxfp4_expert_linear.h"
#include "internal.h"

namespace mxfp4el {
namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kMaxPairs = (int64_t)1 << 30;       // pair ids are int32
constexpr int64_t kMaxDim = ((int64_t)1 << 31) - 1;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool sizes_ok(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K) {
  if (T > kMaxDim || E > kMaxDim || I > kMaxDim || O > kMaxDim || K > kMaxDim)
    return false;
  if (K > 0 && T > kMaxPairs / K) return false;
  const int64_t P = T * K;
  if (O > 0 && P > (((int64_t)1 << 62) / 4) / O) return false;
  return true;
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  if (an == 0 || bn == 0 || a == nullptr || b == nullptr) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

std::atomic<int64_t> g_launches{0};

struct StageEvents {
  cudaEvent_t start = nullptr, end = nullptr;
};
StageEvents g_stage[MXFP4EL_NUM_STAGES];

void mark(int stage, bool begin, cudaStream_t stream) {
  const cudaEvent_t ev = begin ? g_stage[stage].start : g_stage[stage].end;
  if (ev != nullptr) cudaEventRecord(ev, stream);
}

}  // namespace

// Argument checks of every routed-linear entry point, in the order the
// header documents; returns MXFP4EL_OK or the first error found.
int validate_linear(const void* x, const uint8_t* packed, const uint8_t* scales,
             const void* sel, const float* p, const void* ys, void* out,
             int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
             int token_dtype, int index_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (index_dtype != MXFP4EL_INDEX_I32 && index_dtype != MXFP4EL_INDEX_I64)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (!sizes_ok(T, E, I, O, K)) return MXFP4EL_ERR_TOO_LARGE;
  if (T == 0 || O == 0) return MXFP4EL_OK;
  if (ys == nullptr || out == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && (x == nullptr || sel == nullptr || p == nullptr))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && E > 0 && (packed == nullptr || scales == nullptr))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  // 128-bit loads of tokens and packed groups need 16-byte aligned bases.
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(packed)) % 16)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  const size_t tb = token_dtype == MXFP4EL_DTYPE_BF16 ? 2 : 4;
  const size_t ib = index_dtype == MXFP4EL_INDEX_I64 ? 8 : 4;
  const size_t G = (size_t)I / 32;
  const size_t out_bytes = (size_t)T * O * tb;
  const void* inputs[] = {x, packed, scales, sel, p, ys};
  const size_t sizes[] = {(size_t)T * I * tb, (size_t)E * O * G * 16,
                          (size_t)E * O * G, (size_t)T * K * ib,
                          (size_t)T * K * 4, (size_t)T * O * tb};
  for (int i = 0; i < 6; ++i)
    if (overlaps(out, out_bytes, inputs[i], sizes[i])) return MXFP4EL_ERR_ALIAS;
  return MXFP4EL_OK;
}

// The same checks for the call on prepared weights: the prepared copy
// (mxfp4_expert_linear_prepared_bytes(E, I, O) bytes, 256-byte aligned) in
// place of the packed weights and scale bytes.
int validate_prepared(const void* x, const void* prepared, const void* sel, const float* p,
                      const void* ys, void* out, int64_t T, int64_t E, int64_t I, int64_t O,
                      int64_t K, int token_dtype, int index_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (index_dtype != MXFP4EL_INDEX_I32 && index_dtype != MXFP4EL_INDEX_I64)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (!sizes_ok(T, E, I, O, K) || !gemv_uses_stream(I, true)) return MXFP4EL_ERR_TOO_LARGE;
  if (T == 0 || O == 0) return MXFP4EL_OK;
  if (ys == nullptr || out == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && (x == nullptr || sel == nullptr || p == nullptr))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && E > 0 && prepared == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(prepared) % 256)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  const size_t tb = token_dtype == MXFP4EL_DTYPE_BF16 ? 2 : 4;
  const size_t ib = index_dtype == MXFP4EL_INDEX_I64 ? 8 : 4;
  const size_t out_bytes = (size_t)T * O * tb;
  const void* inputs[] = {x, prepared, sel, p, ys};
  const size_t sizes[] = {(size_t)T * I * tb, prepared_bytes(E, I, O), (size_t)T * K * ib,
                          (size_t)T * K * 4, (size_t)T * O * tb};
  for (int i = 0; i < 5; ++i)
    if (overlaps(out, out_bytes, inputs[i], sizes[i])) return MXFP4EL_ERR_ALIAS;
  return MXFP4EL_OK;
}

LinearPath choose_path(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, int token_dtype) {
  const bool tc_ok = token_dtype == MXFP4EL_DTYPE_BF16 && E > 0 && gemm_tc_supported(E, I, O);
  // Test knob: MXFP4EL_PATH=gemv or gemm forces a kernel where it applies.
  if (const char* env = std::getenv("MXFP4EL_PATH")) {
    if (std::strcmp(env, "gemv") == 0) return LinearPath::kGemv;
    if (std::strcmp(env, "gemm") == 0 && tc_ok) return LinearPath::kGemm;
  }
  if (!tc_ok) return LinearPath::kGemv;
  // Tensor cores pay off once experts average about 16 tokens: the GEMV's
  // CUDA-core work grows with the tokens per expert, the GEMM's MMA does not
  // until N passes 16.
  const int64_t P = T * K;
  const int64_t slots = std::max<int64_t>(1, std::min<int64_t>(E, P));
  return P >= 16 * slots ? LinearPath::kGemm : LinearPath::kGemv;
}

int linear_partial_columns(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                           int token_dtype) {
  return choose_path(T, E, I, O, K, token_dtype) == LinearPath::kGemm ? 1
                                                                       : gemv_partial_columns(I);
}

namespace {

// Route and linear for K > 0: the float32 partial results land in ws.part
// (linear_partial_columns() columns per pair).
// prep: the weights as prepared blocks (packed and scales then unused).
cudaError_t run_linear(const void* x, const uint8_t* packed, const uint8_t* scales,
                       const void* sel, int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                       int token_dtype, int index_dtype, const Workspace& ws,
                       cudaStream_t stream, const SwigluTiles& swiglu = SwigluTiles{},
                       const PreparedView* prep_w = nullptr) {
  unsigned long long* status = device_status_words();
  if (status == nullptr) return cudaErrorUnknown;
  if (E == 0) {
    // Every id is out of range: the bucketer counts them, nothing else runs.
    mark(MXFP4EL_STAGE_ROUTE, true, stream);
    const cudaError_t err = launch_route(sel, index_dtype, T, K, 0, ws.wc_global, ws.plan,
                                         TokenPrep{nullptr, nullptr, nullptr, I},
                                         UnitSplit{0, 0, 0, 1000}, stream);
    mark(MXFP4EL_STAGE_ROUTE, false, stream);
    return err;
  }
  const bool gemm = choose_path(T, E, I, O, K, token_dtype) == LinearPath::kGemm;
  // Small batches on the GEMV: each GEMV CTA routes for itself.
  const bool pw = prep_w != nullptr;
  const bool self = !gemm && gemv_self_route(T, E, I, O, K, pw);
  const bool prep =
      !gemm && !self && token_dtype == MXFP4EL_DTYPE_BF16 && gemv_uses_stream(I, pw);
  const bool prep_in_route = prep && prep_fits_route(T, I);
  TokenPrep tp = {prep_in_route ? x : nullptr, ws.x16, ws.sigma, I};
  const UnitSplit split = gemm ? UnitSplit{0, 0, 0, 1000} : gemv_unit_split(T, E, I, O, K, pw);
  mark(MXFP4EL_STAGE_ROUTE, true, stream);
  cudaError_t err = cudaSuccess;
  if (!self)
    err = launch_route(sel, index_dtype, T, K, E, ws.wc_global, ws.plan, tp, split, stream);
  if (err == cudaSuccess && prep && !prep_in_route)
    err = launch_prep_tokens(x, ws.x16, ws.sigma, T, I, stream);
  mark(MXFP4EL_STAGE_ROUTE, false, stream);
  if (err != cudaSuccess) return err;
  if (gemm) {
    mark(MXFP4EL_STAGE_GATHER, true, stream);
    // Prepared weights carry their tile modes and row offsets.
    if (!pw) err = launch_tile_scan(scales, E, I, O, swiglu.F, ws.tile_mode, ws.row_off, stream);
    if (err == cudaSuccess)
      err = launch_group_tokens(x, ws.plan, ws.grouped, ws.gsigma, T, I, K, swiglu.sel2, stream);
    mark(MXFP4EL_STAGE_GATHER, false, stream);
    if (err != cudaSuccess) return err;
  }
  mark(MXFP4EL_STAGE_LINEAR, true, stream);
  if (gemm) {
    TcTokens tok;
    tok.rows = ws.grouped;
    tok.sigma = ws.gsigma;
    tok.f16 = true;
    tok.nrows = T * K;
    TcTileModes modes;
    modes.tile_mode = pw ? prep_w->tile_mode : ws.tile_mode;
    modes.row_off = pw ? prep_w->row_off : ws.row_off;
    err = launch_gemm_tc(tok, modes, packed, scales, ws.plan, ws.part, status, E, I, O, K, swiglu,
                         stream, kMetaUnitCounter, pw ? prep_w->blocks : nullptr);
  } else
    err = launch_gemv(x, token_dtype, ws.x16, ws.sigma, sel, index_dtype, packed, scales,
                      ws.plan, ws.part, status, T, E, I, O, K, stream, prep_w);
  mark(MXFP4EL_STAGE_LINEAR, false, stream);
  return err;
}

int run(const void* x, const uint8_t* packed, const uint8_t* scales,
        const void* sel, const float* p, const void* ys, void* out, int64_t T,
        int64_t E, int64_t I, int64_t O, int64_t K, int token_dtype,
        int index_dtype, const Workspace& ws, cudaStream_t stream,
        const PreparedView* prep_w = nullptr) {
  if (K > 0 && run_linear(x, packed, scales, sel, T, E, I, O, K, token_dtype, index_dtype, ws,
                          stream, SwigluTiles{}, prep_w) != cudaSuccess)
    return MXFP4EL_ERR_CUDA;
  mark(MXFP4EL_STAGE_COMBINE, true, stream);
  // With K > 0 and E > 0 a linear kernel of the library ran just before
  // (the launchers skip only an empty grid, E == 0).
  const cudaError_t err =
      launch_combine(ys, sel, index_dtype, p, ws.part,
                     linear_partial_columns(T, E, I, O, K, token_dtype), out, token_dtype, T, E,
                     O, K, K > 0 && E > 0, stream);
  mark(MXFP4EL_STAGE_COMBINE, false, stream);
  return err == cudaSuccess ? MXFP4EL_OK : MXFP4EL_ERR_CUDA;
}

// The SwiGLU expert: gate/up projection (2F stacked rows) -> SwiGLU -> down
// projection with every pair as its own token -> combine.
int validate_swiglu(const void* x, const uint8_t* gu_packed, const uint8_t* gu_scales,
                    const uint8_t* dn_packed, const uint8_t* dn_scales, const void* sel,
                    const float* p, const void* ys, void* out, int64_t T, int64_t E,
                    int64_t I, int64_t F, int64_t O, int64_t K, int token_dtype,
                    int index_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (index_dtype != MXFP4EL_INDEX_I32 && index_dtype != MXFP4EL_INDEX_I64)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0 || F <= 0 || F % 32 != 0)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (F > kMaxDim / 2 || !sizes_ok(T, E, I, 2 * F, K) || !sizes_ok(T * K, E, F, O, 1))
    return MXFP4EL_ERR_TOO_LARGE;
  if (T == 0 || O == 0) return MXFP4EL_OK;
  if (ys == nullptr || out == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && (x == nullptr || sel == nullptr || p == nullptr))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (K > 0 && E > 0 &&
      (gu_packed == nullptr || gu_scales == nullptr || dn_packed == nullptr ||
       dn_scales == nullptr))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(gu_packed) |
       reinterpret_cast<uintptr_t>(dn_packed)) % 16)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  const size_t tb = token_dtype == MXFP4EL_DTYPE_BF16 ? 2 : 4;
  const size_t ib = index_dtype == MXFP4EL_INDEX_I64 ? 8 : 4;
  const size_t Gi = (size_t)I / 32, Gf = (size_t)F / 32;
  const size_t out_bytes = (size_t)T * O * tb;
  const void* inputs[] = {x, gu_packed, gu_scales, dn_packed, dn_scales, sel, p, ys};
  const size_t sizes[] = {(size_t)T * I * tb,        (size_t)E * 2 * F * Gi * 16,
                          (size_t)E * 2 * F * Gi,    (size_t)E * O * Gf * 16,
                          (size_t)E * O * Gf,        (size_t)T * K * ib,
                          (size_t)T * K * 4,         (size_t)T * O * tb};
  for (int i = 0; i < 8; ++i)
    if (overlaps(out, out_bytes, inputs[i], sizes[i])) return MXFP4EL_ERR_ALIAS;
  return MXFP4EL_OK;
}

// Whether the gate/up projection of a SwiGLU call runs on the tensor cores
// in gate/up tiles. Test knob: MXFP4EL_SWIGLU_TILES=0 keeps the separate
// SwiGLU kernel.
bool swiglu_tiles_used(int64_t T, int64_t E, int64_t I, int64_t F, int64_t K,
                       int token_dtype) {
  if (const char* env = std::getenv("MXFP4EL_SWIGLU_TILES"))
    if (std::strcmp(env, "0") == 0) return false;
  return choose_path(T, E, I, 2 * F, K, token_dtype) == LinearPath::kGemm &&
         gemm_tc_swiglu_supported(E, I, F);
}

// Whether the down projection of a SwiGLU call whose gate/up projection
// runs in gate/up tiles also runs on the tensor cores, on the gate/up lists.
bool down_reuses_lists(int64_t P, int64_t E, int64_t F, int64_t O, int token_dtype) {
  return choose_path(P, E, F, O, 1, token_dtype) == LinearPath::kGemm;
}

struct SwigluWorkspace {
  Workspace gate_up, down;   // the two projections' own workspaces
  void* h = nullptr;         // (P, F) token dtype
  int32_t* sel2 = nullptr;   // (P,) the down projection's expert per pair
  size_t bytes = 0;
};

void carve_swiglu(void* base, int64_t T, int64_t E, int64_t I, int64_t F, int64_t O,
                  int64_t K, int token_dtype, SwigluWorkspace* sw) {
  const int64_t P = T * K;
  const size_t tb = token_dtype == MXFP4EL_DTYPE_BF16 ? 2 : 4;
  auto at = [&](size_t off) { return base ? static_cast<char*>(base) + off : nullptr; };
  // Gate/up tiles write h directly: no partial results for that projection.
  const bool tiles = K > 0 && E > 0 && swiglu_tiles_used(T, E, I, F, K, token_dtype);
  carve_workspace(base, T, E, I, 2 * F, K, token_dtype, &sw->gate_up, !tiles, tiles ? F : 0);
  size_t off = align_up(sw->gate_up.bytes);
  carve_workspace(at(off), P, E, F, O, 1, token_dtype, &sw->down);
  off = align_up(off + sw->down.bytes);
  sw->h = at(off);
  off = align_up(off + (size_t)P * F * tb);
  sw->sel2 = reinterpret_cast<int32_t*>(at(off));
  off = align_up(off + (size_t)P * sizeof(int32_t));
  sw->bytes = off;
}

int run_swiglu(const void* x, const uint8_t* gu_packed, const uint8_t* gu_scales,
               const uint8_t* dn_packed, const uint8_t* dn_scales, const void* sel,
               const float* p, const void* ys, void* out, int64_t T, int64_t E, int64_t I,
               int64_t F, int64_t O, int64_t K, int token_dtype, int index_dtype,
               const SwigluWorkspace& sw, cudaStream_t stream) {
  const int64_t P = T * K;
  if (K > 0) {
    // Invalid ids are counted here, once; the down projection sees expert 0
    // with h = 0 in their place and the combine skips them.
    // On the tensor cores the gate/up kernel forms h itself (tiles of gate
    // rows and their up rows), so the partial results never leave it.
    const bool tiles = E > 0 && swiglu_tiles_used(T, E, I, F, K, token_dtype);
    // With the down projection on the tensor cores too, it runs on the
    // gate/up lists (the same experts, the pairs in the same order), so the
    // gate/up tiles write h already grouped by expert: no second bucketer,
    // no gather.
    const bool reuse = tiles && down_reuses_lists(P, E, F, O, token_dtype);
    SwigluTiles st;
    if (tiles) {
      st.F = F;
      st.h = sw.h;
      st.sel2 = reuse ? nullptr : sw.sel2;
      st.grouped = reuse;
    }
    if (run_linear(x, gu_packed, gu_scales, sel, T, E, I, 2 * F, K, token_dtype, index_dtype,
                   sw.gate_up, stream, st) != cudaSuccess)
      return MXFP4EL_ERR_CUDA;
    if (E > 0) {
      if (!tiles &&
          launch_swiglu(sw.gate_up.part,
                        linear_partial_columns(T, E, I, 2 * F, K, token_dtype), sel,
                        index_dtype, E, P, F, token_dtype, sw.h, sw.sel2,
                        stream) != cudaSuccess)
        return MXFP4EL_ERR_CUDA;
      if (reuse) {
        unsigned long long* status = device_status_words();
        if (status == nullptr) return MXFP4EL_ERR_CUDA;
        mark(MXFP4EL_STAGE_LINEAR, true, stream);
        // The down projection's token rows are h's rows, already in the
        // lists' order (bf16 operands: h has no f16 copy).
        TcTokens tok;
        tok.rows = sw.h;
        tok.nrows = P;
        const cudaError_t err =
            launch_gemm_tc(tok, TcTileModes{}, dn_packed, dn_scales, sw.gate_up.plan,
                           sw.down.part, status, E, F, O, 1, SwigluTiles{}, stream,
                           kMetaUnitCounter2);
        mark(MXFP4EL_STAGE_LINEAR, false, stream);
        if (err != cudaSuccess) return MXFP4EL_ERR_CUDA;
      } else if (run_linear(sw.h, dn_packed, dn_scales, sw.sel2, P, E, F, O, 1, token_dtype,
                            MXFP4EL_INDEX_I32, sw.down, stream) != cudaSuccess) {
        return MXFP4EL_ERR_CUDA;
      }
    }
  }
  mark(MXFP4EL_STAGE_COMBINE, true, stream);
  const cudaError_t err =
      launch_combine(ys, sel, index_dtype, p, sw.down.part,
                     linear_partial_columns(P, E, F, O, 1, token_dtype), out, token_dtype, T, E,
                     O, K, K > 0 && E > 0, stream);
  mark(MXFP4EL_STAGE_COMBINE, false, stream);
  return err == cudaSuccess ? MXFP4EL_OK : MXFP4EL_ERR_CUDA;
}

// Library-owned workspace: one grow-only buffer per (device, stream).
struct Cached {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_cache_mu;
std::map<std::pair<int, cudaStream_t>, Cached>& cache() {
  static auto* m = new std::map<std::pair<int, cudaStream_t>, Cached>();
  return *m;
}

// The stream's cached workspace, grown (stream-ordered) to at least `bytes`.
// Growing is refused while the stream is being captured.
int cached_workspace(size_t bytes, cudaStream_t s, void** base) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4EL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  Cached& c = cache()[{dev, s}];
  if (c.bytes < bytes) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MXFP4EL_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return MXFP4EL_ERR_WORKSPACE;
    if (c.ptr) {
      if (cudaFreeAsync(c.ptr, s) != cudaSuccess) return MXFP4EL_ERR_CUDA;
      c.ptr = nullptr;
      c.bytes = 0;
    }
    const size_t want = std::max(bytes, c.bytes + c.bytes / 4);
    if (cudaMallocAsync(&c.ptr, want, s) != cudaSuccess) {
      c.ptr = nullptr;
      return MXFP4EL_ERR_CUDA;
    }
    c.bytes = want;
  }
  *base = c.ptr;
  return MXFP4EL_OK;
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool carve_workspace(void* base, int64_t T, int64_t E, int64_t I, int64_t O,
                     int64_t K, int token_dtype, Workspace* ws, bool with_part,
                     int64_t tiles_F, bool prepared) {
  const int64_t P = T * K;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return base ? static_cast<char*>(base) + at : nullptr;
  };
  ws->plan.meta = reinterpret_cast<int*>(take(kMetaWords * sizeof(int)));
  ws->plan.counts = reinterpret_cast<int*>(take((size_t)E * sizeof(int)));
  ws->plan.offsets = reinterpret_cast<int*>(take((size_t)(E + 1) * sizeof(int)));
  ws->plan.active = reinterpret_cast<int*>(take((size_t)E * sizeof(int)));
  ws->plan.pair_list = reinterpret_cast<int*>(take((size_t)P * sizeof(int)));
  const bool gemm = K > 0 && choose_path(T, E, I, O, K, token_dtype) == LinearPath::kGemm;
  ws->plan.pos_of_pair = gemm ? reinterpret_cast<int*>(take((size_t)P * sizeof(int))) : nullptr;
  const bool self = K > 0 && !gemm && gemv_self_route(T, E, I, O, K, prepared);
  const bool prep = token_dtype == MXFP4EL_DTYPE_BF16 && K > 0 && !gemm && !self;
  const bool prep_in_route = prep && gemv_uses_stream(I, prepared) && prep_fits_route(T, I);
  const size_t wc_words = route_global_counter_words(T, K, E, prep_in_route);
  ws->wc_global = wc_words ? reinterpret_cast<int*>(take(wc_words * sizeof(int))) : nullptr;
  ws->x16 = prep ? reinterpret_cast<__half*>(take((size_t)T * I * sizeof(__half))) : nullptr;
  ws->sigma = prep ? reinterpret_cast<int*>(take((size_t)T * sizeof(int))) : nullptr;
  ws->grouped = gemm ? reinterpret_cast<__half*>(take(gemm_tc_grouped_bytes(T, K, I))) : nullptr;
  ws->gsigma = gemm ? reinterpret_cast<int*>(take((size_t)P * sizeof(int))) : nullptr;
  // Prepared weights carry their own tile modes and row offsets.
  const bool scan = gemm && !prepared;
  ws->tile_mode = scan ? reinterpret_cast<uint8_t*>(
                             take((size_t)E * (size_t)gemm_tc_row_tiles(O, tiles_F)))
                       : nullptr;
  ws->row_off = scan ? reinterpret_cast<int16_t*>(take((size_t)E * O * sizeof(int16_t))) : nullptr;
  ws->plan.unit_begin =
      K > 0 && !gemm ? reinterpret_cast<int*>(take((kMaxSplitCtas + 1) * sizeof(int))) : nullptr;
  const size_t ncol = (size_t)linear_partial_columns(T, E, I, O, K, token_dtype);
  ws->part = with_part
                 ? reinterpret_cast<float*>(take((size_t)P * ncol * (size_t)O * sizeof(float)))
                 : nullptr;
  ws->bytes = off;
  return true;
}

}  // namespace mxfp4el

using namespace mxfp4el;

extern "C" size_t mxfp4_expert_linear_workspace_size(int64_t T, int64_t E, int64_t I,
                                                     int64_t O, int64_t K,
                                                     int token_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return (size_t)-1;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0) return (size_t)-1;
  if (!sizes_ok(T, E, I, O, K)) return (size_t)-1;
  if (T == 0 || O == 0) return 0;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws);
  return ws.bytes;
}

extern "C" int mxfp4_expert_linear_with_workspace(
    const void* latent_tokens, const uint8_t* packed_weights,
    const uint8_t* scale_bytes, const void* selected_experts,
    const float* mixture_weights, const void* shared_output, void* out,
    int64_t T, int64_t E, int64_t I, int64_t O, int64_t K, int token_dtype,
    int index_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate_linear(latent_tokens, packed_weights, scale_bytes, selected_experts,
                    mixture_weights, shared_output, out, T, E, I, O, K,
                    token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws);
  if (workspace == nullptr || workspace_bytes < ws.bytes ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return MXFP4EL_ERR_WORKSPACE;
  carve_workspace(workspace, T, E, I, O, K, token_dtype, &ws);
  return run(latent_tokens, packed_weights, scale_bytes, selected_experts,
             mixture_weights, shared_output, out, T, E, I, O, K, token_dtype,
             index_dtype, ws, static_cast<cudaStream_t>(stream));
}

extern "C" int mxfp4_expert_linear(const void* latent_tokens,
                                   const uint8_t* packed_weights,
                                   const uint8_t* scale_bytes,
                                   const void* selected_experts,
                                   const float* mixture_weights,
                                   const void* shared_output, void* out,
                                   int64_t T, int64_t E, int64_t I, int64_t O,
                                   int64_t K, int token_dtype, int index_dtype,
                                   void* stream) {
  int rc = validate_linear(latent_tokens, packed_weights, scale_bytes, selected_experts,
                    mixture_weights, shared_output, out, T, E, I, O, K,
                    token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  rc = cached_workspace(ws.bytes, s, &base);
  if (rc != MXFP4EL_OK) return rc;
  carve_workspace(base, T, E, I, O, K, token_dtype, &ws);
  return run(latent_tokens, packed_weights, scale_bytes, selected_experts,
             mixture_weights, shared_output, out, T, E, I, O, K, token_dtype,
             index_dtype, ws, s);
}

extern "C" size_t mxfp4_expert_linear_prepared_bytes(int64_t E, int64_t I, int64_t O) {
  if (E < 0 || O < 0 || I <= 0 || I % 32 != 0) return (size_t)-1;
  if (!sizes_ok(0, E, I, O, 0) || !gemv_uses_stream(I, true)) return (size_t)-1;
  return prepared_bytes(E, I, O);
}

extern "C" int mxfp4_expert_linear_prepare(const uint8_t* packed_weights,
                                           const uint8_t* scale_bytes, int64_t E, int64_t I,
                                           int64_t O, void* prepared, size_t prepared_bytes_,
                                           void* stream) {
  if (E < 0 || O < 0 || I <= 0 || I % 32 != 0) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (!sizes_ok(0, E, I, O, 0) || !gemv_uses_stream(I, true)) return MXFP4EL_ERR_TOO_LARGE;
  if (E == 0 || O == 0) return MXFP4EL_OK;
  if (packed_weights == nullptr || scale_bytes == nullptr || prepared == nullptr)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(packed_weights) % 16) return MXFP4EL_ERR_INVALID_ARGUMENT;
  const size_t need = prepared_bytes(E, I, O);
  if (prepared_bytes_ < need || reinterpret_cast<uintptr_t>(prepared) % 256 != 0)
    return MXFP4EL_ERR_WORKSPACE;
  const size_t G = (size_t)I / 32;
  if (overlaps(prepared, need, packed_weights, (size_t)E * O * G * 16) ||
      overlaps(prepared, need, scale_bytes, (size_t)E * O * G))
    return MXFP4EL_ERR_ALIAS;
  return launch_prepare(packed_weights, scale_bytes, E, I, O, prepared,
                        static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MXFP4EL_OK
             : MXFP4EL_ERR_CUDA;
}

extern "C" int mxfp4_expert_linear_prepared_with_workspace(
    const void* latent_tokens, const void* prepared, const void* selected_experts,
    const float* mixture_weights, const void* shared_output, void* out, int64_t T, int64_t E,
    int64_t I, int64_t O, int64_t K, int token_dtype, int index_dtype, void* workspace,
    size_t workspace_bytes, void* stream) {
  int rc = validate_prepared(latent_tokens, prepared, selected_experts, mixture_weights,
                             shared_output, out, T, E, I, O, K, token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws, true, 0, true);
  if (workspace == nullptr || workspace_bytes < ws.bytes ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return MXFP4EL_ERR_WORKSPACE;
  carve_workspace(workspace, T, E, I, O, K, token_dtype, &ws, true, 0, true);
  const PreparedView v = prepared_view(prepared, E, I, O);
  return run(latent_tokens, nullptr, nullptr, selected_experts, mixture_weights, shared_output,
             out, T, E, I, O, K, token_dtype, index_dtype, ws, static_cast<cudaStream_t>(stream),
             &v);
}

extern "C" size_t mxfp4_expert_linear_prepared_workspace_size(int64_t T, int64_t E, int64_t I,
                                                              int64_t O, int64_t K,
                                                              int token_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return (size_t)-1;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0) return (size_t)-1;
  if (!sizes_ok(T, E, I, O, K) || !gemv_uses_stream(I, true)) return (size_t)-1;
  if (T == 0 || O == 0) return 0;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws, true, 0, true);
  return ws.bytes;
}

extern "C" int mxfp4_expert_linear_prepared(const void* latent_tokens, const void* prepared,
                                            const void* selected_experts,
                                            const float* mixture_weights,
                                            const void* shared_output, void* out, int64_t T,
                                            int64_t E, int64_t I, int64_t O, int64_t K,
                                            int token_dtype, int index_dtype, void* stream) {
  int rc = validate_prepared(latent_tokens, prepared, selected_experts, mixture_weights,
                             shared_output, out, T, E, I, O, K, token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  Workspace ws;
  carve_workspace(nullptr, T, E, I, O, K, token_dtype, &ws, true, 0, true);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  rc = cached_workspace(ws.bytes, s, &base);
  if (rc != MXFP4EL_OK) return rc;
  carve_workspace(base, T, E, I, O, K, token_dtype, &ws, true, 0, true);
  const PreparedView v = prepared_view(prepared, E, I, O);
  return run(latent_tokens, nullptr, nullptr, selected_experts, mixture_weights, shared_output,
             out, T, E, I, O, K, token_dtype, index_dtype, ws, s, &v);
}

extern "C" int mxfp4_router_topk(const float* router_logits, const float* router_bias,
                                 int64_t T, int64_t E, int64_t K, float scaling,
                                 int32_t* selected_experts, float* mixture_weights,
                                 void* stream) {
  if (T < 0 || E < 0 || K < 0 || K > E) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (T > kMaxDim || E > kMaxDim || (K > 0 && T > kMaxPairs / K)) return MXFP4EL_ERR_TOO_LARGE;
  if (T == 0 || K == 0) return MXFP4EL_OK;
  if (router_logits == nullptr || selected_experts == nullptr || mixture_weights == nullptr)
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (router_warps_per_block(E, K) <= 0) return MXFP4EL_ERR_TOO_LARGE;
  const size_t nl = (size_t)T * E * sizeof(float), nb = (size_t)E * sizeof(float);
  const size_t ns = (size_t)T * K * sizeof(int32_t), np = (size_t)T * K * sizeof(float);
  if (overlaps(selected_experts, ns, router_logits, nl) ||
      overlaps(selected_experts, ns, router_bias, nb) ||
      overlaps(mixture_weights, np, router_logits, nl) ||
      overlaps(mixture_weights, np, router_bias, nb) ||
      overlaps(selected_experts, ns, mixture_weights, np))
    return MXFP4EL_ERR_ALIAS;
  return launch_router(router_logits, router_bias, T, E, K, scaling, selected_experts,
                       mixture_weights, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MXFP4EL_OK
             : MXFP4EL_ERR_CUDA;
}

extern "C" int mxfp4_expert_linear_routed(const void* latent_tokens,
                                          const uint8_t* packed_weights,
                                          const uint8_t* scale_bytes,
                                          const float* router_logits,
                                          const float* router_bias, float scaling,
                                          const void* shared_output, void* out,
                                          int32_t* selected_experts, float* mixture_weights,
                                          int64_t T, int64_t E, int64_t I, int64_t O,
                                          int64_t K, int token_dtype, void* stream) {
  // Check the linear's arguments first: nothing is enqueued for a call that
  // would fail half way.
  int rc = validate_linear(latent_tokens, packed_weights, scale_bytes, selected_experts,
                    mixture_weights, shared_output, out, T, E, I, O, K, token_dtype,
                    MXFP4EL_INDEX_I32);
  if (rc != MXFP4EL_OK) return rc;
  if (K > E) return MXFP4EL_ERR_INVALID_ARGUMENT;
  if (T == 0 || O == 0) return MXFP4EL_OK;
  rc = mxfp4_router_topk(router_logits, router_bias, T, E, K, scaling, selected_experts,
                         mixture_weights, stream);
  if (rc != MXFP4EL_OK) return rc;
  return mxfp4_expert_linear(latent_tokens, packed_weights, scale_bytes, selected_experts,
                             mixture_weights, shared_output, out, T, E, I, O, K, token_dtype,
                             MXFP4EL_INDEX_I32, stream);
}

extern "C" size_t mxfp4_swiglu_expert_workspace_size(int64_t T, int64_t E, int64_t I,
                                                     int64_t F, int64_t O, int64_t K,
                                                     int token_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16) return (size_t)-1;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0 || F <= 0 || F % 32 != 0)
    return (size_t)-1;
  if (F > kMaxDim / 2 || !sizes_ok(T, E, I, 2 * F, K) || !sizes_ok(T * K, E, F, O, 1))
    return (size_t)-1;
  if (T == 0 || O == 0) return 0;
  SwigluWorkspace sw;
  carve_swiglu(nullptr, T, E, I, F, O, K, token_dtype, &sw);
  return sw.bytes;
}

extern "C" int mxfp4_swiglu_expert_with_workspace(
    const void* latent_tokens, const uint8_t* gate_up_packed, const uint8_t* gate_up_scales,
    const uint8_t* down_packed, const uint8_t* down_scales, const void* selected_experts,
    const float* mixture_weights, const void* shared_output, void* out, int64_t T, int64_t E,
    int64_t I, int64_t F, int64_t O, int64_t K, int token_dtype, int index_dtype,
    void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = validate_swiglu(latent_tokens, gate_up_packed, gate_up_scales, down_packed,
                                 down_scales, selected_experts, mixture_weights, shared_output,
                                 out, T, E, I, F, O, K, token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  SwigluWorkspace sw;
  carve_swiglu(nullptr, T, E, I, F, O, K, token_dtype, &sw);
  if (workspace == nullptr || workspace_bytes < sw.bytes ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return MXFP4EL_ERR_WORKSPACE;
  carve_swiglu(workspace, T, E, I, F, O, K, token_dtype, &sw);
  return run_swiglu(latent_tokens, gate_up_packed, gate_up_scales, down_packed, down_scales,
                    selected_experts, mixture_weights, shared_output, out, T, E, I, F, O, K,
                    token_dtype, index_dtype, sw, static_cast<cudaStream_t>(stream));
}

extern "C" int mxfp4_swiglu_expert(const void* latent_tokens, const uint8_t* gate_up_packed,
                                   const uint8_t* gate_up_scales, const uint8_t* down_packed,
                                   const uint8_t* down_scales, const void* selected_experts,
                                   const float* mixture_weights, const void* shared_output,
                                   void* out, int64_t T, int64_t E, int64_t I, int64_t F,
                                   int64_t O, int64_t K, int token_dtype, int index_dtype,
                                   void* stream) {
  int rc = validate_swiglu(latent_tokens, gate_up_packed, gate_up_scales, down_packed,
                           down_scales, selected_experts, mixture_weights, shared_output, out,
                           T, E, I, F, O, K, token_dtype, index_dtype);
  if (rc != MXFP4EL_OK || T == 0 || O == 0) return rc;
  SwigluWorkspace sw;
  carve_swiglu(nullptr, T, E, I, F, O, K, token_dtype, &sw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  rc = cached_workspace(sw.bytes, s, &base);
  if (rc != MXFP4EL_OK) return rc;
  carve_swiglu(base, T, E, I, F, O, K, token_dtype, &sw);
  return run_swiglu(latent_tokens, gate_up_packed, gate_up_scales, down_packed, down_scales,
                    selected_experts, mixture_weights, shared_output, out, T, E, I, F, O, K,
                    token_dtype, index_dtype, sw, s);
}

extern "C" int mxfp4el_device_errors(void* stream, int64_t* bad_pairs) {
  if (bad_pairs == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  return read_and_reset_status(static_cast<cudaStream_t>(stream), kStatusBadPairs,
                               bad_pairs) == cudaSuccess
             ? MXFP4EL_OK
             : MXFP4EL_ERR_CUDA;
}

extern "C" int mxfp4el_wait_timeouts(void* stream, int64_t* count) {
  if (count == nullptr) return MXFP4EL_ERR_INVALID_ARGUMENT;
  return read_and_reset_status(static_cast<cudaStream_t>(stream), kStatusWaitTimeouts,
                               count) == cudaSuccess
             ? MXFP4EL_OK
             : MXFP4EL_ERR_CUDA;
}

extern "C" int mxfp4el_set_stage_events(int stage, void* start_event,
                                        void* end_event) {
  if (stage < 0 || stage >= MXFP4EL_NUM_STAGES) return MXFP4EL_ERR_INVALID_ARGUMENT;
  g_stage[stage].start = static_cast<cudaEvent_t>(start_event);
  g_stage[stage].end = static_cast<cudaEvent_t>(end_event);
  return MXFP4EL_OK;
}

extern "C" int64_t mxfp4el_kernel_launches(void) { return g_launches.load(); }

extern "C" int mxfp4el_linear_path(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                                   int token_dtype) {
  if (token_dtype != MXFP4EL_DTYPE_F32 && token_dtype != MXFP4EL_DTYPE_BF16)
    return MXFP4EL_ERR_UNSUPPORTED_DTYPE;
  if (T < 0 || E < 0 || O < 0 || K < 0 || I <= 0 || I % 32 != 0 || !sizes_ok(T, E, I, O, K))
    return MXFP4EL_ERR_INVALID_ARGUMENT;
  return choose_path(T, E, I, O, K, token_dtype) == LinearPath::kGemm ? MXFP4EL_PATH_GEMM
                                                                       : MXFP4EL_PATH_GEMV;
}

extern "C" const char* mxfp4el_status_string(int status) {
  switch (status) {
    case MXFP4EL_OK: return "ok";
    case MXFP4EL_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MXFP4EL_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case MXFP4EL_ERR_ALIAS: return "output overlaps an input";
    case MXFP4EL_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MXFP4EL_ERR_CUDA: return "CUDA error";
    case MXFP4EL_ERR_TOO_LARGE: return "size beyond library limits";
    default: return "unknown status";
  }
}

extern "C" int mxfp4el_version(void) { return 100; }
