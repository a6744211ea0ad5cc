/*
 * mxfp4_expert_linear.h -- C ABI of the MXFP4 routed expert linear for GB300.
 *
 * The operation (problem statement "MXFP4 Routed Expert Linear", Kimi K3,
 * sections "What is stored in one group" through "Route, weight, and add the
 * shared path"; the same problem stated formally as "MXFP4 Experts" on
 * tensortonic):
 *
 *   W_e[o, 32 g + 2 j    ] = LUT[ b & 15 ] * 2^(s - 127)
 *   W_e[o, 32 g + 2 j + 1] = LUT[ b >> 4 ] * 2^(s - 127)
 *         b = packed_weights[e, o, g, j],  s = scale_bytes[e, o, g]
 *   LUT   = { 0, .5, 1, 1.5, 2, 3, 4, 6, -0, -.5, -1, -1.5, -2, -3, -4, -6 }
 *   out[t, :] = shared_output[t, :] + sum_{k < K} p[t, k] * W_{sel[t, k]} x[t, :]
 *
 * Only the experts some token selects are ever read ("Decode only selected
 * experts"). The K routed contributions are added onto the shared output in
 * slot order k = 0, 1, ..., K-1 in float32, then rounded once to the token
 * dtype, so a call is deterministic: the same inputs give the same bits.
 *
 * Everything here is plain C: pointers, sizes and status codes. Every pointer
 * argument of the compute calls is a DEVICE pointer (CUDA global memory of
 * the device current on the calling thread) owned by the caller; the library
 * never frees or retains them. Inputs are never written ("Requirements": do
 * not mutate packed weights, routing data, or shared output). All GPU work is
 * enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 * the calls return without waiting for it.
 *
 * Dense row-major layouts (no padding, element strides as listed):
 *   latent_tokens     (T, I)          token dtype (fp32 or bf16)
 *   packed_weights    (E, O, G, 16)   uint8, G = I / 32
 *   scale_bytes       (E, O, G)       uint8 (E8M0 exponent, bias 127)
 *   selected_experts  (T, K)          int32 or int64 expert ids
 *   mixture_weights   (T, K)          float32
 *   shared_output     (T, O)          token dtype
 *   out               (T, O)          token dtype, written by the call
 */
#ifndef MXFP4_EXPERT_LINEAR_H
#define MXFP4_EXPERT_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. 0 is success; every error is negative and is returned before
 * any GPU work is enqueued, except MXFP4EL_ERR_CUDA, which reports a failed
 * launch or allocation (work enqueued before it may have run). */
#define MXFP4EL_OK                     0
#define MXFP4EL_ERR_INVALID_ARGUMENT  -1  /* null pointer, negative size,
                                             I <= 0 or I % 32 != 0          */
#define MXFP4EL_ERR_UNSUPPORTED_DTYPE -2  /* token or index dtype not listed */
#define MXFP4EL_ERR_ALIAS             -3  /* out overlaps an input           */
#define MXFP4EL_ERR_WORKSPACE         -4  /* caller workspace too small or
                                             misaligned                      */
#define MXFP4EL_ERR_CUDA              -5  /* a CUDA call failed              */
#define MXFP4EL_ERR_TOO_LARGE         -6  /* a size exceeds the library limit */

/* Token dtype: latent_tokens, shared_output and out share it ("Preserve the
 * latent token dtype"). */
#define MXFP4EL_DTYPE_F32   0
#define MXFP4EL_DTYPE_BF16  1

/* Dtype of selected_experts. */
#define MXFP4EL_INDEX_I32   0
#define MXFP4EL_INDEX_I64   1

/*
 * mxfp4_expert_linear -- the routed expert linear on one GPU.
 *
 * Sizes: T tokens, E experts, I input width (a positive multiple of 32,
 * "Constraints"), O output width, K picks per token. T, E, O, K >= 0.
 * T == 0 or O == 0 enqueues nothing. K == 0 copies shared_output to out.
 *
 * selected_experts: the pages require valid ids. An id outside [0, E) is
 * not read from memory: that (t, k) pair contributes nothing, and it is
 * counted in a per-device error counter read by mxfp4el_device_errors().
 * A token may repeat an id; each slot is then added separately.
 *
 * mixture_weights are used as given (the pages state they sum to one per
 * token; nothing renormalises them).
 *
 * Scratch memory (routing lists and one float32 partial per (pair, row),
 * see mxfp4_expert_linear_workspace_size) is owned by the library: one
 * grow-only buffer per (device, stream), grown with the stream-ordered
 * cudaFreeAsync/cudaMallocAsync on `stream` the first time a call needs
 * more, and kept until the process exits. A call that would grow it while
 * `stream` is being captured into a CUDA graph returns MXFP4EL_ERR_WORKSPACE
 * instead: make a first call of the largest size before capturing, or use
 * mxfp4_expert_linear_with_workspace. Calls on one stream are ordered; calls
 * on different streams use different buffers.
 *
 * Returns MXFP4EL_OK or one of the negative codes above.
 */
int mxfp4_expert_linear(const void* latent_tokens,
                        const uint8_t* packed_weights,
                        const uint8_t* scale_bytes,
                        const void* selected_experts,
                        const float* mixture_weights,
                        const void* shared_output,
                        void* out,
                        int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                        int token_dtype, int index_dtype,
                        void* stream);

/*
 * mxfp4_router_topk -- the sigmoid top-K router that feeds the routed expert
 * linear ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact
 * Experts", section 1, the sigmoid router; the Hy3 decode write-up, the
 * router after its logits).
 *
 * router_logits (T, E) float32, row-major; router_bias (E) float32 or NULL
 * (no bias). Per token: score = sigmoid(logit) in float32, choice = score +
 * bias; selected_experts (T, K) int32 receives the K experts of highest
 * choice, highest first, ties to the lower index; mixture_weights (T, K)
 * float32 receives their raw scores (the bias steers the choice only),
 * summed left to right, each divided by that sum plus 1e-20 and multiplied by
 * `scaling`. An expert whose choice is NaN is never selected; a slot left
 * without an expert gets id -1 (skipped by the linear) and weight 0.
 * All pointers are device pointers owned by the caller; the outputs may not
 * overlap the inputs or each other (MXFP4EL_ERR_ALIAS). Requires
 * 0 <= K <= E and (2E + K) * 4 <= 49152 bytes (MXFP4EL_ERR_TOO_LARGE
 * beyond). Stream-ordered on `stream`; returns MXFP4EL_OK or a negative code.
 */
int mxfp4_router_topk(const float* router_logits, const float* router_bias,
                      int64_t T, int64_t E, int64_t K, float scaling,
                      int32_t* selected_experts, float* mixture_weights,
                      void* stream);

/*
 * mxfp4_expert_linear_routed -- the router above, then the routed expert
 * linear on its selection, on one stream: selected_experts (T, K) int32 and
 * mixture_weights (T, K) float32 are caller-owned outputs of the router and
 * inputs of the linear (the linear's first kernel waits for the router).
 * Every other argument, and the result in `out`, as mxfp4_expert_linear with
 * index_dtype MXFP4EL_INDEX_I32. All arguments are checked before anything is
 * enqueued.
 */
int mxfp4_expert_linear_routed(const void* latent_tokens,
                               const uint8_t* packed_weights,
                               const uint8_t* scale_bytes,
                               const float* router_logits,
                               const float* router_bias, float scaling,
                               const void* shared_output, void* out,
                               int32_t* selected_experts, float* mixture_weights,
                               int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                               int token_dtype, void* stream);

/*
 * Bytes of scratch one call of these sizes needs when the caller supplies it
 * (mxfp4_expert_linear_with_workspace). Returns 0 for a no-op call and
 * (size_t)-1 for sizes the library rejects.
 */
size_t mxfp4_expert_linear_workspace_size(int64_t T, int64_t E, int64_t I,
                                          int64_t O, int64_t K,
                                          int token_dtype);

/*
 * Same operation with caller-owned scratch: `workspace` is a device buffer of
 * at least mxfp4_expert_linear_workspace_size(...) bytes, 256-byte aligned.
 * The library allocates nothing. The call may overwrite all of it; it must
 * not overlap any argument, and two calls in flight at once (on different
 * streams) must not share it. Errors as mxfp4_expert_linear, plus
 * MXFP4EL_ERR_WORKSPACE when the buffer is too small or misaligned.
 */
int mxfp4_expert_linear_with_workspace(const void* latent_tokens,
                                       const uint8_t* packed_weights,
                                       const uint8_t* scale_bytes,
                                       const void* selected_experts,
                                       const float* mixture_weights,
                                       const void* shared_output,
                                       void* out,
                                       int64_t T, int64_t E, int64_t I,
                                       int64_t O, int64_t K,
                                       int token_dtype, int index_dtype,
                                       void* workspace,
                                       size_t workspace_bytes,
                                       void* stream);

/*
 * Prepared weights -- a load-time copy of (packed_weights, scale_bytes) laid
 * out for the kernels ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant
 * Compact Experts", section 2, the weight preparation built once at load
 * time). It holds the same values; calls on it give the same bits as
 * mxfp4_expert_linear on the plain layout.
 *
 * Layout (mtiles = ceil(O / 128), nk = ceil(G / 2), G = I / 32), one
 * 4352-byte block per (expert e, 128-row tile mt, 64-wide K chunk kc) at
 * byte ((e * mtiles + mt) * nk + kc) * 4352:
 *   bytes 32 m .. 32 m + 31: row o = 128 mt + m, the packed bytes of groups
 *     2kc and 2kc+1, the two 16-byte halves swapped when bit 2 of m is set;
 *   bytes 4096 + 2 m, 4097 + 2 m: its scale bytes of those groups.
 * Rows past O hold zero codes and the scale bytes of row O - 1; for odd G the
 * missing group G holds zero codes and the scale byte of group G - 1. Then,
 * each part starting 256-byte aligned: int16 [E][O] and uint8 [E][mtiles]
 * values that the tensor-core kernel derives from the scale bytes (per-row
 * offsets and per-tile flags of its exact f16 operand mode).
 *
 * mxfp4_expert_linear_prepared_bytes: bytes of the copy, or (size_t)-1 for
 * invalid sizes or I > 15360 (the prepared calls' limit).
 */
size_t mxfp4_expert_linear_prepared_bytes(int64_t E, int64_t I, int64_t O);

/*
 * mxfp4_expert_linear_prepare -- writes the prepared copy of the weights into
 * `prepared`, a caller-owned device buffer of at least `prepared_bytes`
 * (>= mxfp4_expert_linear_prepared_bytes) bytes, 256-byte aligned, that
 * overlaps neither input. Stream-ordered on `stream`; the kernels start only
 * after earlier work on the stream has finished, so a buffer that an earlier
 * call on the same stream still reads may be refilled. packed_weights must be
 * 16-byte aligned. Returns MXFP4EL_OK, MXFP4EL_ERR_INVALID_ARGUMENT (null
 * pointer, negative size, I % 32 != 0), MXFP4EL_ERR_TOO_LARGE,
 * MXFP4EL_ERR_WORKSPACE (buffer too small or misaligned), MXFP4EL_ERR_ALIAS
 * or MXFP4EL_ERR_CUDA. E == 0 or O == 0 enqueues nothing.
 */
int mxfp4_expert_linear_prepare(const uint8_t* packed_weights,
                                const uint8_t* scale_bytes,
                                int64_t E, int64_t I, int64_t O,
                                void* prepared, size_t prepared_bytes,
                                void* stream);

/*
 * mxfp4_expert_linear_prepared -- mxfp4_expert_linear on prepared weights:
 * `prepared` (256-byte aligned, written by mxfp4_expert_linear_prepare for
 * the same E, I, O) replaces packed_weights and scale_bytes; every other
 * argument, the scratch and the errors are as mxfp4_expert_linear, plus
 * MXFP4EL_ERR_TOO_LARGE for I > 15360. The _with_workspace form takes
 * caller-owned scratch of mxfp4_expert_linear_prepared_workspace_size(...)
 * bytes, as mxfp4_expert_linear_with_workspace does.
 */
int mxfp4_expert_linear_prepared(const void* latent_tokens,
                                 const void* prepared,
                                 const void* selected_experts,
                                 const float* mixture_weights,
                                 const void* shared_output,
                                 void* out,
                                 int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                                 int token_dtype, int index_dtype,
                                 void* stream);
size_t mxfp4_expert_linear_prepared_workspace_size(int64_t T, int64_t E, int64_t I,
                                                   int64_t O, int64_t K,
                                                   int token_dtype);
int mxfp4_expert_linear_prepared_with_workspace(const void* latent_tokens,
                                                const void* prepared,
                                                const void* selected_experts,
                                                const float* mixture_weights,
                                                const void* shared_output,
                                                void* out,
                                                int64_t T, int64_t E, int64_t I,
                                                int64_t O, int64_t K,
                                                int token_dtype, int index_dtype,
                                                void* workspace,
                                                size_t workspace_bytes,
                                                void* stream);

/*
 * mxfp4_swiglu_expert -- the whole routed SwiGLU expert with MXFP4 weights
 * ("MoE Expert Kernels: Grouped Prefill and Mixed-Quant Compact Experts",
 * section 1, the expert shape: down(silu(gate(x)) * up(x)) per routed expert,
 * accumulated with the routing weight in float32; the Hy3 decode write-up:
 * gate and up stacked along their output rows, one gathered row per
 * token-expert pair):
 *
 *   g = Wg_e x_t,  u = Wu_e x_t          (gate/up: rows 0..F-1 and F..2F-1)
 *   h[f] = silu(g[f]) * u[f],  silu(v) = v / (1 + exp(-v))
 *   out[t, :] = shared_output[t, :] + sum_{k < K} p[t, k] * Wd_e h,  e = sel[t, k]
 *
 * Every matrix decodes as in mxfp4_expert_linear. Layouts (dense, row-major):
 *   latent_tokens   (T, I)                 token dtype
 *   gate_up_packed  (E, 2F, I/32, 16)      uint8; rows 0..F-1 gate, F..2F-1 up
 *   gate_up_scales  (E, 2F, I/32)          uint8
 *   down_packed     (E, O, F/32, 16)       uint8
 *   down_scales     (E, O, F/32)           uint8
 *   selected_experts, mixture_weights, shared_output, out: as mxfp4_expert_linear.
 * I and F are positive multiples of 32. g and u are float32 sums; h is
 * computed in float32 and rounded once to the token dtype (the down
 * projection's input); the K contributions are added in slot order in
 * float32 and rounded once, so a call is deterministic.
 *
 * Ids outside [0, E): the pair contributes nothing and is counted once per
 * call for mxfp4el_device_errors(). Scratch is library-owned exactly as for
 * mxfp4_expert_linear (the same grow-only buffer per device and stream).
 * All pointers are caller-owned device pointers; out may not overlap an
 * input (MXFP4EL_ERR_ALIAS); latent_tokens, gate_up_packed and down_packed
 * must be 16-byte aligned. Returns MXFP4EL_OK or a negative code, checked
 * before anything is enqueued except MXFP4EL_ERR_CUDA.
 */
int mxfp4_swiglu_expert(const void* latent_tokens,
                        const uint8_t* gate_up_packed, const uint8_t* gate_up_scales,
                        const uint8_t* down_packed, const uint8_t* down_scales,
                        const void* selected_experts, const float* mixture_weights,
                        const void* shared_output, void* out,
                        int64_t T, int64_t E, int64_t I, int64_t F, int64_t O, int64_t K,
                        int token_dtype, int index_dtype, void* stream);

/* Bytes of caller-owned scratch for mxfp4_swiglu_expert_with_workspace: 0 for
 * a no-op call, (size_t)-1 for sizes the library rejects. */
size_t mxfp4_swiglu_expert_workspace_size(int64_t T, int64_t E, int64_t I, int64_t F,
                                          int64_t O, int64_t K, int token_dtype);

/* mxfp4_swiglu_expert with caller-owned scratch, with the rules of
 * mxfp4_expert_linear_with_workspace. */
int mxfp4_swiglu_expert_with_workspace(const void* latent_tokens,
                                       const uint8_t* gate_up_packed,
                                       const uint8_t* gate_up_scales,
                                       const uint8_t* down_packed,
                                       const uint8_t* down_scales,
                                       const void* selected_experts,
                                       const float* mixture_weights,
                                       const void* shared_output, void* out,
                                       int64_t T, int64_t E, int64_t I, int64_t F,
                                       int64_t O, int64_t K, int token_dtype,
                                       int index_dtype, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * mxfp4_expert_linear_static_scratch -- the same operation for callers that
 * cannot allocate device memory (for example a serving process whose memory
 * budget is fixed at start-up, or a plugin of a host framework that owns
 * every device allocation). The pages have no counterpart: it is a property
 * of this library's interface, not of the method.
 *
 * Arguments, results and errors are those of mxfp4_expert_linear. The caller
 * still passes every input and `out`; the scratch lives in a fixed device
 * array compiled into the library, mxfp4_expert_linear_static_scratch_bytes()
 * bytes (8 MiB) on every GPU that loads the library, held until the process
 * exits. The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine). Sizes whose scratch
 * (mxfp4_expert_linear_workspace_size) exceeds the array are rejected with
 * MXFP4EL_ERR_TOO_LARGE before any GPU work. The scratch is dominated by
 * float32 partial results per (token, slot, output row); for example a batch
 * of T=8 tokens, K=4, I=2880, O=5760 needs about 2.2 MiB and fits, while
 * T=16, K=8, I=7168, O=4096 needs about 14 MiB and is refused.
 *
 * Arguments are checked exactly as by mxfp4_expert_linear, in the same
 * order, so a call that has another error returns that error's code; only a
 * call those checks accept can be refused with MXFP4EL_ERR_TOO_LARGE.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the device current); make that first
 * call before any stream capture. The address is kept until the process
 * exits: do not use this entry point on a device after cudaDeviceReset (or
 * any other teardown of its primary context). Every call on a device shares the one
 * array, which keeps the previous call's contents; nothing in it needs to
 * start at zero, because the kernels initialise everything they read. Calls
 * that overlap on the GPU (on different streams, or from different threads
 * without ordering) race on the array and give undefined results: order them.
 */
int mxfp4_expert_linear_static_scratch(const void* latent_tokens,
                                       const uint8_t* packed_weights,
                                       const uint8_t* scale_bytes,
                                       const void* selected_experts,
                                       const float* mixture_weights,
                                       const void* shared_output,
                                       void* out,
                                       int64_t T, int64_t E, int64_t I,
                                       int64_t O, int64_t K,
                                       int token_dtype, int index_dtype,
                                       void* stream);

/* Size in bytes of the fixed scratch array of the entry point above. */
size_t mxfp4_expert_linear_static_scratch_bytes(void);

/*
 * Synchronises `stream`, then returns in *bad_pairs the number of (t, k)
 * pairs with an expert id outside [0, E) seen on the current device since the
 * last call of this function, and resets that count to zero.
 */
int mxfp4el_device_errors(void* stream, int64_t* bad_pairs);

/*
 * Synchronises `stream`, then returns in *count the number of kernel waits
 * (on a copy or on another warp of the same CTA) that gave up after their
 * time limit on the current device since the last call, and resets it. Every
 * wait in the library's kernels is bounded (2 s); a kernel whose wait gave up
 * returns early, so the outputs of the calls involved are not valid. A
 * healthy device always reports 0.
 */
int mxfp4el_wait_timeouts(void* stream, int64_t* count);

/*
 * Instrumentation for benchmarks. Stage ids name the kernels a call launches,
 * in launch order. Once events are set for a stage, every later call records
 * `start_event` on its stream just before that stage's kernel launch and
 * `end_event` just after it (cudaEvent_t handles the caller created on the
 * current device). NULL, NULL clears a stage. The setting is process-wide and
 * not thread-safe against concurrent calls; it does not change any result.
 * Returns MXFP4EL_ERR_INVALID_ARGUMENT for an unknown stage.
 */
#define MXFP4EL_STAGE_ROUTE    0   /* routing bucketer (+ token prep) */
#define MXFP4EL_STAGE_LINEAR   1   /* routed expert linear (GEMV or GEMM) */
#define MXFP4EL_STAGE_COMBINE  2   /* weighted combine onto y_shared */
#define MXFP4EL_STAGE_GATHER   3   /* tokens grouped by expert (GEMM path) */
#define MXFP4EL_NUM_STAGES     4
int mxfp4el_set_stage_events(int stage, void* start_event, void* end_event);

/*
 * Which kernel computes the routed linear for these sizes: MXFP4EL_PATH_GEMV
 * (CUDA cores, decode regime) or MXFP4EL_PATH_GEMM (tensor cores, bf16
 * tokens, experts averaging 16 or more tokens). Negative for sizes the
 * library rejects. The environment variable MXFP4EL_PATH=gemv|gemm, read at
 * every call, forces one where it applies (a testing aid).
 */
#define MXFP4EL_PATH_GEMV 0
#define MXFP4EL_PATH_GEMM 1
int mxfp4el_linear_path(int64_t T, int64_t E, int64_t I, int64_t O, int64_t K,
                        int token_dtype);

/* Kernel launches this process has made through the library so far. */
int64_t mxfp4el_kernel_launches(void);

/* Human-readable text for a status code (static storage, never NULL). */
const char* mxfp4el_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int mxfp4el_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_EXPERT_LINEAR_H */
