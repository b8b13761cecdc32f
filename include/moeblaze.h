/*
 * moeblaze.h - C ABI of a GB300 (sm_103a) dropless top-K Mixture-of-Experts
 * layer in the style of MoEBlaze ("MoEBlaze: Breaking the Memory Wall for
 * Efficient MoE Training on Modern GPUs", MLSys 2026).
 *
 * The layer (MoEBlaze, awesome-system-papers page, section "核心方法"):
 *   y[t] = sum_k g[t,k] * expert_{e}(x[t]),  e = topk_ids[t,k]
 *   SwiGLU expert:  (SiLU(x W1_e) * (x W2_e)) W3_e
 *   SiLU expert:    SiLU(x W1_e) W3_e
 *   identity:       x
 * computed without a routed (L*K, d) buffer: the dispatch builds integer
 * index structures only, the expert GEMMs gather rows of x through them, and
 * the down-projection is gate-weighted and reduced back into (L, d).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument named "device" is device memory owned by the
 *     caller; the library never allocates or frees device memory and keeps
 *     no state between calls (apart from a per-device SM count).
 *   - Every device pointer must be 16-byte aligned (MOEBLAZE_ERR_INVALID_ARG
 *     otherwise); row-major layouts, no padding between rows.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and is asynchronous, except dispatch_build with
 *     validate != 0 and moeblaze_device_error, which synchronise `stream`.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned as a status; nothing is thrown across the ABI and there
 *     is no CPU fallback.
 *   - dtype: MOEBLAZE_BF16 = bf16 storage, fp32 accumulation (tensor cores,
 *     needs d % 128 == 0 and h % 128 == 0); MOEBLAZE_F32 = fp32 storage and
 *     fp32 SIMT arithmetic (no TF32), any d, h with d % 4 == 0 and h % 4 == 0.
 *   - Limits: 1 <= K <= min(E, 8), 1 <= E <= 512, 0 <= L, L*K < 2^31.
 */
#ifndef MOEBLAZE_H
#define MOEBLAZE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOEBLAZE_API __attribute__((visibility("default")))
#else
#define MOEBLAZE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* moeblaze_stream;

typedef enum {
  MOEBLAZE_OK = 0,
  MOEBLAZE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape, K > E */
  MOEBLAZE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. bf16 with d % 128 != 0) */
  MOEBLAZE_ERR_BAD_ROUTING = 3,  /* an id out of [0,E) or repeated within a token */
  MOEBLAZE_ERR_WORKSPACE = 4,    /* workspace smaller than the matching *_bytes() */
  MOEBLAZE_ERR_TIMEOUT = 5,      /* a device-side wait ran out; results invalid */
  MOEBLAZE_ERR_CUDA = 6          /* a CUDA runtime/driver call failed */
} moeblaze_status;

enum { MOEBLAZE_F32 = 0, MOEBLAZE_BF16 = 1 };
enum { MOEBLAZE_SWIGLU = 0, MOEBLAZE_SILU = 1, MOEBLAZE_IDENTITY = 2 };

/* Layer shape.  L tokens, model dim d, expert hidden dim h (ignored for the
 * identity expert), E experts, top-K slots per token, and option flags. */
typedef struct {
  int64_t L;
  int32_t d, h, E, K;
  int32_t dtype;  /* MOEBLAZE_F32 | MOEBLAZE_BF16 */
  int32_t act;    /* MOEBLAZE_SWIGLU | MOEBLAZE_SILU | MOEBLAZE_IDENTITY */
  int32_t flags;  /* 0 or MOEBLAZE_RECOMPUTE_H; other bits: MOEBLAZE_ERR_INVALID_ARG */
} moeblaze_shape;

/* MOEBLAZE_RECOMPUTE_H: keep no H = SiLU(A)*B (SiLU: SiLU(A)) and no
 * Hg = g*H temporary (MoEBlaze, awesome-system-papers page, section
 * "SwiGLU kernel 融合 + activation checkpoint": the fused kernels write only
 * their final outputs).  Applies to the bf16 SwiGLU and SiLU layers (ignored
 * otherwise): the down projection and the dW3 GEMM then recompute H and Hg
 * tile by tile from the saved A and B inside their operand pipelines.  The
 * forward and the backward workspace each shrink by padded_rows x h
 * elements (the saved buffer grows by one fp32 gate per padded row); those
 * two GEMMs do the extra recompute, and the backward runs its dW3 GEMM
 * first, while the saved A and B are still intact.  Results agree with the default within
 * the bf16 tolerance (SiLU is then evaluated as a/2 (1 + tanh(a/2)) with the
 * hardware tanh approximation). */
#define MOEBLAZE_RECOMPUTE_H 1

/* The index structures of MoEBlaze (awesome-system-papers page, section
 * "免物化 token dispatch", data-structure table).  All device, int32,
 * written by moeblaze_dispatch_build:
 *   expert_token_indices [L*K]  token ids expert by expert, ascending token id
 *                                within an expert
 *   expert_token_offsets [E+1]  expert e owns [off[e], off[e+1]); off[E] = L*K
 *   token_expert_indices [L*K]  (L,K) row-major: the expert of (t,k) (= topk_ids)
 *   token_index_map      [L*K]  (L,K) row-major: position of (t,k) in
 *                                expert_token_indices
 *   meta                         moeblaze_dispatch_meta_bytes() bytes, 16-byte
 *                                aligned: per-expert counts, padded row offsets,
 *                                the GEMM tile table, a device error word and
 *                                the (L, E, K) the build was made for; read by
 *                                forward/backward, otherwise opaque to the caller.
 * A dispatch serves only forward/backward calls with the L, E and K of the
 * shape it was built for.  Their kernels compare the three with the values
 * the build recorded in meta before they read any of the structures; on a
 * mismatch they read none of them, leave their outputs unspecified and set
 * bit 4 of the device error word (moeblaze_device_error then returns
 * MOEBLAZE_ERR_INVALID_ARG).
 */
typedef struct {
  int32_t* expert_token_indices;
  int32_t* expert_token_offsets;
  int32_t* token_expert_indices;
  int32_t* token_index_map;
  void* meta;
} moeblaze_dispatch;

/* Byte sizes.  0 is a valid size (nothing needed).  An invalid shape gives 0;
 * the matching entry point then reports the error. */
MOEBLAZE_API size_t moeblaze_dispatch_meta_bytes(const moeblaze_shape* s);
MOEBLAZE_API size_t moeblaze_dispatch_workspace_bytes(const moeblaze_shape* s);
/* Activations kept from forward to backward: A = x W1 and (SwiGLU) B = x W2,
 * expert-major with each expert's rows padded to a multiple of 256, in the
 * layer dtype (bf16 with MOEBLAZE_RECOMPUTE_H: followed by one fp32 gate per
 * padded row).  0 for the identity expert. */
MOEBLAZE_API size_t moeblaze_saved_bytes(const moeblaze_shape* s);
MOEBLAZE_API size_t moeblaze_forward_workspace_bytes(const moeblaze_shape* s);
MOEBLAZE_API size_t moeblaze_backward_workspace_bytes(const moeblaze_shape* s);

/*
 * Atomic-free three-step dispatch build (MoEBlaze, awesome-system-papers
 * page, section "Atomic-free 三步 dispatch 构建"):
 *   1. a dense token-expert bitmap (bit-packed, one 32-bit word per expert
 *      per 32 tokens), each (token, expert) bit written once; it is built
 *      per chunk of 1024 tokens in on-chip memory and never stored to HBM;
 *   2. per-(expert, chunk) counts by population count, and from the same
 *      bitmap the in-chunk rank of every (token, slot) (set bits before it
 *      in its expert's row); prefix sums over chunks and experts into
 *      expert_token_offsets;
 *   3. each (token, slot)'s final position = expert offset + chunk base +
 *      in-chunk rank, then parallel writes of the three (L,K)-sized maps.
 * topk_ids: device int32 (L,K) row-major, the router's top-K expert ids.
 * out: the five device buffers above.  ws: device scratch of
 * moeblaze_dispatch_workspace_bytes(s) bytes (contents on entry ignored).
 * validate != 0: synchronise `stream` once and return
 * MOEBLAZE_ERR_BAD_ROUTING if any id is out of range or repeated within a
 * token.  With validate == 0 such ids leave the outputs unspecified (but all
 * writes stay inside the buffers) and the device error word records them
 * (see moeblaze_device_error).
 */
MOEBLAZE_API moeblaze_status moeblaze_dispatch_build(const moeblaze_shape* s, const int32_t* topk_ids,
                                        const moeblaze_dispatch* out, void* ws, size_t ws_bytes,
                                        int validate, moeblaze_stream stream);

/*
 * Dispatch build for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that are handed their input and output buffers and have no way to obtain
 * a scratch buffer: for example a runtime whose device memory is one
 * fixed, fully claimed pool, or code on a path where a new device
 * allocation is not allowed.  It runs the same three-step build as
 * moeblaze_dispatch_build and writes the same outputs into `out`, but keeps
 * its scratch (the in-chunk positions and the per-chunk counts) in a fixed array that
 * lives inside the library: MOEBLAZE_STATIC_SCRATCH_BYTES bytes on every GPU
 * that loads the library, held until the process exits.
 *   - A shape whose scratch would exceed MOEBLAZE_STATIC_SCRATCH_BYTES
 *     (moeblaze_dispatch_workspace_bytes(s) > the limit; roughly
 *     4 * L * K + 4 * E * ceil(L / 1024) bytes) is rejected with
 *     MOEBLAZE_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address on the
 *     current device (a one-time set-up per device); make that first call
 *     before any stream capture.
 *   - Nothing is allocated or freed: no cudaMalloc, no cudaFree.
 *   - Every call, on any stream, shares the one array and it keeps the last
 *     call's contents (the build rewrites every scratch word it reads, so
 *     nothing has to start at zero).  Calls whose GPU work overlaps in time
 *     race on the array: serialise them (one stream, or events).
 * Arguments, outputs, validate and errors are as for moeblaze_dispatch_build.
 */
#define MOEBLAZE_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
MOEBLAZE_API moeblaze_status moeblaze_dispatch_build_static(const moeblaze_shape* s, const int32_t* topk_ids,
                                                         const moeblaze_dispatch* out, int validate,
                                                         moeblaze_stream stream);

/*
 * Forward pass (MoEBlaze, awesome-system-papers page, sections
 * "免物化 token dispatch" (Forward) and "SwiGLU kernel 融合 + activation
 * checkpoint"): for every expert, its rows of x are gathered on the fly
 * through expert_token_indices, W1 and W2 are applied from one load of x,
 * SiLU(a)*b is formed in the GEMM epilogue, and the down-projection output
 * is gate-weighted and reduced into y through the index maps.
 *   x      device (L,d) dtype          gates device (L,K) fp32
 *   disp   as written by moeblaze_dispatch_build for the same ids
 *   W1, W2 device (E,d,h) dtype        W3 device (E,h,d) dtype
 *          (W2 NULL for SiLU; W1, W2, W3 NULL for identity)
 *   y      device (L,d) dtype, overwritten
 *   saved  device moeblaze_saved_bytes(s) bytes: A (and B), overwritten;
 *          needed by moeblaze_backward (NULL allowed when the size is 0)
 *   ws     device moeblaze_forward_workspace_bytes(s) bytes of scratch
 * The fp32 reduction into y sums the K contributions of a token in an
 * unspecified order (bitwise reproducible for K <= 2).
 */
MOEBLAZE_API moeblaze_status moeblaze_forward(const moeblaze_shape* s, const void* x, const float* gates,
                                 const moeblaze_dispatch* disp, const void* W1, const void* W2,
                                 const void* W3, void* y, void* saved, void* ws, size_t ws_bytes,
                                 moeblaze_stream stream);

/*
 * Backward pass of the loss <y, dY> with the routing ids held constant
 * (MoEBlaze, awesome-system-papers page, sections "免物化 token dispatch"
 * (Backward) and "SwiGLU kernel 融合 + activation checkpoint"): dY is
 * gathered to the expert rows through the same indices (no (L*K, d)
 * expansion), SiLU(A) is recomputed from the saved A and B, the two
 * branches' input gradients are accumulated in one accumulator, and dX is
 * reduced back into (L, d).
 *   dY      device (L,d) dtype                 x, gates, disp, W*: as forward
 *   saved   as written by moeblaze_forward.  bf16: consumed - the dH GEMM,
 *           the last reader of A and B, writes dA and dB over them in place
 *           (no separate (rows x 2h) gradient buffer), so after the call it
 *           no longer holds the forward's activations; run the forward again
 *           before another backward.  fp32: left unchanged.
 *   dX      device (L,d) dtype, overwritten
 *   dW1,dW2 device (E,d,h) dtype, overwritten  dW3 device (E,h,d) dtype, overwritten
 *           (dW2 NULL for SiLU; all three NULL for identity)
 *   dgates  device (L,K) fp32, overwritten, or NULL: the gate gradients
 *           dg[t,k] = <dY[t], expert_{ids[t,k]}(x[t])> (y is linear in the
 *           gates), for a router's backward; not on the pages, whose backward
 *           holds the router fixed.  Summed in fp32 over h by float atomic
 *           adds, one per (token, slot) and 256-column tile of h, in the
 *           order the CTAs finish their tiles, so repeated calls can differ
 *           in the last bits (the other bf16 outputs are bitwise repeatable
 *           for K <= 2).
 *   ws      device moeblaze_backward_workspace_bytes(s) bytes of scratch
 */
MOEBLAZE_API moeblaze_status moeblaze_backward(const moeblaze_shape* s, const void* dY, const void* x,
                                  const float* gates, const moeblaze_dispatch* disp,
                                  const void* W1, const void* W2, const void* W3,
                                  void* saved, void* dX, void* dW1, void* dW2, void* dW3,
                                  float* dgates, void* ws, size_t ws_bytes, moeblaze_stream stream);

/* ------------------------------------------------------------------ router
 * The token-choice top-K softmax router, the step before the dispatch
 * (MoEBlaze, awesome-system-papers page, assumptions of the problem
 * statement: token-choice, top-K routing), and its backward, which takes the
 * gate gradients of moeblaze_backward.  Shape fields used: L, d, E, K, dtype
 * (h and act are ignored).  Supported: E <= 256, K <= min(E, 8), d a
 * multiple of 64; otherwise MOEBLAZE_ERR_UNSUPPORTED.  fp32 arithmetic.
 *
 * moeblaze_router_forward:
 *   x       device (L,d) dtype, 16-byte aligned
 *   Wr      device (d,E) fp32 row-major (column e is expert e's weights)
 *   bias    device (E) fp32 or NULL
 *   topk_ids device (L,K) int32, overwritten: the K largest logits
 *           x[t].Wr[:,e] + bias[e], equal logits ordered by the lower expert
 *           index, slot 0 the largest
 *   gates   device (L,K) fp32, overwritten: the softmax over the K selected
 *           logits (they sum to 1 per token)
 * No scratch.  Ready to feed moeblaze_dispatch_build and moeblaze_forward. */
MOEBLAZE_API moeblaze_status moeblaze_router_forward(const moeblaze_shape* s, const void* x, const float* Wr,
                                                     const float* bias, int32_t* topk_ids, float* gates,
                                                     moeblaze_stream stream);

/* Bytes of scratch moeblaze_router_backward needs for shape s (0 when s is
 * not supported). */
MOEBLAZE_API size_t moeblaze_router_backward_workspace_bytes(const moeblaze_shape* s);

/* moeblaze_router_backward: gradients through the router given
 * dgates = dLoss/dgates.  The selection is piecewise constant, so only the
 * selected logits get a gradient: dlogit[t, ids[t,k]] = g_k (dg_k - sum_j
 * g_j dg_j).  Then dWr = x^T dlogit, dbias = sum_t dlogit[t] and
 * dx = dlogit Wr^T (the router's share of the input gradient; the caller
 * adds it to the layer's dX).
 *   x, Wr   as moeblaze_router_forward
 *   topk_ids, gates  device (L,K): the router forward's outputs
 *   dgates  device (L,K) fp32 (moeblaze_backward's dgates)
 *   dWr     device (d,E) fp32, overwritten
 *   dbias   device (E) fp32, overwritten, or NULL
 *   dx      device (L,d) dtype, overwritten, 16-byte aligned, or NULL
 *   ws      device moeblaze_router_backward_workspace_bytes(s) bytes
 * dWr and dbias are summed over the tokens in a fixed order (repeatable to
 * the bit).  Ids must be pairwise distinct per token and < E. */
MOEBLAZE_API moeblaze_status moeblaze_router_backward(const moeblaze_shape* s, const void* x, const float* Wr,
                                                      const int32_t* topk_ids, const float* gates,
                                                      const float* dgates, float* dWr, float* dbias, void* dx,
                                                      void* ws, size_t ws_bytes, moeblaze_stream stream);

/* The router fused with the first step of the dispatch build (MoEBlaze,
 * awesome-system-papers page: the token-choice top-K routing ahead of the
 * section "Atomic-free 三步 dispatch 构建").  One call gives what
 * moeblaze_router_forward followed by moeblaze_dispatch_build on its ids
 * gives: topk_ids and gates as moeblaze_router_forward writes them, and
 * `out` as moeblaze_dispatch_build writes it.
 *   - bf16 x, E <= 64 and L >= 128: one kernel computes the logits on the tensor cores
 *     (Wr split into three bf16 parts, hi + mid + lo, whose products with x
 *     are exact and summed in fp32: the logits carry fp32 precision, though
 *     not the same rounding as moeblaze_router_forward's, so near-equal
 *     logits may be ordered differently), selects the top K, and builds the
 *     dispatch bitmap of each 1024-token chunk in on-chip memory while the
 *     ids are still in registers; the rest of the dispatch build follows.
 *     The ids are not read back from HBM for the bitmap.
 *   - any other router shape (fp32 x, E > 64, L < 128): moeblaze_router_forward, then
 *     moeblaze_dispatch_build's kernels, in the same call.
 * Shape: as for moeblaze_dispatch_build and moeblaze_router_forward (both
 * sets of limits apply).  Arguments as for those two calls; ws: device
 * scratch of moeblaze_router_dispatch_workspace_bytes(s) bytes (contents on
 * entry ignored; 0 for an unsupported shape).  The ids it produces are
 * always valid routing. */
MOEBLAZE_API size_t moeblaze_router_dispatch_workspace_bytes(const moeblaze_shape* s);
MOEBLAZE_API moeblaze_status moeblaze_router_dispatch_build(const moeblaze_shape* s, const void* x, const float* Wr,
                                                            const float* bias, int32_t* topk_ids, float* gates,
                                                            const moeblaze_dispatch* out, void* ws, size_t ws_bytes,
                                                            moeblaze_stream stream);

/* Synchronise `stream` and read the device error word of `disp->meta`:
 * *code = 0 when every kernel since the last dispatch_build on this meta
 * finished normally; otherwise a bitwise OR of 1 (bad routing), 2 (a
 * bounded device-side wait ran out) and 4 (a forward/backward call whose L,
 * E or K differ from the build's).  Returns MOEBLAZE_ERR_BAD_ROUTING,
 * MOEBLAZE_ERR_TIMEOUT or MOEBLAZE_ERR_INVALID_ARG accordingly (in that order
 * of precedence), MOEBLAZE_OK when *code == 0. */
MOEBLAZE_API moeblaze_status moeblaze_device_error(const moeblaze_shape* s, const moeblaze_dispatch* disp,
                                      int32_t* code, moeblaze_stream stream);

/* Host-side check of a dispatch against a shape, on a HOST copy of the
 * first 32 bytes of its meta buffer (the header the build writes): OK when
 * the build was made for s's L, E and K (for L = 0: when it was made for no
 * tokens), MOEBLAZE_ERR_INVALID_ARG otherwise or when meta_header is NULL.
 * The same comparison the forward/backward kernels make on the device. */
MOEBLAZE_API moeblaze_status moeblaze_dispatch_meta_check(const moeblaze_shape* s, const void* meta_header);

/* Diagnostics.
 *
 * moeblaze_set_stage_events: when `events` is non-NULL, later
 * moeblaze_forward / moeblaze_backward calls made from the calling thread
 * record events[i] (each a cudaEvent_t created by the caller) on the call's
 * stream at the stage boundaries of the bf16/fp32 expert paths:
 *   forward : [0] before the up-projection, [1] after it, [2] after the
 *             down-projection + combine, [3] after the final conversion;
 *   backward: [0] before the dH GEMM, [1] after it, [2] after the dX GEMM,
 *             [3] after the dW1/dW2 GEMM, [4] after the dW3 GEMM,
 *             [5] after the final conversion; bf16 with MOEBLAZE_RECOMPUTE_H
 *             the dW3 GEMM runs first: [0] before it, [1] after it, [2]
 *             after dH, [3] after dX, [4] after dW1/dW2, [5] after the
 *             conversion.
 * Only the first `n` events are recorded.  NULL switches recording off.
 *
 * moeblaze_kernel_launches: number of CUDA kernels this library has launched
 * in the process so far (memsets and copies not counted). */
MOEBLAZE_API void moeblaze_set_stage_events(void** events, int32_t n);
MOEBLAZE_API int64_t moeblaze_kernel_launches(void);

/* Failure-path test hook (for tests; not for production runs).
 *
 * moeblaze_set_fault_injection: later calls made from the calling thread run
 * their bf16 expert GEMMs with `wait_limit_ns` as the limit of every bounded
 * device-side wait (> 0; 0 restores the default of 4 s).  With withhold != 0
 * the down projection of a later moeblaze_forward (default mode, not
 * MOEBLAZE_RECOMPUTE_H) issues nothing for the first stage of each CTA's
 * first tile, so that stage's barrier is never completed: the CTA's MMA wait
 * runs out after the limit, the CTA records bit 2 (timeout) in the device
 * error word, lets the copies it has in flight land, frees its tensor memory
 * and returns; moeblaze_device_error then returns MOEBLAZE_ERR_TIMEOUT.  The
 * GPU context stays usable and the next dispatch build clears the word.
 * (0, 0) switches the hook off. */
MOEBLAZE_API void moeblaze_set_fault_injection(int64_t wait_limit_ns, int32_t withhold);

/* Static description of a status code. */
MOEBLAZE_API const char* moeblaze_status_string(moeblaze_status st);

/* Library version, major*10000 + minor*100 + patch. */
MOEBLAZE_API int32_t moeblaze_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEBLAZE_H */
