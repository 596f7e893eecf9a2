/*
 * qsmoe: the quantized sparse mixture-of-experts FFN layer of a
 * Qwen3.6-35B-A3B-style model, as a C ABI over hand-written CUDA kernels
 * for sm_103a (GB300).
 *
 * The layer, in the terms of the pages it follows:
 *   "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026),
 *     section "Qwen creates three distinct workload shapes": a router scores
 *     256 experts per token and selects eight, next to a shared expert that
 *     processes every token;
 *     section "Keeping expert routing on the GPU": a histogram of the
 *     assignments per expert, a prefix scan into start offsets, a scatter
 *     of the rows into their expert groups and a block map of fixed-size
 *     row blocks, all without a host round trip;
 *     section "Dequantizing weights during matrix multiplication": 4-bit
 *     affine weights in groups of 64 with a scale and a bias, expanded on
 *     chip tile by tile, fp32 accumulation;
 *     section "Reducing intermediate and state traffic": the two input
 *     projections fused with their gated activation, and the output
 *     projection fused with its routing score and the shared expert;
 *   "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", section
 *     "融合原理": gate and up weights concatenated along the output axis in
 *     [gate, up] order, one quantized matmul, per-row bit-identical results;
 *   "Ember: packed Q8 decode" (voidwest.dev): the Q8_0 row format, 32 int8
 *     codes with one fp16 scale.
 *
 * Conventions (every entry point):
 *  - Pointers named in the argument lists are DEVICE pointers unless said
 *    otherwise; all arrays are dense row-major.  bf16 and fp16 values are
 *    passed as their 16-bit patterns (uint16_t).
 *  - The caller owns every buffer, including workspaces, and the stream.
 *    The library allocates nothing, never synchronises the stream and never
 *    reads device data on the host: every call only enqueues work on
 *    `stream` (stream-ordered, capturable into a CUDA graph).
 *  - The return value reports argument errors, found synchronously before
 *    anything is enqueued, and launch errors.  Problems only visible on the
 *    device (an expert id out of range, a non-finite logit, an fp16 operand
 *    out of range) are OR-ed into *dev_status as QSM_DEV_* bits; the kernels
 *    then skip the offending item and never trap.  *dev_status is never
 *    cleared by the library; the caller zeroes it and reads it after the
 *    stream has synchronised.
 *  - Pointers must be 16-byte aligned, except dev_status and logit_bias
 *    (4-byte).
 */
#ifndef QSMOE_H
#define QSMOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSM_ABI_VERSION 4

#if defined(__GNUC__)
#define QSM_API __attribute__((visibility("default")))
#else
#define QSM_API
#endif

typedef enum {
  QSM_OK = 0,
  QSM_ERR_INVALID_ARGUMENT = 1, /* null / misaligned pointer, bad size */
  QSM_ERR_UNSUPPORTED = 2,      /* valid but not implemented (shape, type) */
  QSM_ERR_WORKSPACE_TOO_SMALL = 3,
  QSM_ERR_CUDA = 4              /* a CUDA launch or runtime call failed */
} qsm_status;

/* Bits of the device status word. */
#define QSM_DEV_BAD_EXPERT_ID 1 /* topk_idx entry outside [0, E) */
#define QSM_DEV_NONFINITE 2     /* non-finite router logit */
#define QSM_DEV_FP16_RANGE 4    /* a value staged in fp16 overflowed */
#define QSM_DEV_TIMEOUT 8       /* a bounded wait (on a copy, or on the
                                   tagged logits or h of
                                   moe_decode_layer) ran out: the kernel
                                   returned, its results are invalid */

typedef enum { QSM_Q8_0 = 0, QSM_AFFINE4_G64 = 1 } qsm_qtype;

/* A quantized weight tensor of shape [experts, rows, cols], rows = outputs,
 * cols = inputs (reduction axis).
 *  QSM_Q8_0:        codes int8 [experts, rows, cols]; scales fp16
 *                   [experts, rows, cols/32]; weight = code * scale of its
 *                   block of 32 inputs.  biases must be NULL.
 *  QSM_AFFINE4_G64: codes uint32 [experts, rows, cols/8], input c stored in
 *                   bits 4*(c%8)..4*(c%8)+3 of word c/8; scales and biases
 *                   fp16 [experts, rows, cols/64]; weight = scale*code + bias
 *                   for its group of 64 inputs. */
typedef struct {
  int32_t qtype;
  int32_t experts, rows, cols;
  const void* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} qsm_qweights;

/* One MoE FFN layer: hidden size H, expert (and shared expert) intermediate
 * size I, E routed experts of which each token uses k.
 *   gate_up        [E, 2I, H]  rows 0..I-1 gate, rows I..2I-1 up
 *   down           [E, H, I]
 *   shared_gate_up [1, 2I, H], shared_down [1, H, I]
 *   shared_gate    [H] fp32, or NULL: the shared expert's output of token t
 *                  is scaled by sigmoid(x[t] . shared_gate) (a gated shared
 *                  expert); NULL keeps weight 1 (the pages' shared expert).
 * All four tensors must share one qtype.  Requires H % 64 == 0,
 * I % 64 == 0, 1 <= k <= E <= 1024, shared_gate 16-byte aligned. */
typedef struct {
  int32_t H, I, E, k;
  qsm_qweights gate_up, down, shared_gate_up, shared_down;
  const float* shared_gate;
} qsm_moe_layer;

/* The token grouping produced by moe_group_tokens (all device arrays).
 * Assignment a = t*k + j is token t's j-th selected expert.
 *   counts   [E]     assignments per expert
 *   offsets  [E+1]   exclusive prefix sum of counts (offsets[E] = T*k when
 *                    every expert id is valid)
 *   perm     [T*k]   assignment at each sorted position, sorted by
 *                    (expert, assignment id): stable
 *   inv_perm [T*k]   sorted position of each assignment, -1 if its expert
 *                    id is invalid
 *   tile_map [2*max_tiles]  (expert, first sorted row) of every block of at
 *                    most tile_rows rows of one expert, experts ascending;
 *                    entries n_tiles .. max_tiles-1 are set to (-1, -1)
 *   n_tiles  [1]     number of blocks written (stays on the device)
 * tile_rows and max_tiles are host values chosen by the caller:
 * max_tiles >= moe_group_max_tiles(T, k, E, tile_rows), tile_rows as
 * returned by moe_ffn_tile_rows() when the grouping feeds moe_ffn_forward. */
typedef struct {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* tile_map;
  int32_t* n_tiles;
  int32_t tile_rows;
  int32_t max_tiles;
} qsm_grouping;

/* ----------------------------------------------------------------- router */

/* Bytes of workspace moe_route needs for T tokens, hidden size H and E
 * experts. */
QSM_API size_t moe_route_workspace_bytes(int32_t T, int32_t H, int32_t E);

/* Route flags (the `renormalize` argument of the routing calls). */
#define QSM_ROUTE_RENORMALIZE 1      /* weights: softmax over the selection */
#define QSM_ROUTE_BIAS_SELECT_ONLY 2 /* logit_bias picks experts, not weights */

/* Router: logits l[t,e] = sum_h x[t,h] * w_router[e,h] (fp32 accumulation)
 * and selection logits s[t,e] = l[t,e] + logit_bias[e]; per token the k
 * largest s (ties to the lower expert index) in descending order, and their
 * weights from w = s, or w = l with QSM_ROUTE_BIAS_SELECT_ONLY:
 *   QSM_ROUTE_RENORMALIZE set:   softmax of w over the k selected experts;
 *   QSM_ROUTE_RENORMALIZE clear: softmax of w over all E, at the selected.
 * (`renormalize` is these flags; 0 and 1 keep their old meaning.)
 * [Perplexity page, "Qwen creates three distinct workload shapes".]
 *   x          [T, H] bf16
 *   w_router   [E, H] fp32
 *   logit_bias [E] fp32 or NULL (added to the logits before selection)
 *   topk_idx   [T, k] int32 (out), topk_w [T, k] fp32 (out)
 *   workspace  >= moe_route_workspace_bytes(T, H, E) bytes.  It must hold
 *              zeros before its first use; every call leaves the part that
 *              must start at zero zeroed again.
 * Few tokens run on CUDA cores (fp32 FMA); many tokens (T > 64, E a multiple
 * of 16 up to 256, k <= 8) run one tcgen05 GEMM over an exact three-way
 * bf16 split of w_router, which keeps fp32-accurate logits.
 * Requires H % 64 == 0, 1 <= k <= min(E, 32), E <= 1024, T >= 0, no flag
 * bits beyond the two above.  A non-finite logit sets QSM_DEV_NONFINITE. */
QSM_API qsm_status moe_route(const uint16_t* x, const float* w_router,
                     const float* logit_bias, int32_t T, int32_t H, int32_t E,
                     int32_t k, int32_t renormalize, int32_t* topk_idx,
                     float* topk_w, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, cudaStream_t stream);

/* --------------------------------------------------------------- grouping */

/* Upper bound on the number of blocks of tile_rows rows over any routing:
 * n + floor((T*k - n) / tile_rows) with n = min(E, T*k). */
QSM_API int32_t moe_group_max_tiles(int32_t T, int32_t k, int32_t E,
                            int32_t tile_rows);

/* Histogram, exclusive scan, stable scatter and block map of the
 * assignments [Perplexity page, "Keeping expert routing on the GPU"]; see
 * qsm_grouping for the outputs.  An expert id outside [0, E) sets
 * QSM_DEV_BAD_EXPERT_ID; that assignment is left out of every group
 * (inv_perm = -1) and the FFN skips it.
 * Requires 1 <= k, E <= 1024, tile_rows >= 1, T*k <= 2^24. */
QSM_API qsm_status moe_group_tokens(const int32_t* topk_idx, int32_t T, int32_t k,
                            int32_t E, const qsm_grouping* g,
                            int32_t* dev_status, cudaStream_t stream);

/* moe_route followed by moe_group_tokens in one launch, for a few tokens
 * (decode): topk_idx, topk_w and every array of g are the same bits as the
 * two calls give.  The router's CTAs split the experts as in moe_route; the
 * CTA that finishes last selects the top k and then builds the grouping of
 * the T*k assignments from the ids it holds in shared memory
 * [Perplexity page, "Qwen creates three distinct workload shapes" and
 * "Keeping expert routing on the GPU"].
 *   workspace  as for moe_route (moe_route_workspace_bytes(T, H, E)).
 * Supported: 1 <= T <= 8, H % 64 == 0, 1 <= E <= 256, 1 <= k <= min(E, 32);
 * otherwise returns QSM_ERR_UNSUPPORTED and enqueues nothing (use the two
 * calls).  Argument errors as for the two calls. */
QSM_API qsm_status moe_route_group(const uint16_t* x, const float* w_router,
                                   const float* logit_bias, int32_t T, int32_t H,
                                   int32_t E, int32_t k, int32_t renormalize,
                                   int32_t* topk_idx, float* topk_w,
                                   const qsm_grouping* g, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status,
                                   cudaStream_t stream);

/* -------------------------------------------------------------------- FFN */

/* The tile_rows moe_ffn_forward expects in its grouping for T tokens. */
QSM_API int32_t moe_ffn_tile_rows(int32_t T);

/* Bytes of workspace moe_ffn_forward needs for layer L and T tokens. */
QSM_API size_t moe_ffn_workspace_bytes(const qsm_moe_layer* L, int32_t T);

/* The expert FFNs and the combine:
 *   for every assignment (t, j) with expert e = topk_idx[t, j]:
 *     gu = W_gate_up[e] x[t]            (one fused quantized matmul)
 *     h  = silu(gu[:I]) * gu[I:]        (SwiGLU, silu(g) = g / (1 + e^-g))
 *     o  = W_down[e] h
 *   the same for the shared expert, then
 *     y[t] = sum_j topk_w[t, j] * o(t, j) + o_shared(t)
 * [Perplexity page, "Reducing intermediate and state traffic"; oMLX page,
 * "融合原理" and "前向传播补丁"].
 *   x          [T, H] bf16;  y [T, H] bf16 (out, round-to-nearest-even of
 *              the fp32 result);  y_f32 [T, H] fp32 (out, optional: the
 *              same result before rounding, for parity checks) or NULL
 *   topk_idx, topk_w  as written by moe_route;  g as written by
 *              moe_group_tokens for the same topk_idx, with tile_rows ==
 *              moe_ffn_tile_rows(T)
 *   workspace  >= moe_ffn_workspace_bytes(L, T) bytes, no initial content.
 * T <= 64 runs the decode kernels (weight streaming GEMV), larger T the
 * grouped-GEMM prefill kernels (tcgen05, weights of either type expanded to
 * fp16 tile by tile on chip; they need H % 256 == 0 and I % 128 == 0, else
 * QSM_ERR_UNSUPPORTED). */
QSM_API qsm_status moe_ffn_forward(const qsm_moe_layer* L, const uint16_t* x,
                           int32_t T, const int32_t* topk_idx,
                           const float* topk_w, const qsm_grouping* g,
                           uint16_t* y, float* y_f32, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status,
                           cudaStream_t stream);

/* ------------------------------------------------------------ whole layer */

/* Bytes of workspace moe_layer_forward needs for T tokens in chunks of at
 * most `chunk` tokens (sized for one chunk: the router's, the grouping's
 * and the FFN's workspaces of the largest chunk).  0 if the layer is
 * unsupported or an argument is invalid. */
QSM_API size_t moe_layer_workspace_bytes(const qsm_moe_layer* L, int32_t T,
                                         int32_t chunk);

/* The whole layer: moe_route -> moe_group_tokens -> moe_ffn_forward over the
 * tokens in consecutive chunks of at most `chunk` tokens, all enqueued on
 * `stream` [Perplexity page, "Qwen creates three distinct workload shapes"
 * (long prompts in chunks) and "Keeping expert routing on the GPU"].  A
 * token's routing does not depend on the chunking; its output differs
 * between chunkings at most by the order of the prefill combine's fp32
 * additions (or by the decode / prefill kernel choice of its chunk's size).
 *   x [T, H] bf16;  w_router [E, H] fp32;  logit_bias [E] fp32 or NULL;
 *   topk_idx [T, k] int32 and topk_w [T, k] fp32 (out);  y [T, H] bf16 (out);
 *   y_f32 [T, H] fp32 (out) or NULL;
 *   workspace  >= moe_layer_workspace_bytes(L, T, chunk) bytes; it must hold
 *              zeros before its first use, and every call leaves it so.
 * Errors as for the three calls. */
QSM_API qsm_status moe_layer_forward(const qsm_moe_layer* L, const uint16_t* x,
                                     int32_t T, int32_t chunk,
                                     const float* w_router,
                                     const float* logit_bias, int32_t renormalize,
                                     int32_t* topk_idx, float* topk_w,
                                     uint16_t* y, float* y_f32, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_status,
                                     cudaStream_t stream);

/* The whole layer for a few tokens (1 <= T <= 8) in one launch: router,
 * selection, gate_up + SwiGLU, down + combine, separated by grid-wide
 * exchanges of call-tagged words (the logits, then h between gate_up and
 * down), instead of three dependent launches
 * [Perplexity page, "Keeping expert routing on the GPU", "Reducing
 * intermediate and state traffic", "Overlapping independent GPU work"].  Results: topk_idx and topk_w
 * bit-identical to moe_route's; y the layer output as moe_ffn_forward
 * computes it (same arithmetic per product; the combine's fp32 additions in
 * another order).
 *   Arguments as for moe_layer_forward, without a chunk size.
 *   Supported: Q8_0 or affine-4 (all four weight planes alike), H % 256 ==
 *   0, H / 16 <= the device's SM count (a CTA per SM, at least one per 16
 *   output rows, all resident for the two exchanges),
 *   I % 128 == 0 (Q8_0) or % 256 == 0
 *   (affine-4), E <= 1024, k <= 32; all pointers 16-byte aligned except
 *   topk_idx, topk_w, y, y_f32 and logit_bias (4 bytes).  Otherwise
 *   QSM_ERR_UNSUPPORTED (moe_layer_forward serves every shape).
 *   workspace  >= moe_decode_layer_workspace_bytes(L, T) bytes, zeros before
 *              its first use.  Its first 8 bytes count calls (one arrival
 *              per CTA): the calls that share a workspace must have the
 *              same layer shape (H, I, E, k), and after a
 *              QSM_DEV_TIMEOUT it must be zeroed again.
 *              From byte 256: the tagged logits [8, E] (64-bit words, the
 *              call's tag in the high half), then h as 64-bit words (tag,
 *              two fp16 values).
 * Every wait in the kernel is bounded: an exchange or copy that
 * does not complete sets QSM_DEV_TIMEOUT and the call's results are
 * invalid. */
QSM_API size_t moe_decode_layer_workspace_bytes(const qsm_moe_layer* L, int32_t T);

/* The check moe_decode_layer makes before it launches, with the device's
 * figures passed in: 1 when the layer and T are supported on a device of
 * `sm_count` SMs and the kernel's whole grid (one CTA per SM, at least one
 * per 16 rows of y) can be resident at once with `blocks_per_sm` CTAs per
 * SM, else 0.  moe_decode_layer takes sm_count from the current device and
 * blocks_per_sm from the occupancy calculator at the call's shared-memory
 * size; when the check fails it returns QSM_ERR_UNSUPPORTED (and
 * moe_decode_layer_workspace_bytes returns 0), so that callers take the
 * route / group / FFN launches instead.  The check cannot see SMs that other
 * work holds while the kernel runs (another stream, MPS limits): there the
 * bounded waits run out and the call reports QSM_DEV_TIMEOUT with invalid
 * results.  Pure host logic; needs no GPU. */
QSM_API int32_t qsm_decode_layer_fits(const qsm_moe_layer* L, int32_t T, int32_t sm_count,
                                      int32_t blocks_per_sm);
QSM_API qsm_status moe_decode_layer(const qsm_moe_layer* L, const uint16_t* x, int32_t T,
                                    const float* w_router, const float* logit_bias,
                                    int32_t flags, int32_t* topk_idx, float* topk_w,
                                    uint16_t* y, float* y_f32, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status,
                                    cudaStream_t stream);

/* moe_ffn_forward without a workspace argument, for callers that cannot
 * allocate device memory (code running inside another runtime's memory
 * pool, latency-critical threads where an allocation and the device
 * synchronisation it may cause are not allowed, hosts that own only the
 * activations and the stream).  The pages have no counterpart: this is an
 * interface convenience of this library, not a step of the method.
 *   Arguments and results are those of moe_ffn_forward.  The scratch comes
 *   from an array inside the library (1 MiB per device, held by every GPU
 *   that loads the library until the process exits), so T must be <= 64 and
 *   the scratch that moe_ffn_forward would need for this call
 *   (moe_ffn_workspace_bytes(L, T) on the path in force: the decode path's
 *   h, (T*k + T) * I * 2 bytes, and T fp32 shared-expert gates) must fit in
 *   1 MiB; otherwise QSM_ERR_UNSUPPORTED is returned and nothing is
 *   enqueued.  T < 0 is QSM_ERR_INVALID_ARGUMENT; T == 0 enqueues nothing.
 *   The call allocates nothing.  `stream` must belong to the current
 *   device (else QSM_ERR_INVALID_ARGUMENT): the scratch used is that
 *   device's copy.  The first call on each device looks up that device's
 *   copy of the array; make that first call before any stream capture.  The
 *   address found stays in use for the life of the device's context: calls
 *   after cudaDeviceReset are not supported.  All calls on a device share
 *   the one array and it keeps the last call's contents (no value has to
 *   start at zero); calls whose work overlaps on the GPU (different
 *   streams, or different threads without ordering) race on it and must be
 *   serialised by the caller. */
QSM_API qsm_status moe_ffn_forward_noalloc(const qsm_moe_layer* L,
                                           const uint16_t* x, int32_t T,
                                           const int32_t* topk_idx,
                                           const float* topk_w,
                                           const qsm_grouping* g, uint16_t* y,
                                           float* y_f32, int32_t* dev_status,
                                           cudaStream_t stream);

/* ------------------------------------------------------------ dense GEMV */

/* Batch-1 Q8_0 projection y[n] = sum_c q[n,c] * d[n, c/32] * x[c]
 * [Perplexity page, "Optimizing the single-row weight path"; Ember page,
 * Q8_0 rows].
 *   x [K] bf16;  q [N, K] int8;  d [N, K/32] fp16;  y [N] bf16 (out).
 * Requires K % 64 == 0, 64 <= K <= 16384, N >= 1; x, q, d, y 16-byte
 * aligned.  With K % 256 == 0 the weight tiles arrive by TMA copies whose
 * waits are bounded: a copy that never completes sets QSM_DEV_TIMEOUT in
 * *dev_status (which may be NULL: nothing is reported then).  A row's
 * result does not depend on N (K is summed in fixed 512-wide segments, in
 * segment order). */
QSM_API qsm_status q8_gemv(const uint16_t* x, const int8_t* q, const uint16_t* d,
                   int32_t N, int32_t K, uint16_t* y, int32_t* dev_status,
                   cudaStream_t stream);

/* Int8-activation mode of the Q8_0 GEMV ["Ember: packed Q8 decode": the
 * projections that read one activation share its quantization, and the dot
 * products run on 8-bit groups].  Reading: blocks of 32 inputs, per block
 * an fp32 scale dx = max|x| / 127 and codes qx = round-half-away(x / dx)
 * clamped to [-127, 127] (fp32 arithmetic; an all-zero block has dx = 0).
 *   q8_quantize_x:  x [K] bf16 -> qx [K] int8 (out), dx [K/32] fp32 (out);
 *                   K % 32 == 0.
 *   q8_gemv_i8:     y[n] = sum_b d[n,b] * dx[b] * sum_{c in b} q[n,c] * qx[c]
 *                   (each block's integer dot product exact, the rest fp32),
 *                   y [N] bf16 (out); N >= 1, K % 64 == 0, K <= 16384, qx,
 *                   q, d, y 16-byte aligned.  A row's result does not depend
 *                   on N.
 * This changes the numerics against q8_gemv by the activation's rounding
 * (at most half a step dx/2 per input). */
QSM_API qsm_status q8_quantize_x(const uint16_t* x, int32_t K, int8_t* qx, float* dx,
                                 int32_t* dev_status, cudaStream_t stream);
QSM_API qsm_status q8_gemv_i8(const int8_t* qx, const float* dx, const int8_t* q,
                              const uint16_t* d, int32_t N, int32_t K, uint16_t* y,
                              int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------ misc */

/* Static description of a status code. */
QSM_API const char* qsm_status_str(qsm_status s);

/* QSM_ABI_VERSION of the loaded library. */
QSM_API int32_t qsm_abi_version(void);

/* Kernels this library has launched since it was loaded, process-wide:
 * every launch of every entry point counts once, including launches
 * recorded into a CUDA graph under stream capture (a replay of the graph
 * launches them again without counting).  Never fails. */
QSM_API uint64_t qsm_launch_count(void);

/* Test hook: 0 = choose the FFN path by T (default), 1 = always the decode
 * kernels, 2 = always the prefill kernels (when T allows).  Process-wide. */
QSM_API qsm_status qsm_debug_force_path(int32_t mode);

/* Test hook for the bounded waits: make moe_decode_layer's logit exchange
 * wait for a call tag `skew` ahead of the call's own (0 = off, the
 * default), so that no call can complete it: every wait runs out, the kernel sets QSM_DEV_TIMEOUT
 * in *dev_status, finishes with invalid results and returns, and the
 * context stays usable.  The call ticket stays consistent (every CTA still
 * arrives once).  Process-wide; skew in [0, 1024]. */
QSM_API qsm_status qsm_debug_barrier_skew(int32_t skew);

/* Test hook for the per-row identity of the fused gate_up projection
 * ("oMLX MoE gate/up 融合优化", "融合原理": the rows of the [gate; up]
 * concatenation come out bit-identical to separate gate and up
 * projections).  With buf set (a device buffer of n_floats fp32), every
 * kernel that computes gate_up also writes, before SwiGLU, the fp32 gate
 * value of intermediate i to buf[row * 2I + i] and the up value to
 * buf[row * 2I + I + i], where row is the row of h the kernel writes:
 *   moe_ffn_forward (decode and prefill paths): the sorted assignment row
 *     (< T*k), then T*k + t for token t of the shared expert: at least
 *     (T*k + T) * 2I floats;
 *   moe_decode_layer: slot * T + t, slot 0 the shared expert and slots
 *     1.. the distinct selected experts in ascending id order: at least
 *     (min(E, T*k) + 1) * T * 2I floats.
 * A call whose buffer is too small returns QSM_ERR_INVALID_ARGUMENT.
 * buf = NULL, n_floats = 0 turns the hook off.  Process-wide, not
 * thread-safe; for tests only. */
QSM_API qsm_status qsm_debug_gu_dump(float* buf, size_t n_floats);

#ifdef __cplusplus
}
#endif

#endif /* QSMOE_H */
