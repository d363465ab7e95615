/*
 * moe.h -- C ABI of libmoe.so: the forward pass of a Mixtral-style sparse
 * mixture-of-experts feed-forward layer on one NVIDIA B300 (sm_103a).
 *
 * What the layer computes (Mixtral of Experts, arXiv 2401.04088, as given on
 * the paper-graph-ui summary, section 3.4 "MoE Layer Formulation", and the
 * xyznot reading guide, "Method (with the key equations)"):
 *
 *   logits  l = x . W_g                          (router, no bias)
 *   G(x)    = Softmax(TopK(l))                   (TopK keeps the K largest, -inf elsewhere)
 *   E_i(x)  = (SiLU(x . W1[i]) (.) (x . W3[i])) . W2[i]     SiLU(z) = z sigma(z)
 *             ("Expert Network Structure (SwiGLU)", written here in row-vector
 *             form: W1 is the SiLU branch, W3 the linear branch, W2 the down
 *             projection)
 *   y       = sum_i G(x)_i . E_i(x)              (only the K selected experts compute)
 *
 * Choices the pages leave open, fixed here:
 *   - equal logits rank by lower expert index (for every TopK position);
 *   - slot 0 of a token is its larger logit;
 *   - router, TopK and the softmax run in fp32; the expert GEMMs take bf16
 *     operands with fp32 accumulation; the SwiGLU hidden activations are
 *     stored as bf16; the per-slot expert outputs are fp32 and summed in a
 *     fixed order (slot 0 then slot 1), so results are bitwise reproducible.
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise, on
 *     the current CUDA device, 16-byte aligned, to a dense row-major tensor.
 *   - dtype selects the element type shared by x, W_g, W1, W3, W2 and y:
 *     MOE_BF16 (tensor-core path) or MOE_F32 (exact fp32 SIMT path, no TF32).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) except moe_read_status, which synchronises it.
 *   - The caller owns and allocates every buffer, including the workspace.
 *     The library allocates no device memory and keeps no per-call state; its
 *     only global state is a cached device-attribute table.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     failed check returns an error code and launches nothing.  Launch
 *     failures map to MOE_ERR_CUDA.  Errors found on the device (a bounded
 *     wait that expired, an out-of-range index, non-finite router input under
 *     MOE_DEBUG_CHECKS) are written to a status word in the workspace and read
 *     with moe_read_status.  Nothing in the library calls exit() or abort().
 *   - Inputs must be finite.  NaN or Inf in x or W_g gives unspecified
 *     routing (reported as MOE_ERR_NONFINITE under MOE_DEBUG_CHECKS).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

/* Status codes (plain int in every signature). */
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, aliasing */
  MOE_ERR_UNSUPPORTED = 2,     /* valid but not implemented (dtype, E, K, device) */
  MOE_ERR_WORKSPACE = 3,       /* workspace pointer null or smaller than required */
  MOE_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait expired */
  MOE_ERR_NONFINITE = 6,       /* NaN/Inf router logit (MOE_DEBUG_CHECKS only) */
  MOE_ERR_DEVICE_BOUNDS = 7    /* device-side index check failed (MOE_DEBUG_CHECKS only) */
};

/* Element types.  MOE_FP8_E4M3 names the e4m3-weight variant (bf16 tokens,
 * router and output; e4m3 expert weights and expert-GEMM activations): it is
 * the dtype of moe_workspace_bytes for moe_forward_fp8. */
enum { MOE_BF16 = 0, MOE_F32 = 1, MOE_FP8_E4M3 = 2 };

/* moe_forward flags. */
#define MOE_ACCUMULATE   0x1u  /* y += MoE(x) instead of y = MoE(x) (residual stream) */
#define MOE_DEBUG_CHECKS 0x2u  /* device-side range and finiteness checks */
/* Failure-path test hook (bf16 only): the gate/up expert GEMM first waits on a
 * barrier that nothing signals, so its bounded wait expires after about one
 * second; the kernel then stops issuing, drains its own copies and MMAs, frees
 * its tensor memory and returns, and the call's status word reads
 * MOE_ERR_DEVICE_TIMEOUT.  The outputs of such a call are unspecified; the
 * context stays usable.  With MOE_F32 the flag is rejected (that path has no
 * waits). */
#define MOE_DEBUG_FORCE_TIMEOUT 0x4u
/* Expert-GEMM form overrides, for measurements (the results are bitwise the
 * same in every form; ignored when the gate/up contraction is split, i.e. for
 * decode-sized batches).  By default batches whose experts average 16 or
 * more 128-row tiles use CTA-pair MMAs (tcgen05 cta_group::2, 256x256 tiles)
 * and all others use pairs of 128x256 tiles sharing one operand by TMA
 * multicast. */
#define MOE_GEMM_PAIR_MMA 0x8u   /* CTA-pair MMAs (256x256 tiles) */
#define MOE_GEMM_QUAD     0x10u  /* 2x2 tiles per 4-CTA cluster, both operands multicast */
#define MOE_GEMM_MULTICAST_PAIRS 0x20u  /* pairs of 128x256 tiles, one operand multicast */

/*
 * Workspace size in bytes for moe_forward / moe_route with these sizes, or 0
 * if the sizes are invalid or unsupported.  The layout depends only on the
 * arguments, so one buffer can be reused for every call with the same sizes.
 * It holds the status word, the routing table, the expert grouping and the
 * grouped activations; at T = 4096, d = 4096, f = 14336, E = 8, K = 2, bf16
 * it is about 0.5 GB (including a [T, d] buffer for moe_block_forward).
 */
MOE_API size_t moe_workspace_bytes(int T, int d, int f, int E, int K, int dtype);

/*
 * Number of kernels one moe_forward (dtype MOE_BF16 or MOE_F32) or
 * moe_forward_fp8 (dtype MOE_FP8_E4M3) call with these sizes enqueues: the
 * router and the grouping (one launch for T <= 256, two above), the row
 * gather, the two expert GEMMs, one more for e4m3 (the H quantiser), and a
 * combine kernel unless the down GEMM's epilogue forms y (bf16 and e4m3 calls
 * whose down projection is not split over its contraction, or with T <= 4);
 * 0 for T = 0 or
 * invalid sizes.  Host only.
 */
MOE_API int moe_forward_launches(int T, int d, int f, int E, int K, int dtype);

/*
 * The MoE layer forward pass: y = sum over the K selected experts of
 * gate * SwiGLU_expert(x) (section 3.4 "MoE Layer Formulation", output
 * combination; "Expert Network Structure (SwiGLU)").
 *
 *   x   [T, d]      input tokens
 *   Wg  [d, E]      router weights
 *   W1  [E, d, f]   SiLU-branch projections
 *   W3  [E, d, f]   linear-branch projections
 *   W2  [E, f, d]   down projections
 *   y   [T, d]      output; must not overlap x.  With MOE_ACCUMULATE, y is
 *                   read and the layer output is added to it (in fp32, then
 *                   rounded to dtype).
 *   T >= 0 (T = 0 returns MOE_OK at once; x, y, workspace may then be NULL),
 *   1 <= K <= 2, K <= E <= 32,
 *   d, f >= 1 and multiples of 8 (bf16) or 4 (f32).
 *   workspace / ws_bytes: device buffer of at least moe_workspace_bytes().
 *     Calls sharing one workspace must be ordered on the GPU (same stream or
 *     synchronised); concurrent calls need separate workspaces.
 *   flags: MOE_ACCUMULATE | MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT | one MOE_GEMM_* form.
 * Returns MOE_OK once every kernel is enqueued.
 */
MOE_API int moe_forward(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                void *y, int T, int d, int f, int E, int K, int dtype,
                void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * moe_forward with per-stage device timestamps, for kernel durations measured
 * inside a timed run without separating the kernels: the same kernels, work
 * and results as moe_forward.  Each kernel also reads the GPU's global
 * nanosecond timer: every CTA of the kernel of stage s lowers stamps[s] to the
 * time it starts its work (after waiting for its inputs) and raises
 * stamps[MOE_NUM_STAGES + s] to the time it finishes, so for a stage that ran,
 * stamps[MOE_NUM_STAGES + s] - stamps[s] is its kernel's span in ns.
 *   stamps: DEVICE array of 2 * MOE_NUM_STAGES unsigned 64-bit integers,
 *           8-byte aligned, owned by the caller, who initialises it before
 *           the call (begin times to all ones, end times to zero; the call
 *           itself enqueues nothing extra), so a stage that did not run
 *           reads (UINT64_MAX, 0).
 *   Stages: MOE_STAGE_ROUTE router; MOE_STAGE_GROUP grouping; MOE_STAGE_GATHER
 *           row gather (e4m3: gather and quantise); MOE_STAGE_GATE_UP gate/up
 *           expert GEMM with SwiGLU; MOE_STAGE_QUANT_H quantisation of H
 *           (e4m3 only); MOE_STAGE_DOWN down expert GEMM (x gate; and, when
 *           unsplit, the combine); MOE_STAGE_COMBINE combine kernel (split
 *           down projections and fp32); MOE_STAGE_NORM RMSNorm
 *           (moe_block_forward_stamped only).
 * Returns MOE_ERR_INVALID_ARG if stamps is NULL or misaligned; otherwise as
 * moe_forward.  Calls sharing one stamps array must be ordered on the GPU.
 */
#define MOE_NUM_STAGES 8
enum {
  MOE_STAGE_ROUTE = 0, MOE_STAGE_GROUP = 1, MOE_STAGE_GATHER = 2, MOE_STAGE_GATE_UP = 3,
  MOE_STAGE_QUANT_H = 4, MOE_STAGE_DOWN = 5, MOE_STAGE_COMBINE = 6, MOE_STAGE_NORM = 7
};
MOE_API int moe_forward_stamped(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                      void *y, int T, int d, int f, int E, int K, int dtype,
                      void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                      unsigned long long *stamps);

/*
 * One pre-norm MoE half-block of the attention-free stack, in place:
 *
 *   h <- h + MoE(RMSNorm(h))
 *
 * (paper-graph-ui summary: "Architectural Inheritance from Mistral 7B",
 * RMSNorm before the MoE block; section 3, the MoE output is added to the
 * residual stream).  RMSNorm has unit gain: x_n = h / sqrt(mean(h^2) + eps)
 * per row, fp32 math, rounded to dtype; x_n lives in the workspace.  The MoE
 * part is moe_forward(x_n, ...) with MOE_ACCUMULATE into h, so its results
 * equal moe_rmsnorm followed by that call bit for bit.
 *   h   [T, d]  residual stream, read and updated in place; must not overlap
 *               the workspace.
 *   Wg, W1, W3, W2, T, d, f, E, K, dtype, workspace, ws_bytes, stream: as for
 *   moe_forward (the same workspace size).  eps > 0.
 *   flags: 0 or MOE_DEBUG_CHECKS (accumulation is implied).
 */
MOE_API int moe_block_forward(void *h, const void *Wg, const void *W1, const void *W3, const void *W2,
                      int T, int d, int f, int E, int K, int dtype, float eps,
                      void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);

/* moe_block_forward with the stage timestamps of moe_forward_stamped (the
 * RMSNorm kernel as MOE_STAGE_NORM). */
MOE_API int moe_block_forward_stamped(void *h, const void *Wg, const void *W1, const void *W3, const void *W2,
                      int T, int d, int f, int E, int K, int dtype, float eps,
                      void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                      unsigned long long *stamps);

/*
 * e4m3 expert weights.  The pages name FP8 only as deployment work
 * (paper-graph-ui summary, "Inference and Deployment Infrastructure"), so the
 * scheme is this library's:
 *   e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
 *         largest finite magnitude 448; values round to nearest, ties to the
 *         even code, and saturate at +-448.
 *   weights: from a[e, n] = max_k |W[e, k, n]| per output column n of
 *         each expert bank, the fp32 scale s[e, n] = a / 448 and the factor
 *         u[e, n] = 448 / a (fp32 divisions; both 1 for an all-zero column, a
 *         nonzero a below 2^-100 taken as 2^-100); codes
 *         q[e, n, k] = e4m3(W[e, k, n] * u[e, n]) (one fp32 product),
 *         stored K-contiguous, i.e. transposed from the bf16 bank.
 *   activations: the same with one scale per row, for each grouped token row
 *         (gate/up input) and for each row of the SwiGLU output H after it is
 *         rounded to bf16 (down input).
 * The expert GEMMs multiply e4m3 codes on the tensor cores (fp32
 * accumulation) and apply the row and column scales in their epilogues.
 *
 * moe_quantize_weights_fp8: W [E, K, N] bf16 -> codes Wq (one byte each)
 * and scales [E, N] fp32, all device memory owned by the caller; K, N >= 1.
 * The codes are stored in 128 x 128 tiles, so that the expert GEMMs stream
 * each tile as one contiguous 16 KiB block: Wq is
 * [E, Nt, Kt, 128, 128] with Nt = ceil(N / 128), Kt = ceil(K / 128), and
 * Wq[e, n / 128, k / 128, n % 128, k % 128] = code of W[e, k, n]; codes past
 * N or K are zero.  Its size is moe_fp8_weight_bytes(E, K, N).  For the
 * layer: W1 and W3 ([E, d, f]) give tiles over (N, K) = (f, d) and [E, f]
 * scales, W2 ([E, f, d]) gives tiles over (d, f) and [E, d] scales.
 */
MOE_API int moe_quantize_weights_fp8(const void *W, int E, int K, int N, void *Wq, float *scales,
                             moe_stream_t stream);

/* Bytes of the tiled e4m3 codes of an [E, K, N] bank (0 if a size is below 1). */
MOE_API size_t moe_fp8_weight_bytes(int E, int K, int N);

/*
 * The layer with e4m3 expert weights: y = sum over the K selected experts of
 * gate * SwiGLU_expert(x), as moe_forward, with the expert projections on
 * e4m3 operands (scheme above).  x [T, d], Wg [d, E] and y [T, d] are bf16;
 * W1q, W3q (tiles over f x d) and W2q (tiles over d x f) are e4m3 codes with
 * scales s1, s3 [E, f] and s2 [E, d] from moe_quantize_weights_fp8.  d and f are multiples
 * of 16.  workspace: at least moe_workspace_bytes(T, d, f, E, K,
 * MOE_FP8_E4M3).  flags: as moe_forward.  Other rules as moe_forward.
 */
MOE_API int moe_forward_fp8(const void *x, const void *Wg, const void *W1q, const float *s1, const void *W3q,
                    const float *s3, const void *W2q, const float *s2, void *y, int T, int d, int f, int E,
                    int K, void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);

/* moe_forward_fp8 with the stage timestamps of moe_forward_stamped. */
MOE_API int moe_forward_fp8_stamped(const void *x, const void *Wg, const void *W1q, const float *s1,
                          const void *W3q, const float *s3, const void *W2q, const float *s2, void *y, int T,
                          int d, int f, int E, int K, void *workspace, size_t ws_bytes, unsigned flags,
                          moe_stream_t stream, unsigned long long *stamps);

/*
 * Training: a forward pass that keeps what the backward pass needs, and the
 * backward pass (gradients by the chain rule through y = sum over the K kept
 * experts of G_i E_i(x): the SwiGLU experts, the softmax over the kept
 * logits and the router x Wg; section 3.4 "MoE Layer Formulation" and
 * "Expert Network Structure (SwiGLU)").  The selected set is held fixed: it
 * has no gradient, so gradients reach only the K selected experts of each
 * token and their K logits.
 *
 * Supported: dtype MOE_BF16 with d and f multiples of 64 (others return
 * MOE_ERR_UNSUPPORTED); other limits as moe_forward.
 *
 * moe_train_workspace_bytes: workspace size for both calls (0 if invalid or
 *   unsupported).  Besides the forward's buffers it holds the saved
 *   pre-activations a = x W1, b = x W3 of every grouped row (bf16 [R, 2f])
 *   and the backward's buffers: at T = 4096, d = 4096, f = 14336, E = 8,
 *   K = 2 it is about 1.7 GB.
 *
 * moe_forward_train: moe_forward (same arguments, flags and outputs; the
 *   gate/up contraction is never split) that also leaves in the workspace
 *   the routing, the grouped x, H and the pre-activations.
 *
 * moe_backward: given dy = dL/dy [T, d] (dtype), computes
 *   dx  [T, d]     fp32  dL/dx
 *   dWg [d, E]     fp32  dL/dWg
 *   dW1 [E, d, f]  fp32, dW3 [E, d, f] fp32, dW2 [E, f, d] fp32
 *   from the state the last moe_forward_train on this workspace left (same
 *   x, weights and sizes, ordered before this call; no other call on the
 *   workspace in between -- otherwise the results are unspecified).  x and
 *   the weights are the forward's.  With MOE_ACCUMULATE every gradient is
 *   added to its output buffer instead of overwriting it (an expert that
 *   received no token then leaves its gradients untouched; without the flag
 *   they are written as zeros).  T = 0 writes zero weight gradients (none
 *   with MOE_ACCUMULATE); x, dy and dx may then be NULL.  The outputs must
 *   not overlap one another.  Device-side errors are recorded in the
 *   workspace status word (moe_read_status); the backward does not clear it.
 *   flags: MOE_ACCUMULATE | MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT (the
 *   first grouped product's bounded wait expires: MOE_ERR_DEVICE_TIMEOUT is
 *   recorded and the gradients are unspecified).
 */
MOE_API size_t moe_train_workspace_bytes(int T, int d, int f, int E, int K, int dtype);
MOE_API int moe_forward_train(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                void *y, int T, int d, int f, int E, int K, int dtype,
                void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);
MOE_API int moe_backward(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                const void *dy, float *dx, float *dWg, float *dW1, float *dW3, float *dW2,
                int T, int d, int f, int E, int K, int dtype,
                void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * moe_backward recording MOE_NUM_BWD_STAGE_EVENTS cudaEvent_t handles on the
 * stream (for per-stage timing; otherwise identical): before the prep kernel
 * (dL/dlogits and gate * dy per grouped row), after it, after each grouped
 * product (dH with the SwiGLU backward, dW2, dX, dW1 | dW3), after dx and
 * after dWg.  Returns MOE_ERR_INVALID_ARG if events or one of its entries is
 * NULL.
 */
#define MOE_NUM_BWD_STAGE_EVENTS 8
MOE_API int moe_backward_timed(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                const void *dy, float *dx, float *dWg, float *dW1, float *dW3, float *dW2,
                int T, int d, int f, int E, int K, int dtype,
                void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                void *const *events);

/*
 * Decode-time expert cache (offload).  The routing analysis of the pages finds
 * strong temporal locality -- consecutive tokens often go to the same experts
 * ("Expert caching hint"; the Table 5 discussion) -- and names caching the
 * frequently used experts in GPU memory, with the rest in CPU memory, as the
 * optimisation it enables.  Here all E experts' weights live in pinned host
 * memory and C <= E device slots hold copies; each call loads the experts its
 * tokens need that are not resident, by least-recently-used replacement:
 *   - the needed set N is the experts with at least one routed token;
 *   - resident experts of N are hits; the others are misses, taken in
 *     increasing expert index, each into the lowest-index empty slot or else
 *     the slot of the least recently used resident expert outside N (ties
 *     to the lowest slot index);
 *   - every expert of N is marked used at the current step, then the step
 *     advances; |N| > C is an error (MOE_ERR_UNSUPPORTED, nothing loaded).
 * The state is a plain struct the caller owns; the library keeps none.
 */
#define MOE_CACHE_MAX_E 32
typedef struct moe_expert_cache {
  int E;                                /* experts */
  int C;                                /* device slots */
  int slot_of[MOE_CACHE_MAX_E];         /* expert -> slot, -1 if not resident */
  int expert_in[MOE_CACHE_MAX_E];       /* slot -> expert, -1 if empty */
  long long last_use[MOE_CACHE_MAX_E];  /* slot -> step of its last use, -1 if never */
  long long step;                       /* steps planned so far */
  long long hits, misses;               /* expert lookups so far */
  long long bytes_loaded;               /* host-to-device weight bytes enqueued by moe_forward_cached */
} moe_expert_cache;

/* Empty cache of C slots for E experts (1 <= C <= E <= 32).  Host only. */
MOE_API int moe_expert_cache_init(moe_expert_cache *cache, int E, int C);

/*
 * One step of the policy, host only: needed[E] (non-zero = needed) ->
 * the loads to make, load_expert[i] into load_slot[i] for i < *n_loads
 * (arrays of at least E entries), in the order above; updates the state.
 * Returns MOE_ERR_UNSUPPORTED if more than C experts are needed (the state is
 * then unchanged), MOE_ERR_INVALID_ARG for a null pointer or a state that is
 * not consistent.
 */
MOE_API int moe_expert_cache_plan(moe_expert_cache *cache, const int *needed, int *load_expert, int *load_slot,
                int *n_loads);

/*
 * moe_forward with the expert banks in host memory and a device cache:
 *   W1_host, W3_host [E, d, f], W2_host [E, f, d]   pinned host memory (dtype)
 *   W1_dev, W3_dev [C, d, f], W2_dev [C, f, d]      device slots, contents as
 *                                                   the cache state says
 * Routing runs first; the call then waits (on the host) for the per-expert
 * token counts, plans the step with moe_expert_cache_plan, enqueues one
 * host-to-device copy per missed expert and bank into its slot, and runs the
 * expert GEMMs on the slots.  The result equals moe_forward's bit for bit.
 * bf16 only (other dtypes: MOE_ERR_UNSUPPORTED); flags: MOE_ACCUMULATE |
 * MOE_DEBUG_CHECKS; the workspace is moe_forward's.  A failed call may leave
 * the cache state ahead of the device slots: re-initialise it.
 */
MOE_API int moe_forward_cached(const void *x, const void *Wg, const void *W1_host, const void *W3_host,
                const void *W2_host, void *W1_dev, void *W3_dev, void *W2_dev, moe_expert_cache *cache,
                void *y, int T, int d, int f, int E, int K, int dtype,
                void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * Routing only, for inspection: the router and grouping kernels that
 * moe_forward runs, with their results copied out in unpadded form
 * (section 3.4 gating function; "Top-K Gating Mechanism and Routing").
 *
 *   idx      [T, K] int32   selected experts, slot 0 = larger logit
 *   gate     [T, K] float   softmax weights over the selected logits
 *   perm_tok [T*K]  int32   token id of each row of the expert-grouped order:
 *                           experts ascending, and within one expert the
 *                           (token, slot) pairs in ascending t*K+k order
 *   offsets  [E+1]  int32   start row of each expert in perm_tok; offsets[E] = T*K
 *   pos      [T, K] int32   row of (t, k) in perm_tok order; may be NULL
 * Same size limits and workspace as moe_forward (same dtype).  With T = 0
 * only offsets is written (all zero) and the other pointers may be NULL.
 */
MOE_API int moe_route(const void *x, const void *Wg, int T, int d, int E, int K, int dtype,
              int32_t *idx, float *gate, int32_t *perm_tok, int32_t *offsets, int32_t *pos,
              void *workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_route without a workspace, for callers that cannot allocate device
 * memory: plugin hosts that give a kernel no scratch buffer, code running
 * while another thread captures a CUDA graph in global mode (cudaMalloc is
 * not allowed then), or serving loops that must not risk an allocation on
 * their hot path.  The pages have no counterpart; this is a convenience of
 * the library.
 *
 * Same arguments, outputs and results as moe_route, minus the workspace, plus
 * flags (0 or MOE_DEBUG_CHECKS: non-finite router logits are then recorded as
 * MOE_ERR_NONFINITE).  The scratch is a fixed array of 1 MiB compiled into the
 * library: every GPU that loads libmoe.so reserves it until the process
 * exits, and all calls on a GPU share it, so calls that overlap on the GPU
 * (different streams or host threads) race and must be serialised by the
 * caller.  The first call on each device (and in each new context of it, e.g.
 * after cudaDeviceReset) looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Limits: T <= MOE_ROUTE_NOALLOC_MAX_T, K <= 2,
 * E <= 32; a larger T returns MOE_ERR_UNSUPPORTED without launching.
 * Allocates nothing.  Device-side errors go to a status word in the array,
 * which the next call clears; read it with moe_route_noalloc_status.
 */
#define MOE_ROUTE_NOALLOC_MAX_T 16384
MOE_API int moe_route_noalloc(const void *x, const void *Wg, int T, int d, int E, int K, int dtype,
                      int32_t *idx, float *gate, int32_t *perm_tok, int32_t *offsets, int32_t *pos,
                      unsigned flags, moe_stream_t stream);

/*
 * The device status word of the last moe_route_noalloc call on the current
 * device (MOE_OK if it recorded no error): synchronises `stream` (the stream
 * of that call), then copies the word out of the library's scratch array.
 * MOE_ERR_CUDA if the synchronisation or the copy failed.  Allocates nothing.
 * The pages have no counterpart.
 */
MOE_API int moe_route_noalloc_status(moe_stream_t stream);

/*
 * RMSNorm with unit gain, out = x / sqrt(mean(x^2) + eps) per row, fp32 math
 * (pre-norm before each MoE block; paper-graph-ui summary, "Architectural
 * Inheritance from Mistral 7B", layer normalisation).  x, out: [T, d] of
 * dtype; out may equal x (in place); T >= 0, d >= 1; eps > 0.
 */
MOE_API int moe_rmsnorm(const void *x, void *out, int T, int d, float eps, int dtype, moe_stream_t stream);

/*
 * Synchronises `stream`, then returns the device status word in `workspace`
 * (MOE_OK if no device-side error was recorded since the last moe_forward or
 * moe_route on this workspace cleared it), or MOE_ERR_CUDA if the
 * synchronisation itself failed.  workspace: the device buffer passed to
 * moe_forward.
 */
MOE_API int moe_read_status(const void *workspace, moe_stream_t stream);

/* Static, NUL-terminated description of a status code. */
MOE_API const char *moe_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
MOE_API int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
