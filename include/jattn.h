/*
 * jattn.h -- C ABI of the GB300 (sm_103a) jagged attention library.
 *
 * The operation ("Training GEM at LLM scale", section "Jagged Sequence Flash
 * Attention"): FlashAttention computed directly on variable-length jagged
 * tensors, with asymmetric query / key-value lengths, custom attention biases
 * and a backward pass; section "Generalized Dot-Product Attention (GDPA)": the
 * softmax replaced by a pointwise GELU or SiLU with no normalisation; section
 * "BlockAttention": each 64-token query block attends only to its own 64-token
 * key/value block.
 *
 * For sequence b with local query rows i < Lq_b and keys j < Lk_b, head h:
 *   s_ij = scale * <q_i, k_j> + T[h, min(|i - j|, NB - 1)]     (bias optional, not scaled)
 *   softmax: O_i = sum_j softmax_j(s_ij) v_j,  lse_i = ln sum_j exp(s_ij)
 *   SiLU / tanh-GELU: O_i = sum_j act(s_ij) v_j
 *   BlockAttention: j restricted to floor(j/64) == floor(i/64)
 *
 * Tensor layout (every device tensor, caller-owned):
 *   q, out, dout, dq : [Tq, H, D] row-major (token, head, feature), row stride H*D
 *   k, v, dk, dv     : [Tk, H, D]
 *   offsets          : int32 exclusive prefix sums, length B+1, offsets[0] = 0,
 *                      non-decreasing; Tq = q_offsets[B], Tk = kv_offsets[B]
 *   bias table       : float32 [H, NB] (NB = mode.bias_buckets), or NULL
 *   lse              : float32 [H, Tq] (softmax only)
 *   element type     : bfloat16 (JATTN_BF16) or float32 (JATTN_FP32) for q, k, v,
 *                      out, dout, dq, dk, dv alike; all arithmetic runs in bf16
 *                      tensor-core products with fp32 accumulation.  float32
 *                      data are rounded to bf16 on entry, which keeps softmax
 *                      results inside the tolerances but not the unnormalised
 *                      activation sums: float32 plans take softmax only
 *                      (JATTN_ERR_UNSUPPORTED otherwise).
 * Device pointers must be 16-byte aligned.  D is 32, 64 or 128.  Positions i, j
 * are local to the sequence (also in cross-attention).  A sequence with Lk = 0
 * yields O_i = 0 and lse_i = -inf; a sequence with Lq = 0 yields dk = dv = 0.
 *
 * Errors: argument errors are returned before anything is launched; a failed
 * launch returns JATTN_ERR_CUDA; errors found on the device while a kernel runs
 * (a bounded wait that ran out, a tile record that fails its checks) are
 * written to the plan's device status word and reported, and cleared, by
 * jattn_check_device_status.  Nothing in the library aborts the process or
 * traps on the device.
 *
 * Calls that take a stream are stream-ordered and do not block the host,
 * except jattn_check_device_status (synchronises the stream).  A plan must not
 * be used on two streams at once.
 */
#ifndef JATTN_H_
#define JATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    JATTN_OK = 0,
    JATTN_ERR_INVALID_ARG = 1,    /* bad offsets, sizes, NULL pointers, mode fields */
    JATTN_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. D = 96) */
    JATTN_ERR_ALIGNMENT = 3,      /* a device pointer is not 16-byte aligned */
    JATTN_ERR_WORKSPACE = 4,      /* workspace NULL or smaller than required */
    JATTN_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
    JATTN_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait ran out (device status) */
    JATTN_ERR_DEVICE_CHECK = 7,   /* a kernel rejected a tile record (device status) */
    JATTN_ERR_NO_DEVICE = 8       /* the plan was made host-only (device = -1) */
} jattn_status;

typedef enum { JATTN_SOFTMAX = 0, JATTN_SILU = 1, JATTN_GELU_TANH = 2 } jattn_act;
typedef enum { JATTN_BF16 = 0, JATTN_FP32 = 1 } jattn_dtype;

/* Which operation a plan serves. */
typedef struct {
    int32_t act;          /* jattn_act */
    int32_t block;        /* 0 = full attention, 64 = BlockAttention (needs q_offsets == kv_offsets) */
    float scale;          /* score scale; 0 selects 1/sqrt(D) */
    int32_t bias_buckets; /* 0 = no bias, else NB >= 1 with H * NB <= 256 */
    int32_t dtype;        /* jattn_dtype */
    int32_t window;       /* sliding window W ("Training GEM at LLM scale", section
                             "BlockAttention": each token attends only to nearby
                             events): 0 = off; W > 0 restricts row i to keys j with
                             |i - j| < W, local positions, and the planner skips the
                             tiles outside that band; not combined with block */
    int32_t broadcast_q;  /* 1: the queries are shared by every sequence ("Training GEM at LLM
                             scale", section "Generalized Dot-Product Attention (GDPA)": pooled
                             attention with learned query rows).  Every sequence has the same
                             Lq = n query rows, which are the rows 0..n-1 of one DEVICE Q
                             [n, H, D] (not materialised per sequence); O, dO and lse keep one
                             row per sequence and query ([B*n, ...]); jattn_bwd returns dq
                             [n, H, D] = the sum over the sequences of their query gradients,
                             reduced in a fixed order (bitwise reproducible).  Needs full
                             attention (no block), bf16 data and D in {64, 128}; jattn_step_host
                             does not take it.  0 = off. */
    int32_t mxfp8;        /* 1: MXFP8 attention ("Training GEM at LLM scale", section "Low
                             Precision Flash Attention"): Q, K, V (and dO in the backward) are
                             quantised to the microscaling format, FP8 E4M3 elements with one
                             power-of-two E8M0 scale per 32 local rows x 32 features of a
                             sequence and head (exponent floor(log2 amax) - 8, elements rounded
                             to nearest even and saturated at 448); P is quantised online per
                             query row in 32-key groups against an integer running max in log2
                             units (the row sum from the unquantised P); the backward
                             quantises P and dS in 32 x 32 blocks.  The quantised values are
                             exactly representable in bf16 and the products run on the bf16
                             tensor cores with fp32 accumulation, which gives the products of a
                             block-scaled MMA exactly.  Needs softmax, full attention, bf16 data,
                             D in {64, 128}, no bias, window or broadcast Q, and a host plan at
                             fwd / bwd time; the backward needs jattn_bwd_workspace_bytes.
                             0 = off. */
} jattn_mode;

/* One unit of work: rows [q_start, q_start+q_len) of Q against rows
 * [kv_start, kv_start+kv_len) of K/V for sequence b and head h.  24 bytes. */
typedef struct {
    int32_t b, h, q_start, q_len, kv_start, kv_len;
} jattn_tile;

typedef enum {
    JATTN_TILES_Q = 0,  /* query-major tiles: forward and the dQ pass (128 query rows each) */
    JATTN_TILES_KV = 1  /* key-major tiles: the dK/dV pass (128 key rows each) */
} jattn_tile_list;

typedef struct jattn_plan jattn_plan; /* opaque */

/*
 * Build the tile lists and the persistent-grid schedule for one jagged batch
 * ("Training GEM at LLM scale", section "Generalized Dot-Product Attention
 * (GDPA)": valid tiles are precomputed on the CPU, empty tiles skipped, and the
 * tiles spread over the SMs to remove workload skew).
 *   q_offsets, kv_offsets : HOST int32 arrays of length B+1 (copied; caller keeps ownership)
 *   B >= 1, H >= 1, D in {32, 64, 128}
 *   mode                  : HOST pointer, copied
 *   device                : CUDA device ordinal, or -1 for a host-only plan (tile
 *                           lists only; jattn_fwd / jattn_bwd then return JATTN_ERR_NO_DEVICE)
 *   out                   : receives the plan; free it with jattn_plan_destroy
 * With a device the plan allocates its tile arrays and a status word on that
 * device and uploads the tiles with one host-to-device copy on the default
 * stream (synchronised before return).
 */
jattn_status jattn_plan_create(const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B, int32_t H, int32_t D,
                               const jattn_mode *mode, int32_t device, jattn_plan **out);

/*
 * Re-plan the same plan (same H, D and mode) for a new batch: rebuilds the tile
 * lists on the host and uploads them with an asynchronous copy on `stream`
 * (a cudaStream_t; NULL = default stream) from pinned memory the plan owns.
 * Device buffers grow (stream-synchronising) only when the new batch has more
 * tiles or sequences than any before.  Stream order makes the new tiles visible
 * to every later call on `stream` and keeps earlier calls on the old tiles.
 */
jattn_status jattn_plan_update(jattn_plan *plan, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                               void *stream);

/*
 * Re-plan on the device from offsets already in DEVICE memory ("Training GEM
 * at LLM scale", section "Generalized Dot-Product Attention (GDPA)": the valid
 * tiles are precomputed and spread over the SMs in a zigzag).  One kernel on
 * `stream` builds the same tile records as jattn_plan_update and a zigzag
 * schedule: sequences sorted by tile cost, tiles dealt over the SMs in the order
 * 0..C-1, C-1..0, ...  The host reads no offsets and builds nothing, and later
 * calls on `stream` use the new lists.  Results equal those of a host plan bit
 * for bit.
 *   q_offsets, kv_offsets : DEVICE int32 [B+1], 4-byte aligned; read by the
 *                           kernel, so they must stay valid until it has run
 *   B in [1, 8192]        : more sequences return JATTN_ERR_UNSUPPORTED
 *   Tq, Tk                : the last entries of the offsets (the caller's tensor
 *                           lengths; they size the workspaces and tensor maps)
 * Offsets that do not start at 0, decrease, end elsewhere than Tq / Tk, or
 * (BlockAttention) give a sequence different query and key lengths are found
 * by the kernel: it plans no tile and sets JATTN_ERR_DEVICE_CHECK on the
 * device status word (jattn_check_device_status).  With a device plan,
 * jattn_fwd_rope / jattn_bwd_rope leave the table-length check to the kernels,
 * which report a short table as JATTN_ERR_DEVICE_CHECK.  The device buffer
 * grows, stream-synchronising, when the batch needs more room than any before.
 */
jattn_status jattn_plan_update_device(jattn_plan *plan, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                                      int64_t Tq, int64_t Tk, void *stream);

/*
 * Host view of a scheduled tile list, for inspection and tests.  The records are
 * grouped by CTA: CTA c runs tiles[cta_begin[c] .. cta_begin[c+1]) in order.
 * After jattn_plan_update_device the call first synchronises the plan's device
 * and downloads the device lists (CTA count = the SM count; CTAs past the last
 * tile have empty ranges).
 * The pointers stay valid until the next jattn_plan_update(_device) or
 * jattn_plan_destroy.
 */
jattn_status jattn_plan_tiles(const jattn_plan *plan, int32_t which, const jattn_tile **tiles, int64_t *n_tiles,
                              const int32_t **cta_begin, int32_t *n_ctas);

/*
 * Device scratch for jattn_fwd / jattn_bwd (bytes; 0 = none needed).
 * jattn_fwd needs jattn_fwd_workspace_bytes.  jattn_bwd needs at least
 * jattn_bwd_workspace_bytes_min and takes its fastest path when given
 * jattn_bwd_workspace_bytes: full attention on a host plan without a sliding
 * window or RoPE then keeps every block's dS in the workspace (bf16, 16 KB per
 * 128 keys x 64 queries of a sequence and head; hi and lo parts in the
 * activation modes), written once by the dK/dV pass, and computes dQ as a
 * streaming product of it ("Training GEM at LLM scale", section "Jagged
 * Sequence Flash Attention": dQ without atomic adds and without recomputing
 * the scores).  With less than that (but at least the minimum) it runs a dQ
 * pass that recomputes the scores.  Both are exact to the same tolerances;
 * their dQ may differ in the last bits.  The sizes depend on the batch the
 * plan was last (re)planned for.
 */
size_t jattn_fwd_workspace_bytes(const jattn_plan *plan);
size_t jattn_bwd_workspace_bytes(const jattn_plan *plan);
size_t jattn_bwd_workspace_bytes_min(const jattn_plan *plan);

/* Frees the plan's host and device memory (synchronises its device). NULL is a no-op. */
void jattn_plan_destroy(jattn_plan *plan);

/*
 * Forward.  q, k, v: DEVICE inputs; out: DEVICE output [Tq, H, D];
 * bias: DEVICE [H, NB] float32 iff mode.bias_buckets > 0 (else must be NULL);
 * lse: DEVICE float32 [H, Tq], written when non-NULL in softmax mode (required
 * later by jattn_bwd in full softmax mode), must be NULL otherwise.
 * workspace: DEVICE scratch of jattn_fwd_workspace_bytes (may be NULL when 0).
 * stream: cudaStream_t.
 */
jattn_status jattn_fwd(const jattn_plan *plan, const void *q, const void *k, const void *v, const float *bias,
                       void *out, float *lse, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward.  dout, q, k, v, out: DEVICE inputs (out = the forward output);
 * lse: the forward's lse (required in full softmax mode, ignored otherwise);
 * dq, dk, dv: DEVICE outputs, fully overwritten (no accumulation, no atomics);
 * dbias: DEVICE float32 [H, NB] gradient of the bias table, overwritten when
 * non-NULL (needs a bias; full attention and sliding window only: with block
 * mode the call returns JATTN_ERR_UNSUPPORTED); workspace: DEVICE scratch of at
 * least jattn_bwd_workspace_bytes_min bytes (jattn_bwd_workspace_bytes for the
 * fastest path), 16-byte aligned.
 * dq and dk include the score scale; dbias[h, n] is the plain sum of dS over
 * the pairs of head h in bucket n = min(|i - j|, NB - 1). It is summed with
 * floating-point atomic adds, so it is reproducible to rounding only (dq, dk
 * and dv are bitwise reproducible).
 */
jattn_status jattn_bwd(const jattn_plan *plan, const void *dout, const void *q, const void *k, const void *v,
                       const float *bias, const void *out, const float *lse, void *dq, void *dk, void *dv,
                       float *dbias, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Rotary position embedding (RoPE) on the BlockAttention path ("Training GEM at
 * LLM scale", section "BlockAttention": RoPE, with its backward fused into the
 * attention epilogue).  The angle tables are the caller's.
 */
typedef struct {
    const float *cos; /* DEVICE float32 [rows, D/2], row p = position p: cos of the angle of feature pair d */
    const float *sin; /* DEVICE float32 [rows, D/2]: sin of the same angles */
    int32_t rows;     /* positions 0 .. rows-1; must cover the longest sequence of the batch */
} jattn_rope;

/*
 * jattn_fwd with Q and K rotated before the scores.  Row i of a sequence sits at
 * local position p = i; each feature pair (d, d + D/2), d < D/2, is turned:
 *   q'[d] = q[d] c - q[d + D/2] s,   q'[d + D/2] = q[d + D/2] c + q[d] s,
 * with c = cos[p * D/2 + d] and s = sin[p * D/2 + d]; K likewise.  The kernel
 * rotates each Q and K tile in shared memory as it arrives (in float32, rounded
 * to bf16 for the tensor cores); no rotated copy of Q or K is written.
 * rope = NULL: exactly jattn_fwd.  Otherwise the plan must be softmax
 * BlockAttention (mode.act = JATTN_SOFTMAX, mode.block = 64) on bf16 data with
 * D in {64, 128}, else JATTN_ERR_UNSUPPORTED.  (The rotated rows reach the
 * tensor cores as bf16; a normalised softmax row keeps that rounding inside
 * the tolerances, the unnormalised activation sums do not.)  cos or sin NULL, or rows below the longest sequence:
 * JATTN_ERR_INVALID_ARG.  cos or sin not 16-byte aligned: JATTN_ERR_ALIGNMENT.
 * The tables are read, never written, and must stay valid until the kernel ends.
 */
jattn_status jattn_fwd_rope(const jattn_plan *plan, const void *q, const void *k, const void *v, const float *bias,
                            const jattn_rope *rope, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * jattn_bwd for a forward made by jattn_fwd_rope with the same tables.  q and k
 * are the unrotated inputs; dq and dk are the gradients of the unrotated Q and
 * K.  The kernel rotates the loaded Q and K tiles again.  Its epilogue applies
 * the transposed rotation to dQ and dK in float32, before the bf16 store:
 *   dq[d] = c g[d] + s g[d + D/2],   dq[d + D/2] = c g[d + D/2] - s g[d],
 * where g is the gradient of the rotated rows.  Errors: as jattn_fwd_rope.
 */
jattn_status jattn_bwd_rope(const jattn_plan *plan, const void *dout, const void *q, const void *k, const void *v,
                            const float *bias, const jattn_rope *rope, const void *out, const float *lse, void *dq,
                            void *dk, void *dv, float *dbias, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Profiling hook (optional).  After this call every jattn_fwd / jattn_bwd on
 * the plan records events[0] on its stream before its first kernel and
 * events[i] right after its i-th kernel (i < n_events), so elapsed times
 * between consecutive events are per-kernel device durations.  `events` is a
 * HOST array of cudaEvent_t handles owned by the caller (copied; the handles
 * must stay valid while set; a NULL handle is JATTN_ERR_INVALID_ARG); NULL or
 * n_events = 0 turns the hook off.  A failed event record fails the call with
 * JATTN_ERR_CUDA.
 */
jattn_status jattn_plan_set_events(jattn_plan *plan, void *const *events, int32_t n_events);

/* Number of kernels launched through this plan since it was created (host counter). */
int64_t jattn_plan_launch_count(const jattn_plan *plan);

/*
 * Backward without a caller-provided workspace.  The paper has no counterpart;
 * this entry point exists for callers that cannot call cudaMalloc or hand the
 * library device memory: code running where a framework's allocator owns the
 * whole device, plug-ins and sandboxes without allocation rights, or latency-
 * critical paths that must not take an allocation (which can synchronise the
 * device).  Arguments and results are those of jattn_bwd, minus the workspace.
 *
 * The scratch the backward needs (Delta = rowsum(dO * O), [H, Tq] floats, plus
 * bf16 staging copies for float32 or D = 32 data) lives in a fixed 16 MiB
 * device array inside the library, reserved on every GPU that loads it until
 * the process exits.  A batch whose jattn_bwd_workspace_bytes_min exceeds
 * 16 MiB is rejected with JATTN_ERR_WORKSPACE before anything runs (softmax,
 * bf16: up to H * Tq = 4,194,304).  The call takes jattn_bwd's fastest path
 * when the whole jattn_bwd_workspace_bytes fits the array, and otherwise the
 * path that recomputes the scores for dQ; its results are then bitwise those
 * of jattn_bwd given a workspace of the same size.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress, once per device) and keeps it for the
 * life of the process; make that first call before any stream capture.  A
 * device reset (cudaDeviceReset, or the primary context torn down and made
 * again) unloads the library's module on that device and leaves the kept
 * address stale: do not call this entry point on a device after resetting it.  All calls share the one array and each call
 * overwrites the part it uses (nothing in it has to start at zero), so calls
 * whose work overlaps on the GPU (different streams, or different host threads
 * without ordering) race on it: order them.
 */
jattn_status jattn_bwd_noalloc(const jattn_plan *plan, const void *dout, const void *q, const void *k, const void *v,
                               const float *bias, const void *out, const float *lse, void *dq, void *dk, void *dv,
                               float *dbias, void *stream);

/*
 * One training step whose tensors live in host memory ("Training GEM at LLM
 * scale", "Jagged Sequence Flash Attention": forward and backward of the jagged
 * batch). The call re-plans the plan for the batch given by the host offsets,
 * as jattn_plan_update does. It copies q, k, v, dout (and bias) host -> device,
 * runs jattn_fwd and jattn_bwd, and copies out, dq, dk, dv (and lse)
 * device -> host.
 *
 * Layouts and dtypes are those of jattn_fwd / jattn_bwd, all tensors on the
 * host: q, dout, out, dq [Tq, H, D]; k, v, dk, dv [Tk, H, D] with Tq =
 * q_offsets[B], Tk = kv_offsets[B]; bias [H, NB] fp32 (NULL iff the plan has no
 * bias); lse [H, Tq] fp32 or NULL (not returned; softmax only).
 *
 * Asynchronous and pipelined: the call enqueues its work and returns. The plan
 * owns two device staging sets and three streams for this (upload, compute,
 * download). Consecutive calls therefore overlap: call n's uploads run during
 * call n-1's kernels, and call n-1's downloads during call n's kernels. The work
 * of a call starts after the work already queued on `stream` (the caller's
 * stream, NULL = legacy default stream). The host buffers of a call belong to
 * the library until jattn_step_host_join's wait has passed; they must not be
 * modified or freed before. Page-locked (pinned) host memory gives full
 * overlap; pageable memory is accepted, but its copies do not overlap.
 *
 * Errors: JATTN_ERR_INVALID_ARG for a NULL plan or required pointer, bad
 * offsets or a bias that does not match the plan; JATTN_ERR_NO_DEVICE for a
 * host-only plan; JATTN_ERR_CUDA when a CUDA call fails (details in
 * jattn_last_cuda_error); errors of the enqueued kernels surface through
 * jattn_check_device_status. The first call, and any call whose batch is larger
 * than every earlier one, allocates the staging sets (after waiting for the
 * calls that still use them).
 */
jattn_status jattn_step_host(jattn_plan *plan, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                             const void *q, const void *k, const void *v, const void *dout, const float *bias,
                             void *out, float *lse, void *dq, void *dk, void *dv, void *stream);

/*
 * Makes `stream` (NULL = legacy default stream) wait until every
 * jattn_step_host call issued on the plan so far has finished, its downloads
 * included. Once the stream passes that point, the calls' host buffers may be
 * read and reused. Returns JATTN_ERR_INVALID_ARG for a NULL plan, JATTN_OK when
 * no call was issued, JATTN_ERR_CUDA when the wait cannot be enqueued.
 */
jattn_status jattn_step_host_join(jattn_plan *plan, void *stream);

/*
 * MXFP8 quantisation of one input tensor, as the mxfp8 mode applies it to Q, K,
 * V and dO: blocks of 32 local rows (the sequence's rows under the plan's
 * query offsets, which = JATTN_TILES_Q, or key offsets, JATTN_TILES_KV) x 32
 * features of one head, one E8M0 exponent per block (floor(log2 amax) - 8,
 * clamped to [-127, 127]), E4M3 elements (nearest, ties to even, saturated at
 * +-448).  xq receives the values the blocks stand for, element times scale,
 * as bf16 (exact).  x, xq: DEVICE bf16 [T, H, D], 16-byte aligned; the plan
 * must be an mxfp8 plan (else JATTN_ERR_UNSUPPORTED) made or updated on the
 * host.  Stream-ordered.
 */
jattn_status jattn_mxfp8_quantize(const jattn_plan *plan, const void *x, int32_t which, void *xq, void *stream);

/*
 * Test hook: the error path of a bounded wait on a real launch.  The paper has
 * no counterpart.  Launches a test build of the forward kernel whose
 * score-issuing thread first waits on a barrier that nothing completes; after
 * wait_ns nanoseconds (100 us .. 2 s; the library's own kernels wait 2 s) that
 * wait gives up, writes JATTN_ERR_DEVICE_TIMEOUT to the plan's status word and
 * raises the CTA's abort flag; every other role of the CTA leaves its loop, the
 * copies in flight are drained, TMEM is freed and the kernel returns.  Nothing
 * traps; the device stays usable.  out and lse receive no defined values.  The
 * plan must be full softmax attention on bf16 data without bias, window or
 * broadcast Q, D in {64, 128} (else JATTN_ERR_UNSUPPORTED); the tensors are
 * those of jattn_fwd, lse required.  The status is read with
 * jattn_check_device_status.
 */
jattn_status jattn_test_fwd_stall(const jattn_plan *plan, const void *q, const void *k, const void *v, void *out,
                                  float *lse, uint64_t wait_ns, void *stream);

/* Synchronises `stream`, then returns and clears the plan's device status word. */
jattn_status jattn_check_device_status(const jattn_plan *plan, void *stream);

/* Text of the CUDA error behind the calling thread's most recent JATTN_ERR_CUDA
 * return (thread-local, static storage; "" if none). */
const char *jattn_last_cuda_error(void);

/* Static, human-readable name of a status code. */
const char *jattn_status_str(jattn_status status);

/* ------------------------------------------------------------------------
 * Multi-GPU data parallelism.  Every (sequence, head) pair is independent
 * ("Training GEM at LLM scale", sections "Jagged Sequence Flash Attention"
 * and the data-parallel training it serves), so a batch shards across ranks by
 * whole sequences with no collective on the attention path.  Host only; touches
 * no device.
 *
 * Assigns each of the B sequences of a jagged batch to one of `world` ranks:
 * sequences in decreasing order of the cost Lq*Lk + 64*(Lq + Lk) (the pair
 * work plus a per-row term for the tile set-up and the row traffic), each to
 * the rank with the least cost so far (ties to the lower rank; equal costs keep
 * their batch order), so the result is deterministic and the same on every
 * rank.  q_offsets_host / kv_offsets_host: HOST int32 [B + 1] as for
 * jattn_plan_create (block mode needs no special treatment).  rank_of: HOST
 * int32 [B], caller-owned, receives the rank of each sequence.  Returns
 * JATTN_ERR_INVALID_ARG for NULL pointers, B < 1, world < 1 or offsets that are
 * not a valid prefix sum.
 */
jattn_status jattn_shard(const int32_t *q_offsets_host, const int32_t *kv_offsets_host, int32_t B, int32_t world,
                         int32_t *rank_of);

#ifdef __cplusplus
}
#endif

#endif /* JATTN_H_ */
