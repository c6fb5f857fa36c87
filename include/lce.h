/*
 * lce.h -- memory-bounded fused linear cross-entropy on GB300 (sm_103a): the C ABI.
 *
 * What is computed
 *   For hidden states H [N x d], a vocabulary projection W [V x d] and labels y [N]:
 *     logits  Z = H W^T                                      (never stored)
 *     lse_i   = log sum_v exp(Z_iv)
 *     loss    = sum over valid rows of (lse_i - Z_{i,y_i}), divided by n_valid for MEAN
 *     dH      = G W,  dW = G^T H,  G = scale * (softmax(Z) - onehot(y)) on valid rows, 0 elsewhere
 *   "Running 128K-Sequence MoE RL on 32 H100s" (blog), section "Linear CE: Avoiding
 *   Materialization of Full Logits": the linear output and the cross-entropy are organised so
 *   that the full logits are never generated or retained.
 *   "Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training",
 *   section 3.2 and appendix C (Ring-DTP): each logit strip of the vocabulary is folded into a
 *   running per-token state and released, and backward recomputes each strip's gradient, so
 *   neither the full logits nor the full logit gradient is stored; section 2: the values and
 *   gradients equal those of the dense implementation, only the order of computation changes.
 *   On one GPU the strips are visited by a local loop; the per-token state is the online
 *   log-sum-exp triple (running max, running sum of exp, target logit).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays on the current device.
 *     H and W hold bf16 (LCE_BF16) or fp32 (LCE_F32, LCE_F32_TF32X3) values; dH and dW are
 *     always fp32.
 *     labels are int64.  Every pointer must be 16-byte aligned.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call
 *     only enqueues work on that stream and returns; nothing is synchronised except in
 *     lce_check_error.
 *   - Ownership: the caller owns every buffer, including the workspace.  The library never
 *     allocates or frees device memory and keeps no pointer after a call returns.
 *   - Errors: argument and shape problems are found on the host before anything is enqueued
 *     and returned as a status; nothing is launched then.  Problems found on the device (a
 *     label outside [0, V) that is not ignore_index; a kernel wait that ran out of time) set a
 *     flag in the workspace header that lce_check_error turns into a status.  Rows with such a
 *     label are left out of the loss, of n_valid and of the gradients.  No call aborts the
 *     process or traps the device.
 *   - Shape rules (LCE_ERR_UNSUPPORTED_SHAPE otherwise): N >= 0, V >= 1, d >= 1 with a row of
 *     d elements a multiple of 16 bytes (d % 8 == 0 for LCE_BF16, d % 4 == 0 for LCE_F32 and
 *     LCE_F32_TF32X3), strip_V >= 128 with strip_V % 128 == 0, N, d, V, strip_V < 2^31.
 *   - Determinism: for a fixed device, shape and strip_V, every output is bitwise identical from
 *     run to run (no atomics take part in any sum; every reduction has a fixed order).
 *   - Not thread-safe across host threads only for the tracing calls (lce_trace_*).
 */
#ifndef LCE_H
#define LCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LCE_OK = 0,
  LCE_ERR_INVALID_ARG = 1,        /* null or misaligned pointer, unknown enum value            */
  LCE_ERR_UNSUPPORTED_SHAPE = 2,  /* a shape rule above is broken                              */
  LCE_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes < lce_workspace_size(...)                       */
  LCE_ERR_LABEL_OUT_OF_RANGE = 4, /* device found a label outside [0, V) and != ignore_index   */
  LCE_ERR_CUDA = 5,               /* a CUDA runtime call or a kernel launch failed             */
  LCE_ERR_TIMEOUT = 6,            /* a kernel-side wait gave up (the kernel returned early)    */
  LCE_ERR_UNSUPPORTED_DEVICE = 7  /* current device is not compute capability 10.3 (sm_103a)   */
} lce_status_t;

typedef enum { LCE_REDUCTION_MEAN = 0, LCE_REDUCTION_SUM = 1 } lce_reduction_t;
/*
 * Input format and arithmetic.
 *   LCE_BF16        bf16 H and W; tensor-core products, fp32 accumulation.
 *   LCE_F32         fp32 H and W; exact fp32 products and sums on the CUDA cores.
 *   LCE_F32_TF32X3  fp32 H and W on the tensor cores: every operand x is split into tf32 parts
 *                   hi = nearest tf32 of x and lo = nearest tf32 of (x - hi), and every product is
 *                   formed as hi*hi' + hi*lo' + lo*hi' with fp32 accumulation (the dropped lo*lo'
 *                   and the rounding of lo are about 2^-21 relative): about fp32 accuracy at
 *                   tensor-core speed.
 * dH and dW are fp32 in every format.
 */
typedef enum { LCE_BF16 = 0, LCE_F32 = 1, LCE_F32_TF32X3 = 2 } lce_dtype_t;

/*
 * Width of the vocabulary strips (columns): the vocabulary is cut into ceil(V / strip_V) strips
 * of equal width -- every strip but the last is this wide, the last one the rest -- rounded up to
 * the tensor cores' tile width of 256 columns (128 for LCE_F32) when that stays within strip_V,
 * else to 128; never wider than strip_V or V.  strip_V is thus the largest strip, and the last
 * strip is never a sliver.  0 when V < 1 or strip_V breaks its shape rule.
 */
int64_t lce_strip_columns(int64_t V, int64_t strip_V, lce_dtype_t dtype);

/*
 * Bytes of device workspace that lce_forward and lce_backward need for these sizes; 0 when the
 * arguments break a shape rule.  It grows as O(N * min(strip_V, V)) (LCE_F32_TF32X3 adds
 * O((N + min(strip_V, V)) * d) for its operand copies) and never with V beyond the strip: this
 * is the closed-form per-call budget that can be checked before launch
 * ("Flattening Every Memory Peak in Long-Context Mixture-of-Experts Training", sections 3.5
 * and 6: the per-rank budget is fixed by the launch configuration).  Layout: a 256-byte header
 * (error flags) followed by the larger of the forward region (running state, target logits,
 * per-tile partial states of one strip) and the backward region: one strip of the logit gradient
 * (N x strip_V elements of the input dtype), or two for bf16 when the backward of a strip is small
 * (ceil(N/256) * ceil(d/256) <= 512): each backward launch then overlaps dH and dW of one strip
 * with the gradient of the next.  LCE_F32_TF32X3 places the tf32 hi and lo parts of H (2 x N x d
 * fp32) and of one W strip (2 x min(strip_V, V) x d fp32) after the header, and its backward
 * region holds, as hi and lo parts each, H and the W strip transposed, the gradient strip
 * (N x strip_V fp32) and the gradient strip transposed: the tf32 MMAs read every operand with
 * the contracted index contiguous.
 */
size_t lce_workspace_size(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dtype);

/*
 * Forward.  Visits the vocabulary in strips of lce_strip_columns(V, strip_V, dtype) columns; for
 * each strip it forms the logit tiles (tensor cores; CUDA cores for LCE_F32), folds them into the
 * running per-token state in the GEMM epilogue and drops them.  Writes
 *   loss    : device fp32 scalar (MEAN over valid rows; NaN when n_valid == 0.  SUM: the sum)
 *   lse     : device fp32 [N], log-sum-exp of every row (ignored rows included)
 *   n_valid : device int64 scalar, number of rows whose label is in [0, V)
 * ignore_index is any int64 value (conventionally -100).  Clears the workspace error flags.
 */
lce_status_t lce_forward(const void* H, const void* W, const int64_t* labels,
                         int64_t N, int64_t d, int64_t V, int64_t ignore_index, int64_t strip_V,
                         lce_reduction_t reduction, lce_dtype_t dtype,
                         float* loss, float* lse, int64_t* n_valid,
                         void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward from the saved per-token lse and n_valid (outputs of lce_forward on the same H, W,
 * labels) and the incoming gradient dloss (device fp32 scalar).  For each strip it recomputes
 * the logits, forms G = scale * (softmax - onehot) in the epilogue (scale = dloss / n_valid for
 * MEAN, dloss for SUM) into one strip of workspace, then accumulates dH += G_s W_s and writes
 * dW_s = G_s^T H (tensor cores; CUDA cores for LCE_F32).  Writes dH (device fp32 [N x d],
 * overwritten) and dW (device fp32 [V x d], overwritten).  dW rows are each written exactly once
 * (deterministic).
 * The workspace need not come from lce_forward; its header (error flags) is cleared first, so
 * lce_check_error afterwards reports the problems this call found.
 */
lce_status_t lce_backward(const void* H, const void* W, const int64_t* labels,
                          const float* lse, const int64_t* n_valid, const float* dloss,
                          int64_t N, int64_t d, int64_t V, int64_t ignore_index, int64_t strip_V,
                          lce_reduction_t reduction, lce_dtype_t dtype,
                          float* dH, float* dW,
                          void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward, one gradient at a time ("delay wgrad"): "Running 128K-Sequence MoE RL on 32 H100s",
 * section "Backward Trace: Chunk dgrad and Delay wgrad" -- the data gradient is on the critical
 * path of the backward pass, the weight gradient is not and can run later (e.g. on another
 * stream, overlapping the caller's next operation).
 *   parts = LCE_GRAD_DH: only dH (dW may be NULL, is not touched);
 *   parts = LCE_GRAD_DW: only dW (dH may be NULL, is not touched);
 *   parts = LCE_GRAD_DH | LCE_GRAD_DW: exactly lce_backward.
 * Each call recomputes the strips' logits and gradient itself: the full logit gradient is never
 * stored, so splitting the two gradients costs one more logit recompute (8 N d V FLOP for both
 * calls instead of 6 N d V), and takes the dW GEMMs off the critical path (4 N d V FLOP for dH).
 * The dH and dW written are bitwise identical to those of lce_backward.  Same arguments,
 * workspace size, errors and ordering as lce_backward; two calls may not share a workspace while
 * both are in flight.
 */
typedef enum { LCE_GRAD_DH = 1, LCE_GRAD_DW = 2 } lce_grad_part_t;
lce_status_t lce_backward_parts(const void* H, const void* W, const int64_t* labels,
                                const float* lse, const int64_t* n_valid, const float* dloss,
                                int64_t N, int64_t d, int64_t V, int64_t ignore_index,
                                int64_t strip_V, lce_reduction_t reduction, lce_dtype_t dtype,
                                int32_t parts, float* dH, float* dW,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Forward and backward between HOST buffers: lce_forward followed by lce_backward, for callers
 * whose data lives in host memory (a host-side pipeline, offloaded activations, a harness).  The
 * call enqueues on `stream`, in this order, and returns: the copies of H, W, labels and dloss
 * into `device_buffer`, the forward, the backward, and the copies of the requested results back
 * to host memory.  Once the stream has passed that point (e.g. after cudaStreamSynchronize) the
 * results are in host memory and the host inputs may be reused.
 *   - H, W, labels, dloss: HOST inputs (layouts as in lce_forward; dloss is one fp32 value).
 *     In page-locked (pinned) host memory the copies are asynchronous and overlap other work on
 *     the device; pageable memory works, but then the copies may hold the calling thread.
 *   - loss (1 float), lse (N floats), n_valid (1 int64), dH (N x d floats), dW (V x d floats),
 *     device_error_flags (1 uint32: bit 0 a label outside [0, V) that is not ignore_index, bit 1
 *     a kernel wait that timed out; 0 when neither happened): HOST outputs.  Any of them may be
 *     NULL; that result is then not copied back (it is still computed).
 *   - device_buffer: caller-owned DEVICE memory, 16-byte aligned, of at least
 *     lce_host_buffer_size(...) bytes: it holds the workspace, the device copies of the inputs and
 *     the results.  Two calls in flight at the same time need two buffers.
 *   - compute_after, compute_done: optional cudaEvent_t handles (NULL for none), owned by the
 *     caller.  The kernels of this call start only once compute_after has completed (a wait
 *     enqueued after the input copies), and compute_done is recorded once they have finished
 *     (before the result copies).  With them a caller runs consecutive calls on two streams and
 *     two buffers so that one call's copies overlap the other's kernels while the kernels of
 *     the calls still run one after another (kernels of two calls running at the same time
 *     share the SMs and slow each other down).
 * Errors: as lce_forward and lce_backward (LCE_ERR_WORKSPACE_TOO_SMALL when device_bytes is below
 * lce_host_buffer_size); problems found on the device come back through device_error_flags.
 * The results are bitwise those of lce_forward + lce_backward on the same inputs.
 */
size_t lce_host_buffer_size(int64_t N, int64_t d, int64_t V, int64_t strip_V, lce_dtype_t dtype);
lce_status_t lce_forward_backward_host(const void* H, const void* W, const int64_t* labels,
                                       const float* dloss, int64_t N, int64_t d, int64_t V,
                                       int64_t ignore_index, int64_t strip_V,
                                       lce_reduction_t reduction, lce_dtype_t dtype, float* loss,
                                       float* lse, int64_t* n_valid, float* dH, float* dW,
                                       uint32_t* device_error_flags, void* device_buffer,
                                       size_t device_bytes, void* stream,
                                       const void* compute_after, void* compute_done);

/*
 * Forward for callers that cannot allocate device memory.  The pages describe no such entry
 * point: it is an addition of this library, with no counterpart in the papers.
 *
 * Some callers may not call cudaMalloc at all: a plugin of an engine that owns all device memory
 * through its own pool and only lends out the buffers it planned; a service whose device memory
 * budget is fixed at start-up and may not grow per request; latency-critical code that cannot
 * take the cost of an allocation or the device-wide synchronisation of a free.  This entry point
 * computes exactly what lce_forward computes (same kernels, same results) but takes its workspace
 * from a fixed array of LCE_STATIC_SCRATCH_BYTES (16 MiB) that the library keeps in device
 * memory; it allocates nothing and frees nothing.  The caller still passes the inputs and the outputs (loss, lse, n_valid as
 * in lce_forward).
 *   - Size limit: when lce_workspace_size(N, d, V, strip_V, dtype) exceeds
 *     LCE_STATIC_SCRATCH_BYTES the call returns LCE_ERR_WORKSPACE_TOO_SMALL and enqueues nothing
 *     (a smaller strip_V shrinks the workspace).
 *   - device_error_flags (optional, device uint32, may be NULL) receives the device error bits
 *     of this call once it has run: bit 0 = a label outside [0, V) that is not ignore_index,
 *     bit 1 = a kernel wait timed out.  0 means no device-side error.
 *   - Set-up: the first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture begins.
 *   - Sharing: every GPU that loads the library holds the array until the process exits, and
 *     every call on a device uses the same array, which keeps the last call's contents (the call
 *     clears what must start at zero).  Calls whose work can overlap on the GPU -- on different
 *     streams, or from several host threads -- race on the array; order them on one stream.
 */
#define LCE_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
lce_status_t lce_forward_static_scratch(const void* H, const void* W, const int64_t* labels,
                                        int64_t N, int64_t d, int64_t V, int64_t ignore_index,
                                        int64_t strip_V, lce_reduction_t reduction,
                                        lce_dtype_t dtype, float* loss, float* lse,
                                        int64_t* n_valid, uint32_t* device_error_flags,
                                        void* stream);

/*
 * Synchronises stream, then reads the workspace error flags written by the device:
 * LCE_ERR_TIMEOUT, else LCE_ERR_LABEL_OUT_OF_RANGE, else LCE_OK (LCE_ERR_CUDA if the copy or the
 * synchronisation itself fails).
 */
lce_status_t lce_check_error(const void* workspace, void* stream);

/* Static, human-readable name of a status code. */
const char* lce_status_string(lce_status_t status);

/*
 * Name of the CUDA error behind the most recent LCE_ERR_CUDA returned on the calling thread
 * (e.g. "cudaErrorInvalidValue"), or "none".  Static storage; valid until the next call.
 */
const char* lce_last_cuda_error(void);

/*
 * Tile variant of the bf16 tensor-core kernels, process-wide (not thread-safe; for tests and
 * tuning).  0 = automatic (default): CTA pairs whenever the GEMM has more than 128 rows,
 * 1 = single-CTA 128x256 tiles (tcgen05 cta_group::1, 4-stage pipeline),
 * 2 = CTA-pair 256x256 tiles (cta_group::2 on a cluster of 2, 6-stage pipeline).
 * Results are equal within rounding across variants; each variant is deterministic.
 * LCE_ERR_INVALID_ARG for any other value.
 */
lce_status_t lce_set_tile_config(int32_t config);

/*
 * Test hook for the timeout path (process-wide, not thread-safe).  With on = 1 the next bf16
 * tensor-core launch withholds the first k-block of operands it would load: nothing arrives on
 * that stage's barrier, so the MMA issuer's bounded wait runs out after its 2 s limit.  Every role
 * of every CTA then gives up, lets copies in flight land, frees its tensor memory and returns;
 * the launch sets the workspace timeout bit, so lce_check_error reports LCE_ERR_TIMEOUT, and the
 * CUDA context stays usable.  The hook clears itself after that one launch.  No fault, trap or
 * endless loop is involved.  LCE_ERR_INVALID_ARG unless on is 0 or 1.
 */
lce_status_t lce_test_inject_stall(int32_t on);

/*
 * Number of kernels this library has launched in this process so far (all entry points, all
 * threads).  Used to count device launches inside a timed region.
 */
int64_t lce_launch_count(void);

/*
 * Optional launch tracing for profiling.  Between lce_trace_begin and lce_trace_end, every
 * kernel launch made by lce_forward / lce_backward on the calling thread is bracketed by
 * cudaEventRecord(start_events[k]) / cudaEventRecord(stop_events[k]) on its stream and tagged
 * kernel_ids[k] (see lce_kernel_name), for k = 0 .. capacity-1; further launches are not
 * recorded.  The events are caller-owned cudaEvent_t handles created with timing enabled.
 * lce_trace_end returns the number of launches recorded.  Not thread-safe.
 */
lce_status_t lce_trace_begin(void* const* start_events, void* const* stop_events,
                             int32_t* kernel_ids, int32_t capacity);
int32_t lce_trace_end(void);

/*
 * Name of a traced kernel id; NULL if unknown.  Tensor-core launches: "tc_fwd_lse" (forward),
 * "tc_bwd_grad" (a strip's gradient), "tc_dh_dw" (a strip's dH and / or dW), "tc_bwd" (dH and dW
 * of one strip with the gradient of the next, for small backward steps); CUDA-core launches of
 * the exact fp32 path: "simt_fwd_lse", "simt_bwd_grad", "simt_dh", "simt_dw"; and "combine",
 * "finalize", "split_tf32".
 */
const char* lce_kernel_name(int32_t kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H */
