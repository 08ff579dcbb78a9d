/*
 * cbr.h -- C ABI of libcbr.so: the training-mode Conv2d -> BatchNorm -> ReLU (CBR) operator
 * on NVIDIA GB300 (sm_103a), forward, backward and folded inference.
 *
 * What is computed (all citations are to the source pages, by title and section):
 *   z      = conv(x, W)          cross-correlation, no bias, dilation 1
 *                                ("CBR fused operator" (Tech-Renaissance), section 4.1;
 *                                 "TileLang Conv2D+ReLU fusion", basic convolution section)
 *   mean, var over the M = N*P*Q rows of each output channel (biased var for normalising)
 *   inv_std = 1/sqrt(var + eps)
 *   y      = max(0, gamma*(z - mean)*inv_std + beta)        (CBR page, sections 4.2-4.3)
 *   mask   = (gamma*(z - mean)*inv_std + beta > 0), one bit per element (section 4.3, CMP_GT)
 *   running_mean <- (1-momentum)*running_mean + momentum*mean
 *   running_var  <- (1-momentum)*running_var  + momentum*var*M/(M-1)   (unbiased)
 *                                (CBR page section 4.2; "BatchNorm CUDA implementation",
 *                                 section 2.4)
 *   backward: g = dy*mask; dbeta = sum g; dgamma = sum g*xhat;
 *             dz = gamma*inv_std*(g - dbeta/M - xhat*dgamma/M);  dW = wgrad(dz, x);
 *             dx = dgrad(dz, W)   (CBR page sections 5.1-5.3; BatchNorm page section 3.1)
 *   inference: W_fold = W*gamma/sqrt(rv+eps), b_fold = (b - rm)*gamma/sqrt(rv+eps) + beta,
 *             y = relu(conv(x, W_fold) + b_fold)   (CBR page sections 2 and 6;
 *                                                    BatchNorm page section 4.4)
 *
 * Layouts (CBR page, section 8): activations NHWC, filters KRSC ([Cout][R][S][Cin]), both in
 * the storage dtype (fp16 or bf16).  gamma, beta, statistics and dW are fp32.  Output size
 * P = (H + 2*pad - R)/stride + 1, Q likewise.
 *
 * Conventions for every call:
 *   - The caller owns every buffer; pointers are device pointers unless stated otherwise.
 *     The library allocates no device memory on any call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     A returned CBR_OK means the work was validated and enqueued.  Device-side failures
 *     (a bounded wait that ran out) are reported by cbr_stream_status().
 *   - Arguments are validated on the host before anything is enqueued; on any error nothing
 *     is launched and no output is touched.
 *   - Activation / filter / workspace pointers must be 16-byte aligned, fp32 vectors 4-byte.
 *   - No call throws; the library holds no per-call state.
 *   - Supported shapes (else CBR_ERR_UNSUPPORTED): Cout in {16, 32, 64, 128}; and either
 *     stride 1 with Cin a multiple of 8, Cin <= 128, W + 2*pad <= 256; or the first-layer
 *     form Cin = 3 (any stride, R <= 8, S <= 8, pad <= 10, Q <= 128).  Cout % 8 != 0 is
 *     CBR_ERR_INVALID_ARG
 *     (CBR page, section 8: output channels must be a multiple of 8).
 */
#ifndef CBR_H_
#define CBR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cbr_stream_t; /* identical to cudaStream_t */

typedef enum {
  CBR_OK = 0,
  CBR_ERR_INVALID_ARG = 1, /* null pointer, bad shape, bad scalar, dx aliases x, M < 2 */
  CBR_ERR_MISALIGNED = 2,  /* pointer alignment rule violated */
  CBR_ERR_UNSUPPORTED = 3, /* valid arguments outside the shapes/dtypes this library runs */
  CBR_ERR_WORKSPACE = 4,   /* ws_bytes smaller than cbr_workspace_size() requires */
  CBR_ERR_DEVICE = 5,      /* no CUDA device, or the current device is not compute 10.3 */
  CBR_ERR_CUDA = 6,        /* a CUDA runtime / driver call failed */
  CBR_ERR_TIMEOUT = 7      /* (cbr_stream_status) a kernel gave up on a bounded wait */
} cbr_status_t;

typedef enum { CBR_F16 = 0, CBR_BF16 = 1 } cbr_dtype_t;

/* Source of the ReLU mask for cbr_backward. */
typedef enum {
  CBR_MASK_BITS = 0,   /* bit-packed mask written by cbr_forward_train */
  CBR_MASK_FROM_Y = 1, /* recompute the mask as y > 0 from the forward output y */
  CBR_MASK_BYTES = 2   /* one byte per NHWC element, non-zero = active (a standalone ReLU's
                          INT8 mask); packed into the workspace before use */
} cbr_mask_kind_t;

/* One CBR layer.  dtype is a cbr_dtype_t. */
typedef struct {
  int32_t n, h, w, c_in, c_out, r, s, stride, pad;
  int32_t dtype;
} cbr_desc_t;

/* Version of this ABI (major*100 + minor). */
int32_t cbr_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* cbr_status_string(cbr_status_t status);

/*
 * Workspace bytes needed by cbr_forward_train (fwd_bytes) and cbr_backward (bwd_bytes) for
 * `desc`, assuming the caller passes z_saved = NULL (the largest case; with z_saved the calls
 * need less, and check the actual need).  Pure host computation; either output may be NULL.
 * The first 256 bytes of a workspace hold arrival counters: they must be zero the first
 * time a workspace is used (e.g. allocate it zero-filled); every call leaves them at zero.
 */
cbr_status_t cbr_workspace_size(const cbr_desc_t* desc, size_t* fwd_bytes, size_t* bwd_bytes);

/*
 * Training forward (CBR page, sections 4.1-4.3).
 *   x [n][h][w][c_in], w [c_out][r][s][c_in]          storage dtype, read only
 *   gamma, beta [c_out]                                fp32, read only
 *   running_mean, running_var [c_out]                  fp32, updated in place
 *   momentum in [0,1] (weight of the new batch), eps > 0
 *   y [n][p][q][c_out]                                 storage dtype, written
 *   relu_mask: ceil(n*p*q*c_out/32) uint32 words or NULL; bit i of word j is the mask of
 *              NHWC element 32*j + i (bits past the last element are unspecified)
 *   z_saved [n][p][q][c_out] or NULL: receives the conv output; pass it to cbr_backward to
 *              avoid recomputing the convolution there
 *   saved_mean, saved_inv_var [c_out]                  fp32 batch mean and 1/sqrt(var+eps)
 *   ws, ws_bytes                                       workspace (see cbr_workspace_size)
 * Errors: INVALID_ARG (null required pointer, bad desc, momentum/eps out of range,
 * n*p*q < 2), MISALIGNED, UNSUPPORTED, WORKSPACE, DEVICE, CUDA.
 */
cbr_status_t cbr_forward_train(const cbr_desc_t* desc, const void* x, const void* w,
                               const float* gamma, const float* beta, float* running_mean,
                               float* running_var, float momentum, float eps, void* y,
                               uint32_t* relu_mask, void* z_saved, float* saved_mean,
                               float* saved_inv_var, void* ws, size_t ws_bytes,
                               cbr_stream_t stream);

/*
 * The same training forward in one persistent, cooperative kernel launch: the convolution, the
 * statistics, the finalize by the last CTA, then (every CTA waiting, with a time limit, for the
 * finalize) BatchNorm and ReLU applied to the accumulators still held in tensor memory.  z is
 * never re-read (the single-read fusion of the BatchNorm CUDA page, section 4.1).  Arguments,
 * outputs and errors as cbr_forward_train, whose results it reproduces bit for bit (y is
 * computed from the accumulator rounded to the storage dtype, as z is stored).  It takes stride-1
 * convolutions of at most 64 input channels, 32 or 64 output channels, a filter that fits in
 * shared memory, y 32-byte aligned, and batches of at most 4 units of 256 output rows per SM
 * (for example 46 images of 56x56); otherwise it returns CBR_ERR_UNSUPPORTED and does nothing.
 * It is not faster than cbr_forward_train on the measured shapes (the finalize and the apply
 * phase then run one after the other inside one launch); it is there for callers who want one
 * launch per forward.  The runtime refuses the launch (CBR_ERR_CUDA) if the whole grid cannot be
 * resident at once.
 */
cbr_status_t cbr_forward_train_persistent(const cbr_desc_t* desc, const void* x, const void* w,
                                          const float* gamma, const float* beta, float* running_mean,
                                          float* running_var, float momentum, float eps, void* y,
                                          uint32_t* relu_mask, void* z_saved, float* saved_mean,
                                          float* saved_inv_var, void* ws, size_t ws_bytes,
                                          cbr_stream_t stream);

/*
 * Training backward (CBR page, sections 5.1-5.3; BatchNorm page, section 3.1).
 *   dy [n][p][q][c_out]            upstream gradient, storage dtype
 *   x, w                           the forward's inputs
 *   y_or_relu_mask, mask_kind      the forward's relu_mask words (CBR_MASK_BITS, 4-byte
 *                                  aligned), its y (CBR_MASK_FROM_Y) or a byte-per-element
 *                                  mask (CBR_MASK_BYTES, n*p*q*c_out bytes, 16-byte aligned)
 *   z_saved                        the forward's z_saved, or NULL to recompute conv(x, W)
 *   gamma, saved_mean, saved_inv_var   fp32 [c_out] (saved_* from cbr_forward_train)
 *   dx [n][h][w][c_in] or NULL     NULL = first layer: the data gradient is skipped
 *                                  (CBR page, section 5.3).  dx must not overlap x
 *                                  (section 5.2's write-after-read hazard): INVALID_ARG.
 *   dw [c_out][r][s][c_in]         fp32, written
 *   dgamma, dbeta [c_out]          fp32, written
 *   ws, ws_bytes                   workspace (see cbr_workspace_size); it also holds dz, which
 *                                  is evaluated once and read by both convolutions
 * Errors: INVALID_ARG (null required pointer, bad desc or mask_kind, dx overlapping x),
 * MISALIGNED, UNSUPPORTED (also: dx requested with a non-square filter or pad > R-1, or for
 * the 3-channel first layer), WORKSPACE, DEVICE, CUDA.
 */
cbr_status_t cbr_backward(const cbr_desc_t* desc, const void* dy, const void* x, const void* w,
                          const void* y_or_relu_mask, int32_t mask_kind, const void* z_saved,
                          const float* gamma, const float* saved_mean,
                          const float* saved_inv_var, void* dx, float* dw, float* dgamma,
                          float* dbeta, void* ws, size_t ws_bytes, cbr_stream_t stream);

/*
 * Synchronised BatchNorm across data-parallel ranks ("BatchNorm CUDA implementation",
 * section 7.1: the per-channel statistics of every rank's share of the batch are combined
 * before normalising, and so are the backward's per-channel sums).  Each call pair brackets
 * one collective that the caller runs (e.g. with NCCL); the library itself stays on one GPU.
 *
 * Forward, first half: conv and this rank's statistics, no finalize and no apply.
 *   z [n][p][q][c_out]     the conv output (required: the second half normalises it)
 *   moments [2*c_out + 1]  fp32 out: per-channel mean [c_out], M2 (sum of squared deviations
 *                          from the mean) [c_out], then this rank's row count n*p*q
 *   ws, ws_bytes           the forward workspace (cbr_workspace_size's fwd_bytes suffices)
 * The caller gathers every rank's moments, in rank order, into moments_all
 * [world][2*c_out + 1] (an all-gather, not a sum: moments merge exactly, sums of squares
 * would cancel), then calls
 * Forward, second half: merges the `world` moment sets in that order (Chan's parallel
 * formula), writes saved_mean / saved_inv_var, updates the running statistics with the
 * global unbiased variance (M = the sum of the counts), and applies BN + ReLU to this rank's z,
 * as cbr_forward_train does.  Every rank computes identical statistics.
 * Errors: INVALID_ARG (NULL, world < 1, momentum / eps out of range), MISALIGNED,
 * UNSUPPORTED, WORKSPACE, DEVICE, CUDA.
 */
cbr_status_t cbr_forward_train_stats(const cbr_desc_t* desc, const void* x, const void* w, void* z,
                                     float* moments, void* ws, size_t ws_bytes, cbr_stream_t stream);
cbr_status_t cbr_forward_train_finish(const cbr_desc_t* desc, const float* moments_all, int32_t world,
                                      const float* gamma, const float* beta, float* running_mean,
                                      float* running_var, float momentum, float eps, const void* z,
                                      void* y, uint32_t* relu_mask, float* saved_mean,
                                      float* saved_inv_var, void* ws, size_t ws_bytes,
                                      cbr_stream_t stream);

/*
 * Backward, first half: this rank's masked per-channel sums, written to sums [2*c_out] as
 * [sum of dy*mask][sum of dy*mask*(z - saved_mean)] (saved_mean: the merged mean from
 * cbr_forward_train_finish; z and the mask as for cbr_backward; ws: the backward workspace).
 * The caller sums them over the ranks (an all-reduce) into sums_all and calls
 * Backward, second half: dgamma, dbeta and the BN data gradient from the global sums over
 * m_total = the global n*p*q, then wgrad and dgrad of this rank's share, as cbr_backward does.
 * dgamma and dbeta are the global ones (identical on every rank); dW is this rank's share (the
 * caller's data-parallel gradient all-reduce sums it).
 * Errors as for cbr_backward, and INVALID_ARG for a NULL sums / sums_all or m_total < 2.
 */
cbr_status_t cbr_backward_sums(const cbr_desc_t* desc, const void* dy, const void* y_or_relu_mask,
                               int32_t mask_kind, const void* z_saved, const float* saved_mean,
                               float* sums, void* ws, size_t ws_bytes, cbr_stream_t stream);
cbr_status_t cbr_backward_finish(const cbr_desc_t* desc, const float* sums_all, int64_t m_total,
                                 const void* dy, const void* x, const void* w,
                                 const void* y_or_relu_mask, int32_t mask_kind, const void* z_saved,
                                 const float* gamma, const float* saved_mean,
                                 const float* saved_inv_var, void* dx, float* dw, float* dgamma,
                                 float* dbeta, void* ws, size_t ws_bytes, cbr_stream_t stream);

/*
 * BN folding for inference (CBR page, section 2; BatchNorm page, section 4.4):
 *   w_fold[k,...] = w[k,...]*gamma[k]/sqrt(running_var[k]+eps)   (computed in fp32, stored
 *                   rounded to the storage dtype, same layout as w)
 *   b_fold[k]     = (conv_bias[k] - running_mean[k])*gamma[k]/sqrt(running_var[k]+eps)
 *                   + beta[k]                                    (fp32; conv_bias may be NULL)
 */
cbr_status_t cbr_fold_bn(const cbr_desc_t* desc, const void* w, const float* conv_bias,
                         const float* gamma, const float* beta, const float* running_mean,
                         const float* running_var, float eps, void* w_fold, float* b_fold,
                         cbr_stream_t stream);

/*
 * Folded inference forward (CBR page, section 6): y = relu(conv(x, w_fold) + b_fold), with
 * the bias and ReLU applied to the fp32 accumulator before rounding.
 */
cbr_status_t cbr_forward_infer(const cbr_desc_t* desc, const void* x, const void* w_fold,
                               const float* b_fold, void* y, cbr_stream_t stream);

/*
 * Inference with BatchNorm applied to the convolution's fp32 accumulator, the CBR page's
 * single-graph form (section 6: conv, MUL by eq_scale, ADD eq_bias, ReLU):
 *   y = relu(conv(x, w)*scale + shift),  scale = gamma/sqrt(running_var + eps),
 *   shift = beta + (conv_bias - running_mean)*scale          (conv_bias may be NULL: 0)
 * Unlike cbr_fold_bn + cbr_forward_infer, the filter is used as trained, so nothing is rounded
 * to the storage dtype before the convolution.  Stride-1 layers only: the 3-channel first layer
 * returns UNSUPPORTED (fold it instead).  Errors: INVALID_ARG (NULL, eps <= 0), MISALIGNED,
 * UNSUPPORTED, DEVICE, CUDA.
 */
cbr_status_t cbr_forward_infer_bn(const cbr_desc_t* desc, const void* x, const void* w,
                                  const float* conv_bias, const float* gamma, const float* beta,
                                  const float* running_mean, const float* running_var, float eps,
                                  void* y, cbr_stream_t stream);

/*
 * Training forward that allocates nothing and takes no workspace.  The pages have no
 * counterpart; this exists for callers that must not allocate device memory on their
 * execution path, such as plug-ins that run inside another framework's execution loop with
 * no access to its allocator, or latency-critical loops where cudaMalloc's cost and implicit
 * synchronisation are unacceptable.
 *   Same arguments and results as cbr_forward_train, except: no ws / ws_bytes, and z_saved
 *   is required (INVALID_ARG when NULL), because the conv output cannot live in the fixed
 *   scratch.
 *   Scratch: a 320 KiB array compiled into the library, held by every GPU that loads it
 *   until the process exits.  A problem whose scratch need exceeds it returns
 *   CBR_ERR_WORKSPACE before anything is enqueued (with Cout <= 128 the need is about
 *   261 KiB, so supported shapes fit).
 *   The first call on each device looks up the array's device address (one
 *   cudaGetSymbolAddress with that device current); make that first call before any stream
 *   capture.  Each call clears the array's arrival counters with an asynchronous memset on
 *   `stream`.  All calls share the one array: calls that overlap on the GPU (different streams
 *   without ordering) race and give undefined results.  No cudaMalloc, cudaFree or other
 *   allocating routine is called.
 */
cbr_status_t cbr_forward_train_noalloc(const cbr_desc_t* desc, const void* x, const void* w,
                                       const float* gamma, const float* beta, float* running_mean,
                                       float* running_var, float momentum, float eps, void* y,
                                       uint32_t* relu_mask, void* z_saved, float* saved_mean,
                                       float* saved_inv_var, cbr_stream_t stream);

/*
 * ReLU-mask transcoding between this library's bit-packed mask (bit i of 32-bit word j is NHWC
 * element 32*j + i) and one byte per element (0 or 1), the form a standalone ReLU keeps
 * (CBR page, sections 8 and 9: the fused operator's BOOLEAN mask against the standalone
 * ReLU's INT8 mask, transcoded by its equivalence tests).
 *   count       elements (>= 0; 0 is a no-op)
 *   bits        ceil(count/32) uint32 words, 4-byte aligned
 *   bytes       count bytes, 16-byte aligned
 * cbr_mask_bits_to_bytes writes 0 or 1 per element.  cbr_mask_bytes_to_bits sets a bit for
 * every non-zero byte and writes the bits past `count` in the last word as 0.  Asynchronous on
 * `stream`.  Errors: INVALID_ARG (count < 0, or a NULL buffer with count > 0), MISALIGNED,
 * DEVICE, CUDA.
 */
cbr_status_t cbr_mask_bits_to_bytes(const uint32_t* bits, uint8_t* bytes, int64_t count,
                                    cbr_stream_t stream);
cbr_status_t cbr_mask_bytes_to_bits(const uint8_t* bytes, uint32_t* bits, int64_t count,
                                    cbr_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device error word of the current device.
 * Returns CBR_OK, CBR_ERR_TIMEOUT if a kernel abandoned a bounded wait (its outputs are then
 * undefined), or CBR_ERR_CUDA if the stream reports a CUDA error.
 */
cbr_status_t cbr_stream_status(cbr_stream_t stream);

/*
 * Failure-detection self-test (the pages have no counterpart; it exercises the library's own
 * error path).  Launches one warp on `stream` that waits, with the same bounded barrier wait
 * the library's kernels use, on a barrier nothing completes; after `limit_us` microseconds it
 * gives up, records the timeout in the device error word and exits.  The following
 * cbr_stream_status(stream) then returns CBR_ERR_TIMEOUT and clears the word, and the CUDA
 * context stays usable: no fault, trap or hang is involved.  Returns CBR_ERR_INVALID_ARG unless
 * 1 <= limit_us <= 1,000,000, CBR_ERR_DEVICE if the current device is not compute 10.3, else
 * CBR_OK (the wait itself runs asynchronously).
 */
cbr_status_t cbr_selftest_bounded_wait(int32_t limit_us, cbr_stream_t stream);

/*
 * Profiling hook for the calling host thread.  When `events` is non-NULL, the next
 * cbr_forward_train / cbr_backward / cbr_forward_infer call records events[0] before its
 * first kernel and events[i] after its i-th kernel (cudaEvent_t handles owned by the caller,
 * at most `count`), then clears the hook.  cbr_profile_last_count() returns how many events
 * that call recorded.  Used to time each kernel inside the real calls.  When the call is made
 * while its stream is being captured into a CUDA graph, the events are recorded as external
 * event-record nodes (cudaEventRecordExternal), so they timestamp every replay of the graph.
 */
cbr_status_t cbr_profile_next_call(void* const* events, int32_t count);
int32_t cbr_profile_last_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CBR_H_ */
