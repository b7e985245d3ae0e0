/*
 * ccv.h -- C ABI of the GB300 causal depthwise conv1d library (libccv.so).
 *
 * The operation ("Chapter 5: Dao forward CUDA implementation", section
 * "exchanging history"; "Chapter 4: Dao interface and source map", section
 * "interface contract"):
 *
 *     out[b,c,t] = act( bias[c] + sum_{k=0}^{K-1} weight[c,k] * h[b,c,t-K+1+k] )
 *
 * where h is the history-extended input: h[b,c,j] = x[b,c,j] for j >= 0 and,
 * for j < 0, initial_states[b,c,K-1+j] when given, else 0 ("Chapter 5",
 * section "three kinds of boundary").  weight[c,0] multiplies the OLDEST input
 * of the window and weight[c,K-1] the current one.  The sum is accumulated in
 * FP32; act is the identity or SiLU(z) = z * sigmoid(z) ("silu" and "swish"
 * name the same activation), applied before rounding to the output dtype
 * (round to nearest even).
 *
 * Memory model.  Every tensor is described by a device pointer to its logical
 * element [0,...,0] and signed strides counted in ELEMENTS, so that element
 * [b,c,t] of x lives at x + b*x_strides[0] + c*x_strides[1] + t*x_strides[2]
 * ("Chapter 4", section "two layouts").  Contiguous [B,C,L] (strides
 * (C*L, L, 1)), channel-last [B,L,C] seen as [B,C,L] (strides (L*C, 1, C)) and
 * sliced views whose time stride exceeds C are all accepted as they are; the
 * library never repacks, never copies to a staging buffer and never
 * allocates memory.  The caller owns every buffer, including out and
 * final_states_out.
 *
 * Execution.  ccv_fwd validates its arguments on the host (no device
 * synchronisation, no device memory access), picks a kernel from the strides
 * and alignment, and enqueues it on `stream` (a cudaStream_t; NULL means the
 * legacy default stream of the current device).  It returns as soon as the
 * launch is queued.  All pointers must be device-accessible memory of the
 * current device.  The forward and backward kernels are launched with
 * programmatic stream serialization: a kernel may become resident while the
 * previous kernel on the stream drains, but it waits for that kernel to
 * complete before it reads or writes any global memory, so ordering against
 * earlier and later work on the stream is the ordinary stream order (the
 * decode step, ccv_update, is launched plainly).
 *
 * Errors.  On any validation error nothing is launched and a non-zero
 * ccv_status is returned; ccv_last_error() then describes it.  A failed launch
 * returns CCV_ERR_CUDA.  Faults raised later by the kernel (for example from
 * a pointer that does not cover the described extent) surface on the stream
 * like any CUDA error.
 *
 * Thread safety.  All entry points may be called concurrently from several
 * host threads; the error message is kept per thread.
 */
#ifndef CCV_H_
#define CCV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage dtype of x, out, weight, bias, initial_states and final_states_out
 * (one dtype for all of them in ccv_fwd, ccv_update and ccv_bwd; the _mixed
 * entry points take a separate dtype for weight and bias). */
typedef enum {
  CCV_F32 = 0,  /* IEEE binary32 */
  CCV_F16 = 1,  /* IEEE binary16 */
  CCV_BF16 = 2  /* bfloat16 */
} ccv_dtype;

/* Activation applied after the FP32 accumulation ("Chapter 4", section
 * "interface contract": None, "silu" or "swish", the last two identical). */
typedef enum {
  CCV_ACT_NONE = 0,
  CCV_ACT_SILU = 1
} ccv_activation;

typedef enum {
  CCV_OK = 0,
  CCV_ERR_INVALID_ARG = 1,  /* malformed arguments; nothing was launched */
  CCV_ERR_UNSUPPORTED = 2,  /* well-formed but not provided (K outside 2..4,
                               seq_idx together with initial_states) */
  CCV_ERR_CUDA = 3          /* the CUDA runtime reported an error */
} ccv_status;

/*
 * ccv_fwd -- causal depthwise conv1d forward pass.
 *
 *   x                 [B,C,L] input, strides x_strides (elements).
 *   out               [B,C,L] output, strides out_strides.  Must not share
 *                     memory with x, initial_states or final_states_out; an
 *                     exact alias (out == x) and a distinct output that
 *                     repeats some element (a zero stride on a dimension of
 *                     size > 1) are rejected.  Fastest when out has the same
 *                     unit-stride dimension as x.
 *   weight            [C,K] taps, oldest first, strides weight_strides.
 *   bias              [C] or NULL, element stride bias_stride.
 *   seq_idx           int32 [B,L] or NULL, strides seq_idx_strides.  A window
 *                     term contributes only when seq_idx at its source
 *                     position equals seq_idx at the output position (packed
 *                     sequences, "Chapter 5", section "three kinds of
 *                     boundary").  Only equality of ids matters.
 *   initial_states    [B,C,K-1] or NULL, oldest first, strides
 *                     initial_states_strides.  Rejected (CCV_ERR_UNSUPPORTED)
 *                     together with seq_idx.
 *   final_states_out  [B,C,K-1] or NULL; receives h[b,c,L-K+1 .. L-1], the
 *                     last K-1 raw INPUTS (not activated outputs), copied bit
 *                     for bit; taken from initial_states (or zeros) where
 *                     L < K-1.
 *   B, C, L           sizes, >= 0.  B == 0 or C == 0 is a no-op; L == 0 only
 *                     writes final_states_out.
 *   K                 kernel width, 2, 3 or 4.
 *   dtype, activation see above.
 *   stream            cudaStream_t to enqueue on (NULL: default stream).
 *
 * Every strides pointer must be non-NULL when its tensor pointer is.  Data
 * pointers must be aligned to the element size.  Strides are arbitrary signed
 * integers; the extents they describe must fit in int64.
 */
ccv_status ccv_fwd(const void* x, const int64_t x_strides[3],
                   void* out, const int64_t out_strides[3],
                   const void* weight, const int64_t weight_strides[2],
                   const void* bias, int64_t bias_stride,
                   const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                   const void* initial_states, const int64_t initial_states_strides[3],
                   void* final_states_out, const int64_t final_states_strides[3],
                   int64_t B, int64_t C, int64_t L, int K,
                   ccv_dtype dtype, ccv_activation activation, void* stream);

/*
 * ccv_update -- decode step: advance a convolution state by S new inputs, in
 * place ("Chapter 4: Dao interface and source map", section "source map": the
 * update kernel reads the history and advances the state in place).
 *
 * Defined as the forward pass with initial_states = conv_state whose
 * final_states are written back into conv_state:
 *     out[b,c,s] = act(bias[c] + sum_k weight[c,k] * h[b,c,s-K+1+k]),
 *     h = conv_state[b,c,:] ++ x[b,c,:],
 *     conv_state[b,c,:] <- the last K-1 values of h (raw inputs, bit for bit).
 *
 *   x            [B,C,S] new inputs (S is usually 1), strides x_strides.
 *   out          [B,C,S] outputs, strides out_strides; must not alias x or
 *                conv_state.
 *   conv_state   [B,C,K-1], oldest first, read and then overwritten.
 *   weight, bias, K, dtype, activation, stream: as for ccv_fwd.
 * S == 0 leaves the state unchanged; B == 0 or C == 0 is a no-op.  Errors as
 * for ccv_fwd.  One thread per (b, c) row; the call is asynchronous.
 */
ccv_status ccv_update(const void* x, const int64_t x_strides[3],
                      void* out, const int64_t out_strides[3],
                      void* conv_state, const int64_t state_strides[3],
                      const void* weight, const int64_t weight_strides[2],
                      const void* bias, int64_t bias_stride,
                      int64_t B, int64_t C, int64_t S, int K,
                      ccv_dtype dtype, ccv_activation activation, void* stream);

/*
 * ccv_bwd_workspace_size -- bytes of device workspace ccv_bwd needs.
 *
 * The parameter gradients are reductions over b and t.  ccv_bwd makes them in
 * two launches without atomics: the main kernel writes one FP32 partial sum
 * per (time partition, tap, channel) into the workspace, and a second kernel
 * adds the partials in a fixed order, so results are bitwise reproducible.
 * The partition depends only on the layout class of x, dout and dx (unit time
 * stride, unit channel stride, other) and on B, C, L, K, so the size can be
 * queried before the buffers exist.  Pass the same strides and sizes as to
 * ccv_bwd.  Writes 0 when no reduction is needed (B, C or L is 0).  Host only.
 */
ccv_status ccv_bwd_workspace_size(const int64_t x_strides[3], const int64_t dout_strides[3],
                                  const int64_t dx_strides[3], int64_t B, int64_t C, int64_t L,
                                  int K, ccv_dtype dtype, uint64_t* bytes);

/*
 * ccv_bwd -- causal depthwise conv1d backward pass ("Chapter 4: Dao interface
 * and source map", section "autograd": the backward recomputes from the saved
 * x, weight, bias, seq_idx and initial_states, receives dout and, when the
 * forward returned final states, dfinal_states; dweight and dbias are
 * accumulated in FP32 and then returned in the parameter dtype).
 *
 * With z the forward pre-activation (recomputed here, FP32) and
 * dz[b,c,t] = dout[b,c,t] * act'(z[b,c,t]):
 *     dx[b,c,j]        = sum over the taps (t, k) that read h[b,c,j] of weight[c,k] * dz[b,c,t]
 *                        + dfinal_states[b,c,j-L+K-1]   (where final_states copies h[b,c,j])
 *     dweight[c,k]     = sum_{b,t} dz[b,c,t] * h[b,c,t-K+1+k]   (taps the forward used)
 *     dbias[c]         = sum_{b,t} dz[b,c,t]
 *     dinitial_states  = the same as dx for the history positions j < 0.
 * With seq_idx the forward's masks apply to every term.
 *
 *   x, weight, bias, seq_idx, initial_states, K, dtype, activation: the
 *                     forward pass's arguments, as for ccv_fwd.
 *   dout              [B,C,L] gradient of out, strides dout_strides.
 *   dfinal_states     [B,C,K-1] gradient of final_states, or NULL (zero).
 *   dx                [B,C,L] output, required.  Must not share memory with
 *                     any input (in-place over dout is rejected).
 *   dweight           [C,K] output or NULL, strides dweight_strides.
 *   dbias             [C] output or NULL, element stride dbias_stride.
 *   dinitial_states   [B,C,K-1] output or NULL; needs initial_states.
 *   workspace         device buffer of at least ccv_bwd_workspace_size()
 *                     bytes, 16-byte aligned, owned by the caller; needed
 *                     when dweight or dbias is requested (otherwise it may be
 *                     NULL).  Its contents need not be initialised and are
 *                     undefined afterwards.  Two calls in flight at the same
 *                     time must not share a workspace.
 *
 * Gradients are written in dtype (rounded to nearest even from FP32).  Errors
 * as for ccv_fwd; a workspace that is too small is CCV_ERR_INVALID_ARG and
 * the message gives the required size.  Asynchronous: at most two kernels are
 * enqueued on `stream`.
 */
ccv_status ccv_bwd(const void* x, const int64_t x_strides[3],
                   const void* weight, const int64_t weight_strides[2],
                   const void* bias, int64_t bias_stride,
                   const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                   const void* initial_states, const int64_t initial_states_strides[3],
                   const void* dout, const int64_t dout_strides[3],
                   const void* dfinal_states, const int64_t dfinal_states_strides[3],
                   void* dx, const int64_t dx_strides[3],
                   void* dweight, const int64_t dweight_strides[2],
                   void* dbias, int64_t dbias_stride,
                   void* dinitial_states, const int64_t dinitial_states_strides[3],
                   void* workspace, uint64_t workspace_bytes,
                   int64_t B, int64_t C, int64_t L, int K,
                   ccv_dtype dtype, ccv_activation activation, void* stream);

/*
 * ccv_bwd_noalloc -- ccv_bwd without a caller workspace.
 *
 * The pages have no counterpart of this entry point: it is an operational
 * variant of ccv_bwd for callers that cannot allocate device memory where they
 * call the backward pass -- plain C hosts that receive only the tensors
 * themselves and have no device allocator at hand, or services that reserve
 * all device memory at start-up and must not grow it afterwards.  It takes the
 * same arguments as ccv_bwd except the workspace and computes the same
 * results with the same kernels.
 *
 * Scratch.  The parameter-gradient partials go to one 16 MiB scratch array
 * that is part of the library's device image (one per device, present from
 * module load).  Nothing in it has to start at zero: every slot a call uses is
 * written before it is read.  A problem whose ccv_bwd_workspace_size()
 * exceeds 16 MiB is rejected with CCV_ERR_INVALID_ARG before anything is
 * launched (use ccv_bwd with a workspace for it); when neither dweight nor
 * dbias is requested the scratch is not used.
 *
 * Set-up.  A call made outside stream capture looks up the scratch address
 * (cudaGetSymbolAddress, with the caller's device and context current; this
 * allocates nothing) and records it with that context.  A call made during
 * stream capture uses the address recorded for the current context and
 * fails with CCV_ERR_INVALID_ARG when there is none: make one call on each
 * device (and in each context, e.g. again after cudaDeviceReset) before
 * starting a stream capture there.
 *
 * Concurrency.  All calls on one device share the one scratch.  Two calls
 * whose kernels can overlap (issued on different streams, or from different
 * host threads without ordering) race on it and may return wrong dweight and
 * dbias.  Issue them on one stream, which orders them, or give each its own
 * workspace through ccv_bwd.
 *
 * Errors as for ccv_bwd; asynchronous like ccv_bwd.
 */
ccv_status ccv_bwd_noalloc(const void* x, const int64_t x_strides[3],
                           const void* weight, const int64_t weight_strides[2],
                           const void* bias, int64_t bias_stride,
                           const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                           const void* initial_states, const int64_t initial_states_strides[3],
                           const void* dout, const int64_t dout_strides[3],
                           const void* dfinal_states, const int64_t dfinal_states_strides[3],
                           void* dx, const int64_t dx_strides[3],
                           void* dweight, const int64_t dweight_strides[2],
                           void* dbias, int64_t dbias_stride,
                           void* dinitial_states, const int64_t dinitial_states_strides[3],
                           int64_t B, int64_t C, int64_t L, int K,
                           ccv_dtype dtype, ccv_activation activation, void* stream);

/*
 * Separate weight dtype ("Chapter 4: Dao interface and source map", section
 * "v1.5.0 restrictions": input and weight dtypes are dispatched separately,
 * the bias has the weight dtype, the states have the input dtype).
 *
 * ccv_fwd_mixed, ccv_update_mixed and ccv_bwd_mixed take the same arguments
 * as ccv_fwd, ccv_update and ccv_bwd plus weight_dtype, the format of weight
 * and bias (and of dweight and dbias for ccv_bwd_mixed).  x, out, the states,
 * dout, dx and the state gradients keep `dtype`.  Any of the nine pairs of
 * F32 / F16 / BF16 is accepted.  Every value is widened exactly to FP32 from
 * its own format and accumulated in FP32 as in the one-dtype calls; outputs
 * are rounded once to `dtype` (dweight, dbias to weight_dtype).  The pages'
 * reference function instead casts x to the weight dtype first; that cast is
 * not made here, so results can differ from it by that rounding.  Errors and
 * execution as for the one-dtype calls; weight and bias pointers must be
 * aligned to the weight element size.
 */
ccv_status ccv_fwd_mixed(const void* x, const int64_t x_strides[3],
                         void* out, const int64_t out_strides[3],
                         const void* weight, const int64_t weight_strides[2],
                         const void* bias, int64_t bias_stride,
                         const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                         const void* initial_states, const int64_t initial_states_strides[3],
                         void* final_states_out, const int64_t final_states_strides[3],
                         int64_t B, int64_t C, int64_t L, int K,
                         ccv_dtype dtype, ccv_dtype weight_dtype, ccv_activation activation, void* stream);

ccv_status ccv_update_mixed(const void* x, const int64_t x_strides[3],
                            void* out, const int64_t out_strides[3],
                            void* conv_state, const int64_t state_strides[3],
                            const void* weight, const int64_t weight_strides[2],
                            const void* bias, int64_t bias_stride,
                            int64_t B, int64_t C, int64_t S, int K,
                            ccv_dtype dtype, ccv_dtype weight_dtype, ccv_activation activation, void* stream);

ccv_status ccv_bwd_mixed(const void* x, const int64_t x_strides[3],
                         const void* weight, const int64_t weight_strides[2],
                         const void* bias, int64_t bias_stride,
                         const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                         const void* initial_states, const int64_t initial_states_strides[3],
                         const void* dout, const int64_t dout_strides[3],
                         const void* dfinal_states, const int64_t dfinal_states_strides[3],
                         void* dx, const int64_t dx_strides[3],
                         void* dweight, const int64_t dweight_strides[2],
                         void* dbias, int64_t dbias_stride,
                         void* dinitial_states, const int64_t dinitial_states_strides[3],
                         void* workspace, uint64_t workspace_bytes,
                         int64_t B, int64_t C, int64_t L, int K,
                         ccv_dtype dtype, ccv_dtype weight_dtype, ccv_activation activation, void* stream);

/* Message for the last non-OK status returned on the calling thread ("" if
 * none).  The pointer stays valid until the next ccv_* call on that thread. */
const char* ccv_last_error(void);

/* Name of the kernel variant the last successful ccv_fwd, ccv_update or
 * ccv_bwd on this thread enqueued (e.g. "time_vec", "chlast_tma",
 * "chlast_vec", "generic", "update", "bwd_time", "bwd_chlast",
 * "bwd_generic", "none"). */
const char* ccv_last_kernel(void);

/* Library ABI version: (major << 16) | minor. */
int ccv_version(void);

/*
 * ccv_device_fault -- read and clear the fault word of the current device.
 *
 * Kernels that stage data through shared-memory barriers bound every wait;
 * a wait that runs out of its budget (seconds) sets a bit here, the kernel
 * stops early and its outputs are incomplete.  0 means no fault since the
 * last call.  Bits: 1 consumer wait, 2 producer wait, 4 drain wait.
 * Synchronous (it copies one word from the device); not part of the
 * operation on the pages, an operational check of this library.
 */
ccv_status ccv_device_fault(unsigned* fault_bits);

/*
 * ccv_test_bounded_wait -- exercise the bounded-wait path of the channel-last
 * TMA kernel without a fault.
 *
 * The next ccv_fwd / ccv_fwd_mixed call of this process that runs the
 * channel-last TMA kernel (ccv_last_kernel() == "chlast_tma") bounds every
 * barrier wait by `wait_budget_cycles` SM clock cycles instead of seconds and
 * does not issue the tensor copy of stage `skip_stage` (0-based, in the order
 * the stages are consumed) of its first warp.  That warp's wait for the stage
 * then runs out: it sets fault bit 1 (see ccv_device_fault), waits for the
 * copies it did issue and returns, leaving its share of the output unwritten;
 * every other warp completes.  Nothing is issued that could fault: the left
 * out copy is simply never started.  The setting applies to one launch and is
 * then cleared; wait_budget_cycles <= 0 clears a pending setting.  Not part
 * of the operation on the pages: a test hook for this library's own
 * failure handling.  Returns CCV_ERR_INVALID_ARG for skip_stage < 0.
 */
ccv_status ccv_test_bounded_wait(int64_t wait_budget_cycles, int64_t skip_stage);

#ifdef __cplusplus
}
#endif

#endif /* CCV_H_ */
