/*
 * ssm.h -- C ABI of the B300 (sm_103a) selective-scan library (libssm_b300.so).
 *
 * Two operations of the Mamba selective state-space layer, both hand-written CUDA:
 *
 *   ssm_selective_scan_fwd   the fused forward pass over a whole sequence
 *                            (_ws: with a workspace; _ex: from a given start state
 *                            and/or with the zero-order-hold B-bar; _noalloc: with
 *                            built-in scratch)
 *   ssm_state_update         the single-token recurrent update used in decoding
 *                            (_ex: with the step-size bias and softplus applied,
 *                            optionally the zero-order-hold B-bar)
 *   ssm_conv_selective_scan_fwd, ssm_conv_state_update
 *                            the same two with the block's causal width-4 depthwise
 *                            conv + SiLU (the step before the SSM) fused in front
 *   ssm_selective_scan_bwd   the backward pass of the forward pass (all gradients);
 *                            ssm_selective_scan_fwd_train + ssm_selective_scan_bwd_ex:
 *                            the forward pass writing the backward's state checkpoints
 *   ssm_ssd_fwd              the Mamba-2 SSD forward pass (scalar decay per head,
 *                            chunked, tensor cores)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are described by ssm_tensor_t: a DEVICE pointer, an element type and a
 *    shape. Storage is dense row-major (last index fastest); there are no strides.
 *  - Ownership: the caller owns every buffer. The library allocates nothing, frees
 *    nothing and never synchronises; work is enqueued on the caller's stream
 *    (a cudaStream_t passed as void*, NULL = legacy default stream).
 *  - Errors: all arguments are validated on the host before anything is enqueued.
 *    Any status other than SSM_OK means nothing was launched and no output was
 *    written. A failed launch returns SSM_ERR_CUDA (from cudaGetLastError).
 *  - Pointers must be aligned to their element size; ssm_state_update also needs
 *    state and A 16-byte aligned. Faster kernel variants are chosen when every
 *    pointer is 16-byte aligned (a fresh PyTorch allocation always is).
 *  - Outputs must not overlap any input (SSM_ERR_LAYOUT), except where an entry point
 *    says it updates a tensor in place.
 *  - Every I/O tensor (u, delta, z, B, C, x) of one call has the same element type,
 *    SSM_BF16 or SSM_F32. A, D, delta_bias and the states are always SSM_F32.
 *    The output y has the I/O type or SSM_F32 (full-precision output of a bf16 call).
 *  - Arithmetic: fp32 throughout (state, discretisation, contraction); bf16 outputs
 *    are rounded to nearest-even from fp32.
 *  - N (state size) must be 4, 8 or 16, else SSM_ERR_UNSUPPORTED.
 */
#ifndef SSM_B300_H
#define SSM_B300_H

#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

typedef struct {
  void* data;          /* device pointer; may be NULL only when the tensor is empty */
  ssm_dtype_t dtype;
  int32_t ndim;        /* number of valid entries in shape[] */
  int64_t shape[3];
} ssm_tensor_t;

typedef enum {
  SSM_OK = 0,
  SSM_ERR_NULL = 1,            /* a required descriptor or data pointer is NULL */
  SSM_ERR_SHAPE = 2,           /* ndim or a dimension does not match the contract */
  SSM_ERR_DTYPE = 3,           /* element type not allowed, or I/O types differ */
  SSM_ERR_LAYOUT = 4,          /* misaligned pointer, or an output overlaps an input */
  SSM_ERR_UNSUPPORTED = 5,     /* a valid request this build does not implement (e.g. N) */
  SSM_ERR_CUDA = 6,            /* the CUDA runtime reported an error at launch */
  SSM_ERR_DEVICE_TIMEOUT = 7   /* a kernel gave up a bounded wait (see ssm_device_error) */
} ssm_status_t;

/*
 * ssm_selective_scan_fwd -- fused selective-scan forward pass.
 *
 * For each batch row b and channel d, from h = 0 ("8.7 State Space Models (Mamba)",
 * section 2.1, h(0) = 0), for t = 0 .. L-1:
 *   dt        = delta_softplus ? softplus(delta[b,t,d] + bias[d]) : delta[b,t,d] + bias[d]
 *   h[n]      = exp(dt * A[d,n]) * h[n] + dt * B[b,t,n] * u[b,t,d]      (n = 0 .. N-1)
 *   v         = sum_n C[b,t,n] * h[n] + D[d] * u[b,t,d]
 *   y[b,t,d]  = z ? v * silu(z[b,t,d]) : v
 * and finally last_state[b,d,:] = h.
 * Sources: "Mamba and State Space Models" (placement-prep chapter), sections
 * "Selective scan pseudo-code" (the recurrence and read-out) and "Discretization and
 * initialization details" (A-bar = exp(Delta A), B-bar = Delta B, Delta = softplus(Wx + b));
 * "Arch 02: Mamba SSM" deck, continuous form y = Cx + Du (the D skip) and the selective
 * SSM block (per-token B, C of shape (B, L, N)); "8.7 State Space Models (Mamba)",
 * section 6 (the SiLU(z) gate on the SSM output).
 *
 *   u          (batch, L, D)  I/O type        input sequence
 *   delta      (batch, L, D)  I/O type        raw step size (before bias and softplus)
 *   A          (D, N)         f32             diagonal state matrix (any values; normally < 0)
 *   B, C       (batch, L, N)  I/O type        per-token input / output projections
 *   D          (D)            f32, nullable   skip weight (NULL = no skip)
 *   z          (batch, L, D)  I/O type, nullable   gate input (NULL = no gate)
 *   delta_bias (D)            f32, nullable   added to delta before softplus (NULL = 0)
 *   delta_softplus            0 or 1
 *   y          (batch, L, D)  I/O type or f32   output, written
 *   last_state (batch, D, N)  f32, nullable   final state, written (NULL = not written)
 *   stream                    cudaStream_t
 * batch == 0 or L == 0 is a valid no-op; with L == 0 a non-NULL last_state is zeroed.
 * The per-step state never reaches global memory.
 * Long sequences over few channels (too few channel blocks to fill the GPU) run as
 * parallel sequence segments: an aggregate pass gives each segment's end state from zero
 * and its decay product exp(A * sum of dt), a warp scan with the associative operator
 * (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) gives every segment its start state ("8.7
 * State Space Models (Mamba)", section 4.1), and the full pass produces y. Without a
 * workspace those per-segment values live in y itself (each channel's own column of its
 * segment's first rows, overwritten by the full pass), so nothing is allocated. Segments
 * reassociate the recurrence (equal up to rounding); SSM_B300_SEGMENTS=0 in the
 * environment turns them off, for callers who need a prefix plus its continuation to
 * reproduce one pass bit for bit.
 */
SSM_API ssm_status_t ssm_selective_scan_fwd(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                    const ssm_tensor_t* A, const ssm_tensor_t* B,
                                    const ssm_tensor_t* C, const ssm_tensor_t* D,
                                    const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                    int delta_softplus, ssm_tensor_t* y,
                                    ssm_tensor_t* last_state, void* stream);

/*
 * ssm_selective_scan_fwd_workspace_size -- bytes of device workspace that
 * ssm_selective_scan_fwd_ws can use for a problem of this shape (0: none needed).
 * A workspace lets shapes with few channels and a long sequence (for example one
 * sequence of 131072 steps over 2048 channels) cut the sequence into segments that run
 * in parallel: a first pass computes each segment's end state from zero and its decay
 * product exp(A * sum of dt), an associative scan over segments with the operator
 * (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) gives every segment its start state
 * ("8.7 State Space Models (Mamba)", section 4.1; "Mamba and State Space Models",
 * "Hardware-Aware Parallel Scan"), and a second pass produces y. The answer depends only
 * on the shape and the current device. Returns SSM_OK, SSM_ERR_NULL (bytes == NULL) or
 * SSM_ERR_SHAPE (negative sizes).
 */
SSM_API ssm_status_t ssm_selective_scan_fwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N,
                                                          size_t* bytes);

/*
 * ssm_selective_scan_fwd_ws -- ssm_selective_scan_fwd with a caller-owned device
 * workspace (16-byte aligned, workspace_bytes long, not overlapping any tensor of the
 * call). The result is the same computation; with at least the size reported by
 * ssm_selective_scan_fwd_workspace_size the library may use the segmented schedule
 * described there. A smaller (or NULL, 0) workspace falls back to the unsegmented
 * kernels. The workspace contents are scratch: overwritten, not read before written.
 * Errors as ssm_selective_scan_fwd, plus SSM_ERR_NULL (bytes > 0 with NULL) and
 * SSM_ERR_LAYOUT (misaligned or overlapping workspace).
 */
SSM_API ssm_status_t ssm_selective_scan_fwd_ws(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                               const ssm_tensor_t* A, const ssm_tensor_t* B,
                                               const ssm_tensor_t* C, const ssm_tensor_t* D,
                                               const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                               int delta_softplus, ssm_tensor_t* y,
                                               ssm_tensor_t* last_state, void* workspace,
                                               size_t workspace_bytes, void* stream);

/* Flags of the extended entry points (ssm_selective_scan_fwd_ex, ssm_state_update_ex). */
#define SSM_FWD_ZOH 1u /* B-bar from the exact zero-order hold instead of Delta * B */

/*
 * ssm_selective_scan_fwd_ex -- ssm_selective_scan_fwd_ws with two options.
 *
 * Start state h0: the recurrence begins at h(0) = h0 instead of zeros, so a sequence
 * can be processed in pieces (chunked prefill, a cached prompt prefix continued with
 * new tokens): running the prefix, then the rest with h0 = the prefix's last_state,
 * gives the result of one call over the whole sequence. Sources: "Mamba and State
 * Space Models", "Common Pitfalls" (the state after a prefix is reusable) and
 * "Selective scan pseudo-code" (the loop carries h from step to step); "8.7 State Space
 * Models (Mamba)", section 2.1 fixes h(0) = 0 for a sequence start, the case h0 = NULL.
 *
 * flags & SSM_FWD_ZOH: B-bar is the exact zero-order hold of the continuous system,
 *   B-bar[n] = (exp(dt A[d,n]) - 1) / A[d,n] * B[b,t,n]   (dt * B[b,t,n] where A[d,n] = 0)
 * ("Arch 02: Mamba SSM", zero-order-hold discretisation; "8.7 State Space Models
 * (Mamba)", section 3) instead of the simplification dt * B that Mamba uses. This
 * option runs on the general kernel (fp32 arithmetic, expm1 for the B-bar factor),
 * not on the fast bf16 channel kernel.
 *
 *   h0     (batch, D, N)  f32, nullable   start state (NULL = zeros); read only
 *   flags  0 or SSM_FWD_ZOH               other bits: SSM_ERR_UNSUPPORTED
 * last_state may be the same buffer as h0 (same pointer and shape): the start state is
 * read before the final state is written. Any other overlap of h0 with an output is
 * SSM_ERR_LAYOUT. L == 0 copies h0 (or zeros) to last_state. Everything else as
 * ssm_selective_scan_fwd_ws.
 */
SSM_API ssm_status_t ssm_selective_scan_fwd_ex(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                               const ssm_tensor_t* A, const ssm_tensor_t* B,
                                               const ssm_tensor_t* C, const ssm_tensor_t* D,
                                               const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                               int delta_softplus, const ssm_tensor_t* h0, uint32_t flags,
                                               ssm_tensor_t* y, ssm_tensor_t* last_state,
                                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * ssm_selective_scan_fwd_noalloc -- the forward pass for callers that cannot allocate
 * device memory or pass the library a workspace. (Not a method of the pages: the
 * pages have no counterpart; this is an interface convenience.)
 *
 * Who needs it: code that may only touch buffers it was handed -- an inference engine
 * that reserves its whole memory budget when it starts and forbids allocations later,
 * a plugin or callback interface that receives only input and output pointers, or a
 * latency-bound path where an allocation that can stall or fail is not acceptable.
 *
 * Same arguments, result and errors as ssm_selective_scan_fwd. When the shape takes
 * the segmented schedule (see ssm_selective_scan_fwd_workspace_size), its scratch is a
 * fixed array of SSM_NOALLOC_SCRATCH_BYTES that the library keeps on every GPU that
 * loads it, until the process exits; a shape that would need more returns
 * SSM_ERR_UNSUPPORTED. The call itself allocates nothing.
 *  - The first call on a device looks up the array's device address (once per device,
 *    with that device current); make that first call before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU (other
 *    streams, other threads) race on it. Nothing in it needs to start at zero; each
 *    call writes every scratch value before reading it.
 */
#define SSM_NOALLOC_SCRATCH_BYTES (4u << 20)
SSM_API ssm_status_t ssm_selective_scan_fwd_noalloc(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                                    const ssm_tensor_t* A, const ssm_tensor_t* B,
                                                    const ssm_tensor_t* C, const ssm_tensor_t* D,
                                                    const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                                    int delta_softplus, ssm_tensor_t* y,
                                                    ssm_tensor_t* last_state, void* stream);

/*
 * ssm_state_update -- one recurrent decode step, state updated in place.
 *
 * For each batch row b and channel d:
 *   state[b,d,n] = exp(delta[b,d] * A[d,n]) * state[b,d,n] + delta[b,d] * B[b,n] * x[b,d]
 *   v            = sum_n C[b,n] * state[b,d,n] + D[d] * x[b,d]
 *   y[b,d]       = z ? v * silu(z[b,d]) : v
 * delta is the final step size: no bias and no softplus are applied.
 * Sources: "8.7 State Space Models (Mamba)", section 5 (O(1) work and a fixed d*n state
 * per generated token); "Mamba and State Space Models", "Selective scan pseudo-code"
 * (one step of the loop body) and "Common Pitfalls" (the state after a prefix is
 * reusable: last_state of ssm_selective_scan_fwd continues here).
 *
 *   state  (batch, D, N)  f32             read and overwritten in place
 *   x      (batch, D)     I/O type        token input
 *   delta  (batch, D)     I/O type        step size
 *   A      (D, N)         f32
 *   B, C   (batch, N)     I/O type
 *   D      (D)            f32, nullable
 *   z      (batch, D)     I/O type, nullable
 *   y      (batch, D)     I/O type or f32   output, written
 *   stream                cudaStream_t
 * batch == 0 is a valid no-op. Only state may alias itself; y must not overlap any input.
 * With bf16 inputs, N = 16, D a multiple of 128 and 16-byte aligned state, x, delta, z,
 * A, B and C (and delta_bias with ssm_state_update_ex, the conv operands with
 * ssm_conv_state_update; not ZOH) the step runs as a persistent kernel that streams tiles of 128 channels through shared
 * memory; otherwise one thread updates 8 states (4 for N = 4). The two give identical
 * results (SSM_B300_DECODE=plain selects the second always).
 */
SSM_API ssm_status_t ssm_state_update(ssm_tensor_t* state, const ssm_tensor_t* x,
                              const ssm_tensor_t* delta, const ssm_tensor_t* A,
                              const ssm_tensor_t* B, const ssm_tensor_t* C,
                              const ssm_tensor_t* D, const ssm_tensor_t* z,
                              ssm_tensor_t* y, void* stream);

/*
 * ssm_state_update_ex -- ssm_state_update with the forward pass's step-size map applied
 * inside the step: dt = delta[b,d] + delta_bias[d], then softplus(dt) when
 * delta_softplus is 1, and dt replaces delta in the update. This is the decode step of
 * a model whose forward pass uses the same bias and softplus ("Mamba and State Space
 * Models", "Discretization and initialization details": Delta = softplus(W x + b)), so
 * a decode step continues ssm_selective_scan_fwd exactly.
 *
 *   delta_bias  (D)  f32, nullable   added to delta (NULL = 0)
 *   delta_softplus   0 or 1          anything else is SSM_ERR_UNSUPPORTED
 *   flags            0 or SSM_FWD_ZOH (the zero-order-hold B-bar, as in
 *                    ssm_selective_scan_fwd_ex); other bits: SSM_ERR_UNSUPPORTED
 * Everything else as ssm_state_update.
 */
SSM_API ssm_status_t ssm_state_update_ex(ssm_tensor_t* state, const ssm_tensor_t* x,
                                         const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                         const ssm_tensor_t* B, const ssm_tensor_t* C,
                                         const ssm_tensor_t* D, const ssm_tensor_t* z,
                                         const ssm_tensor_t* delta_bias, int delta_softplus,
                                         uint32_t flags, ssm_tensor_t* y, void* stream);

/*
 * ssm_conv_selective_scan_fwd -- the block's conv prologue fused into the forward pass.
 * In the Mamba block the SSM input is the output of a causal depthwise convolution of
 * width 4 followed by SiLU ("Mamba and State Space Models", "The Mamba Block" and the
 * model card's d_conv = 4; "8.7 State Space Models (Mamba)", section 6). This entry
 * takes the convolution's INPUT x and computes, for every (b, t, d),
 *   u[b,t,d] = silu(conv_bias[d] + sum_{k=0..3} conv_weight[d,k] * x[b,t-3+k,d])
 * on the fly, so u is never written to or read from device memory; everything after
 * that is ssm_selective_scan_fwd_ex with this u.
 *
 *   x            (batch, L, D)  I/O type         the convolution's input
 *   conv_weight  (D, 4)         f32              tap k multiplies x[t-3+k]
 *   conv_bias    (D)            f32, nullable
 *   conv_state   (batch, D, 3)  I/O type, nullable
 *                read: the three inputs before x[:,0] (oldest first; NULL = zeros);
 *                then overwritten with the three inputs before step L, i.e. the state
 *                that continues the sequence here or in ssm_conv_state_update
 *   delta ... stream            as ssm_selective_scan_fwd_ex (h0, flags, workspace)
 * conv_state may overlap no other tensor. With bf16 I/O and the channel kernel the
 * SiLU of the prologue uses the SFU tanh (relative error ~5e-4 on u).
 */
SSM_API ssm_status_t ssm_conv_selective_scan_fwd(const ssm_tensor_t* x, const ssm_tensor_t* conv_weight,
                                                 const ssm_tensor_t* conv_bias, ssm_tensor_t* conv_state,
                                                 const ssm_tensor_t* delta, const ssm_tensor_t* A,
                                                 const ssm_tensor_t* B, const ssm_tensor_t* C,
                                                 const ssm_tensor_t* D, const ssm_tensor_t* z,
                                                 const ssm_tensor_t* delta_bias, int delta_softplus,
                                                 const ssm_tensor_t* h0, uint32_t flags, ssm_tensor_t* y,
                                                 ssm_tensor_t* last_state, void* workspace,
                                                 size_t workspace_bytes, void* stream);

/*
 * ssm_conv_state_update -- one decode step of the block's conv prologue and the SSM:
 *   u = silu(conv_bias[d] + w0 cs[0] + w1 cs[1] + w2 cs[2] + w3 x[b,d])   (w = conv_weight[d])
 *   conv_state[b,d] <- (cs[1], cs[2], x[b,d])                           in place
 *   then ssm_state_update_ex with u as the token input.
 *
 *   conv_state  (batch, D, 3)  I/O type   required; read, then shifted in place
 *   x           (batch, D)     I/O type   the convolution's input for this token
 *   conv_weight (D, 4) f32, conv_bias (D) f32 nullable
 * Everything else as ssm_state_update_ex. conv_state may overlap no other tensor.
 */
SSM_API ssm_status_t ssm_conv_state_update(ssm_tensor_t* conv_state, ssm_tensor_t* state,
                                           const ssm_tensor_t* x, const ssm_tensor_t* conv_weight,
                                           const ssm_tensor_t* conv_bias, const ssm_tensor_t* delta,
                                           const ssm_tensor_t* A, const ssm_tensor_t* B,
                                           const ssm_tensor_t* C, const ssm_tensor_t* D,
                                           const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                           int delta_softplus, uint32_t flags, ssm_tensor_t* y,
                                           void* stream);

/*
 * ssm_selective_scan_bwd -- backward pass of the forward pass (Delta * B discretisation,
 * with or without a start state; not the conv prologue or the ZOH option): the
 * gradients of the loss sum(dy * y) + sum(dlast * last_state) with respect to every
 * input. Per channel, in reverse time with g = dL/dh_t (from dlast at t = L-1):
 *   dv = dy silu(z)      dz = dy v silu'(z)     dD += dv u      g += dv C_t     dC_t += dv h_t
 *   dB_t += g dt u       du = dv D + sum_n g dt B_t             dA += g a h_{t-1} dt
 *   ddelta = sum_n g (B_t u + A a h_{t-1}) * (softplus ? sigmoid(delta + bias) : 1)
 *   dbias += ddelta      g *= a                 (after t = 0: dh0 = g)
 * Sources: the recurrence of "Mamba and State Space Models", "Selective scan
 * pseudo-code", differentiated; the states are recomputed from checkpoints rather than
 * stored ("Mamba and State Space Models", "Hardware-Aware Parallel Scan": kernel fusion
 * with recomputation in the backward pass).
 *
 *   u ... delta_softplus, h0    the forward pass's inputs (as ssm_selective_scan_fwd_ex)
 *   dy      (batch, L, D)  gradient type G     dL/dy
 *   dlast   (batch, D, N)  f32, nullable       dL/dlast_state (NULL = 0)
 *   du, ddelta (batch, L, D), dB, dC (batch, L, N): type G, written
 *   dA      (D, N) f32, written                dD, dbias (D) f32: required exactly when
 *   dz      (batch, L, D) type G: required exactly when z is given     D / delta_bias are
 *   dh0     (batch, D, N) f32, nullable: dL/dh0 (also without h0)      given
 *   workspace: at least ssm_selective_scan_bwd_workspace_size bytes, 256-byte aligned,
 *              overlapping no tensor; scratch
 * G is the I/O type or SSM_F32, the same for dy and every gradient of an I/O tensor.
 * Gradients are accumulated in fp32 and summed in a fixed order: the result is
 * deterministic. Outputs may overlap no input and no other output. A missing gradient
 * output for a given optional input (or one for an absent input) is SSM_ERR_NULL; a
 * short workspace is SSM_ERR_SHAPE. L == 0 or batch == 0 writes zeros (dh0 = dlast).
 */
SSM_API ssm_status_t ssm_selective_scan_bwd(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                            const ssm_tensor_t* A, const ssm_tensor_t* B,
                                            const ssm_tensor_t* C, const ssm_tensor_t* D,
                                            const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                            int delta_softplus, const ssm_tensor_t* h0,
                                            const ssm_tensor_t* dy, const ssm_tensor_t* dlast,
                                            ssm_tensor_t* du, ssm_tensor_t* ddelta, ssm_tensor_t* dA,
                                            ssm_tensor_t* dB, ssm_tensor_t* dC, ssm_tensor_t* dD,
                                            ssm_tensor_t* dz, ssm_tensor_t* dbias, ssm_tensor_t* dh0,
                                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * ssm_selective_scan_fwd_train -- the forward pass of a training step: y and last_state
 * exactly as ssm_selective_scan_fwd_ex (flags 0) with h0, plus, into the checkpoint region
 * of a backward workspace, the state before every 16-step chunk that the backward pass
 * recomputes its states from ("Mamba and State Space Models", "Hardware-Aware Parallel
 * Scan": the states are not stored, they are recomputed in the backward pass; storing one
 * state per chunk bounds that recomputation to one chunk).
 *
 *   u ... h0, y, last_state   as ssm_selective_scan_fwd_ex
 *   bwd_workspace             at least ssm_selective_scan_bwd_workspace_size bytes for this
 *                             shape, 256-byte aligned, overlapping no tensor; pass the same
 *                             buffer to ssm_selective_scan_bwd_ex for this step
 *   checkpoints_written       out: 1 when the checkpoints were written (bf16 inputs, N = 8
 *                             or 16, the channel kernel's alignment: 16-byte aligned rows,
 *                             D % 8 == 0), else 0 (y is computed all the same; the backward
 *                             pass then makes its own checkpoints: call it without
 *                             SSM_BWD_CHECKPOINTS)
 * Errors as ssm_selective_scan_fwd_ex; SSM_ERR_NULL (checkpoints_written or, for a
 * non-empty problem, bwd_workspace NULL), SSM_ERR_LAYOUT (misaligned or overlapping
 * workspace), SSM_ERR_SHAPE (workspace too short).
 */
SSM_API ssm_status_t ssm_selective_scan_fwd_train(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                                  const ssm_tensor_t* A, const ssm_tensor_t* B,
                                                  const ssm_tensor_t* C, const ssm_tensor_t* D,
                                                  const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                                  int delta_softplus, const ssm_tensor_t* h0,
                                                  ssm_tensor_t* y, ssm_tensor_t* last_state,
                                                  void* bwd_workspace, size_t bwd_workspace_bytes,
                                                  int32_t* checkpoints_written, void* stream);

#define SSM_BWD_CHECKPOINTS 1u /* the workspace holds ssm_selective_scan_fwd_train's checkpoints */

/*
 * ssm_selective_scan_bwd_ex -- ssm_selective_scan_bwd with flags. flags & SSM_BWD_CHECKPOINTS:
 * the workspace's checkpoint region already holds the checkpoints of this step's forward
 * pass (ssm_selective_scan_fwd_train reported checkpoints_written = 1 for the same inputs,
 * h0 and workspace, and nothing wrote the workspace since), so the checkpoint pass is
 * skipped. Other flag bits:
 * SSM_ERR_UNSUPPORTED. ssm_selective_scan_bwd(...) is ssm_selective_scan_bwd_ex(..., 0, ...).
 * The gradients equal those of ssm_selective_scan_bwd bit for bit when the forward pass ran
 * as one segment, and to rounding when it ran the segmented schedule (long sequences over
 * few channels), whose carried states reassociate the recurrence.
 */
SSM_API ssm_status_t ssm_selective_scan_bwd_ex(const ssm_tensor_t* u, const ssm_tensor_t* delta,
                                               const ssm_tensor_t* A, const ssm_tensor_t* B,
                                               const ssm_tensor_t* C, const ssm_tensor_t* D,
                                               const ssm_tensor_t* z, const ssm_tensor_t* delta_bias,
                                               int delta_softplus, const ssm_tensor_t* h0,
                                               const ssm_tensor_t* dy, const ssm_tensor_t* dlast,
                                               ssm_tensor_t* du, ssm_tensor_t* ddelta, ssm_tensor_t* dA,
                                               ssm_tensor_t* dB, ssm_tensor_t* dC, ssm_tensor_t* dD,
                                               ssm_tensor_t* dz, ssm_tensor_t* dbias, ssm_tensor_t* dh0,
                                               uint32_t flags, void* workspace, size_t workspace_bytes,
                                               void* stream);

/* Bytes of workspace ssm_selective_scan_bwd needs for this shape (0 for an empty problem):
 * the state before every 16-step chunk, per-warp partial sums of dB and dC, and per-row
 * partials of dA, dD, dbias. SSM_ERR_NULL (bytes == NULL) or SSM_ERR_SHAPE (negative). */
SSM_API ssm_status_t ssm_selective_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N,
                                                          size_t* bytes);

/*
 * ssm_ssd_fwd -- Mamba-2 SSD forward pass: the selective SSM with a scalar decay per head
 * and a P x N matrix state per head ("Mamba and State Space Models", "Mamba-2 and State
 * Space Duality"; "8.7 State Space Models (Mamba)", Mamba-2). For batch row b, head h,
 * group g = h / (H / groups):
 *   dt  = delta[b,t,h] + dt_bias[h], then softplus(dt) when dt_softplus
 *   S   = exp(dt A[h]) S + dt x[b,t,h,:] B[b,t,g,:]^T        (S: P x N, from h0 or 0)
 *   y[b,t,h,:] = S C[b,t,g,:] + D[h] x[b,t,h,:]
 * computed in chunks of 64 steps: inside a chunk as the masked quadratic form
 * tril(C B^T o decay) (dt X) plus the carried state read out, across chunks by carrying
 * S (fp32); the contractions per chunk run on the tensor cores (bf16 operands, products
 * of inputs as bf16 high + low pairs, fp32 accumulation).
 *
 * Descriptors are 3-D views (the last two dimensions of each tensor flattened):
 *   groups       number of B/C groups G (divides H)
 *   x            (batch, L, H*P)   bf16    head h, channel p at h*P + p
 *   delta        (batch, L, H)     bf16    raw step size
 *   A            (H)               f32     decay rate per head (negative)
 *   B, C         (batch, L, G*N)   bf16
 *   D, dt_bias   (H)               f32, nullable
 *   dt_softplus  0 or 1
 *   h0           (batch, H, P*N)   f32, nullable   start state (row p, column n at p*N + n)
 *   y            (batch, L, H*P)   bf16 or f32, written
 *   last_state   (batch, H, P*N)   f32, nullable, written
 *   workspace    at least ssm_ssd_fwd_workspace_size bytes, 256-byte aligned, overlapping
 *                no tensor, H <= 65535: the chunk-parallel schedule (step sizes and the
 *                chunks' C B^T first; then the state walked over the chunks by blocks of
 *                32 state rows, writing every chunk's entering state; then every chunk's
 *                outputs at once); NULL / too small: one CTA per (batch, head) walks the
 *                chunks in order with the state on chip. Same arithmetic either way.
 * P = H*P / H and N = G*N / G must each be 64 or 128 (SSM_ERR_UNSUPPORTED otherwise); x,
 * B, C 16-byte aligned; batch <= 65535.
 */
SSM_API ssm_status_t ssm_ssd_fwd(int64_t groups, const ssm_tensor_t* x, const ssm_tensor_t* delta,
                                 const ssm_tensor_t* A, const ssm_tensor_t* B, const ssm_tensor_t* C,
                                 const ssm_tensor_t* D, const ssm_tensor_t* dt_bias, int dt_softplus,
                                 const ssm_tensor_t* h0, ssm_tensor_t* y, ssm_tensor_t* last_state,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace for the chunk-parallel ssm_ssd_fwd schedule (0 for an empty problem):
 * batch x ceil(L/64) x H x (P x N x 2 + 512) bytes (per chunk and head: the entering state
 * in bf16, the step sizes and decay exponents in fp32) plus batch x ceil(L/64) x groups x
 * 18 KiB (C B^T of each chunk and group, rows padded to 72 floats), each part rounded up to
 * 256 bytes.
 * SSM_ERR_NULL / SSM_ERR_SHAPE (negative sizes, groups < 1). */
SSM_API ssm_status_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t H, int64_t groups, int64_t P,
                                                int64_t N, size_t* bytes);

/* Human-readable name of a status code (static string, never NULL). */
SSM_API const char* ssm_status_string(ssm_status_t status);

/*
 * ssm_device_error -- diagnostic read of the library's device-side error word on the
 * current device. It SYNCHRONISES the given stream, returns the word in *code and clears
 * it. Returns SSM_OK, SSM_ERR_NULL (code == NULL) or SSM_ERR_CUDA. Kernels never trap: a
 * wait that runs out records the first failure here and the kernel returns, leaving the
 * context usable. Codes: 0 no error; 1 a TMA load never completed; 2 the consumers never
 * released a staging buffer; 3 a converted B/C tile was never published; 4 a tensor-core
 * MMA never signalled completion.
 * The bounded waits of the forward pass's channel kernel, the streamed decode kernel and the
 * tensor-core SSD kernels last about one second by default; the environment variable SSM_B300_WAIT_LIMIT_CYCLES
 * sets another limit (in SM clock cycles), and SSM_B300_FAULT_INJECT=skip_loads makes their
 * staging thread issue no copies, so that every wait for data runs out (used by the
 * failure-detection tests only).
 *
 * Kernel selection switches (each path computes the same results; tests compare them):
 * SSM_B300_FORWARD_KERNEL=generic|chan|auto (the forward pass's kernel), SSM_B300_SEGMENTS=0
 * (no segmented schedule), SSM_B300_DECODE=plain (the per-thread decode kernel).
 */
SSM_API ssm_status_t ssm_device_error(void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* SSM_B300_H */
