/*
 * linattn.h -- C ABI of the GB300 (sm_103a) kernelized linear-attention
 * library.
 *
 * The library computes linear attention with the Linear Transformer feature
 * map phi(x) = elu(x) + 1 (x + 1 for x > 0, exp(x) otherwise):
 *
 *   o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps)
 *
 * in the three forms described on "Linear Attention Mechanisms"
 * (dileepadev.github.io) and "Attention-Free / Sub-Quadratic Architectures"
 * (blog.vguerra.net):
 *   - causal:     S_i = gamma S_{i-1} + phi(k_i) v_i^T, z_i = gamma z_{i-1} +
 *                 phi(k_i) ("Recurrent Reformulation"; "The recurrent form
 *                 (causal)"; fixed decay gamma from "Gating and Selective
 *                 State Updates" / "Evolution: add decay/gating", applied to
 *                 both S and z);
 *   - non-causal: S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j) over every
 *                 key, shared by every query ("The Kernel Trick for
 *                 Attention"; "Linear Attention (the core trick)");
 *   - decode:     one step of the causal recurrence on a caller-held state;
 *   - gated:      the causal recurrence with a data-dependent gate per key
 *                 feature and token ("Gating and Selective State Updates",
 *                 gated linear attention), forward and decode step;
 *   - Performer:  random exponential features in place of elu + 1
 *                 ("Choosing the Feature Map"), the map alone and the
 *                 attention over it.
 * eps is added to the denominator after the dot product, as in the NumPy
 * listing on "Linear Attention Mechanisms" (sadullah.online), "The linear
 * attention trick".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, row-major, contiguous, in DEVICE memory:
 *     q, k  [B][H][N][D]      v, o  [B][H][N][Dv]     (forward / prefill)
 *     q, k  [B][H][D]         v, o  [B][H][Dv]        (decode step)
 *     S     [B][H][D][Dv] fp32                        (state, caller-owned)
 *     z     [B][H][D]     fp32
 *   q, k, v and o all have the element type `dtype` (LA_F32 or LA_BF16).
 *   Every device pointer must be 16-byte aligned.
 * - gamma is a HOST array of H floats in [0, 1] (one decay per head), or
 *   NULL meaning 1 for every head.  The library copies the values during the
 *   call; the caller keeps ownership.
 * - stream is a cudaStream_t passed as void* (NULL = legacy default stream),
 *   so that this header needs no CUDA header to compile.
 *   Every call is asynchronous on that stream and never synchronises.  The
 *   caller owns all buffers; the library keeps no state between calls
 *   (except la_forward_host's copy streams and memory pool, and the
 *   allocation-free entry point's fixed array, all per device).
 * - Arguments are validated before any CUDA call, so a rejected call has no
 *   side effect.  A launch failure returns LA_ERR_CUDA; an error raised while
 *   a kernel runs surfaces at the caller's next synchronisation.
 * - Supported sizes: D and Dv in {64, 128}; H <= 256; B*H*N < 2^31 tokens per
 *   call.  B, H or N equal to 0 is an empty call that returns LA_OK (for
 *   la_prefill_state with N = 0 the state is set to zero).
 * - Arithmetic: fp32 state and accumulation.  For LA_BF16 the tensor-core
 *   kernels round phi(q), phi(k), the decay-weighted values and the
 *   intra-chunk weights to bf16 as matrix-multiply operands; o is rounded to
 *   bf16 (round to nearest even).
 *
 * Example: a causal pass with one decay per head, then decode steps that
 * continue from its state (all buffers device memory of the documented
 * sizes; error handling shortened):
 *
 *   float gamma[H];                        // host, one decay per head
 *   la_status_t st = la_forward_state(q, k, v, o, S, z, B, H, N, D, Dv,
 *                                     gamma, 1e-6f, LA_BF16, stream);
 *   if (st != LA_OK) fprintf(stderr, "%s\n", la_status_string(st));
 *   for (int t = 0; t < steps; ++t)        // S, z updated in place
 *     st = la_decode_step(q_t, k_t, v_t, S, z, o_t, B, H, D, Dv, gamma,
 *                         1e-6f, LA_BF16, stream);
 *   cudaStreamSynchronize(stream);         // kernel faults surface here
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad eps or
                             gamma, aliasing output, gamma != 1 when
                             non-causal */
  LA_ERR_UNSUPPORTED = 2, /* valid but not implemented: D or Dv not in
                             {64, 128}, H > 256, too many tokens */
  LA_ERR_CUDA = 3         /* a CUDA call or kernel launch failed */
} la_status_t;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype_t;

/*
 * Forward pass over whole sequences.
 *   causal != 0: o_i uses keys/values j <= i (inclusive), decayed by
 *                gamma[h]^(i-j).
 *   causal == 0: o_i uses every key/value of its (b, h); gamma must be NULL
 *                or all 1 (otherwise LA_ERR_INVALID_ARG).  The non-causal
 *                path needs a stream-ordered workspace of about
 *                B*H*(D*Dv + D)*4*(1 + ceil(N/4096)) bytes, taken with
 *                cudaMallocAsync on `stream` and released on it.
 * q, k: [B][H][N][D]; v: [B][H][N][Dv]; o: [B][H][N][Dv] (written).  o must
 * not overlap q, k or v.  eps must be finite and >= 0.
 * Defined on the pages "Linear Attention Mechanisms" (dileepadev.github.io):
 * causal by "Recurrent Reformulation" (S_i, z_i and the read-out o_i), with
 * the per-head decay of "Gating and Selective State Updates" (RetNet, weight
 * gamma^(t-j)) on both S and z; non-causal by "The Kernel Trick for
 * Attention" (S and z once over every key); eps as in the NumPy listing of
 * "Linear Attention Mechanisms" (sadullah.online), "The linear attention
 * trick".
 */
LA_API la_status_t la_forward(const void *q, const void *k, const void *v, void *o,
                       int B, int H, int N, int D, int Dv, int causal,
                       const float *gamma, float eps, la_dtype_t dtype,
                       void *stream);

/*
 * la_forward on HOST buffers: q, k, v are read from host memory and o is
 * written to host memory (same shapes, dtype and arguments as la_forward;
 * no alignment requirement).  The heads are processed in groups (a run of
 * heads of one batch entry each, about eight groups): a group's inputs are
 * copied up on a copy stream the library owns, its forward runs on `stream`
 * once they have landed, and its output is copied down on a second copy
 * stream once the forward is done, so that uploads, kernels and downloads of
 * different groups overlap.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister): pageable memory is correct but its
 * copies do not overlap.  Device memory for the whole problem is a
 * stream-ordered allocation on `stream` from a pool the library keeps per
 * device, which holds released memory for the next call until the process
 * exits (the two copy streams are kept likewise).  Asynchronous: o is complete once
 * `stream` has been synchronised; the host buffers must stay valid until
 * then.  The result equals la_forward's up to the order of summation (each
 * group splits its sequences for its own size).  Errors as la_forward.
 * Defined on the same pages as la_forward.
 */
LA_API la_status_t la_forward_host(const void *q, const void *k, const void *v, void *o,
                                   int B, int H, int N, int D, int Dv, int causal,
                                   const float *gamma, float eps, la_dtype_t dtype,
                                   void *stream);

/*
 * State after a causal pass over N tokens (the prefill of the decode loop):
 *   S = sum_j gamma^(N-1-j) phi(k_j) v_j^T,  z = sum_j gamma^(N-1-j) phi(k_j)
 * k: [B][H][N][D]; v: [B][H][N][Dv] (dtype); S: [B][H][D][Dv] fp32 and
 * z: [B][H][D] fp32 are overwritten.  S and z must not overlap k or v, nor
 * each other.
 * Defined on the pages "Linear Attention Mechanisms" (dileepadev.github.io),
 * "Recurrent Reformulation" (S_i and z_i of the causal recurrence at
 * i = N - 1, the state the recurrent form carries into inference) and
 * "Gating and Selective State Updates" (the decay weight gamma^(N-1-j)).
 */
LA_API la_status_t la_prefill_state(const void *k, const void *v, float *S, float *z,
                             int B, int H, int N, int D, int Dv,
                             const float *gamma, la_dtype_t dtype,
                             void *stream);

/*
 * Causal forward that also returns the state after the last token: o as
 * la_forward(..., causal = 1, ...), and S, z as la_prefill_state over the
 * same k, v (the state the decode loop continues from).  On the tensor-core
 * path for D = Dv = 128 the state comes out of the forward's own pass (the
 * CTA of the last part writes it); otherwise the library runs the forward,
 * then the prefill reduction, on `stream`.
 * q, k: [B][H][N][D]; v, o: [B][H][N][Dv] (dtype); S: [B][H][D][Dv] fp32 and
 * z: [B][H][D] fp32 are overwritten (zero for N = 0).  No written buffer (o,
 * S, z) may overlap any other buffer; the read-only inputs may share memory.
 * Errors as la_forward and la_prefill_state.
 * Defined on the pages "Linear Attention Mechanisms" (dileepadev.github.io),
 * "Recurrent Reformulation" (the state S_i, z_i at i = N - 1) and "Gating
 * and Selective State Updates" (the decay on both).
 */
LA_API la_status_t la_forward_state(const void *q, const void *k, const void *v, void *o,
                                    float *S, float *z, int B, int H, int N, int D, int Dv,
                                    const float *gamma, float eps, la_dtype_t dtype,
                                    void *stream);

/*
 * One recurrent decode step, in place: first
 *   S <- gamma S + phi(k) v^T,  z <- gamma z + phi(k),
 * then  o = phi(q)^T S / (phi(q) . z + eps)  with the updated state.
 * q, k: [B][H][D]; v, o: [B][H][Dv] (dtype); S: [B][H][D][Dv] fp32 and
 * z: [B][H][D] fp32 are read and rewritten.  No written buffer (S, z, o) may
 * overlap any other buffer; q, k and v may share memory.
 * Defined on the pages "Linear Attention Mechanisms" (dileepadev.github.io),
 * "Recurrent Reformulation" (one iteration of the recurrence: update with
 * k, v, then read out with q) and "Practical Tradeoffs" (a fixed-size state
 * per step at inference), with the decay of "Gating and Selective State
 * Updates" on both S and z.
 */
LA_API la_status_t la_decode_step(const void *q, const void *k, const void *v,
                           float *S, float *z, void *o, int B, int H, int D,
                           int Dv, const float *gamma, float eps,
                           la_dtype_t dtype, void *stream);

/*
 * Gated causal forward (gated linear attention): per token t
 *   S_t = diag(a_t) S_{t-1} + phi(k_t) v_t^T,  z_t = a_t (.) z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / (phi(q_t) . z_t + eps),   S_{-1} = 0, z_{-1} = 0,
 * i.e. the data-dependent gate G_t of "Linear Attention Mechanisms"
 * (dileepadev.github.io), "Gating and Selective State Updates", taken as one
 * value per key feature and token, G_t = a_t 1^T (row d of S is scaled by
 * a_t[d]), and applied to the normaliser z as well.  a_t = 1 everywhere is
 * la_forward(causal = 1, gamma = NULL); a_t = gamma[h] everywhere is the
 * fixed decay; a_t[d] = 0 clears row d of the state before token t's update.
 * q, k: [B][H][N][D]; v, o: [B][H][N][Dv] (dtype); a: [B][H][N][D] fp32 in
 * DEVICE memory, every value in [0, 1] (the library cannot check device
 * values: outside [0, 1] the result is unspecified, a NaN gate gives NaN
 * outputs).  S: [B][H][D][Dv] fp32 and z: [B][H][D] fp32 are both NULL or
 * both set; when set they receive the state after the last token (zero for
 * N = 0).  fp32 arithmetic on CUDA cores, or for bf16 with D = Dv = 128
 * and B*H >= 8 the tensor-core form described at la_gated_kernel
 * (bf16 operands, fp32 accumulation and state).  A workspace of about
 * B*H*(P-1)*(D*Dv + 2D)*4 bytes (P <= ceil(N/64) parts), plus for the
 * tensor-core form 2*B*H*N*D*2 + B*H*ceil(N/128)*D*4 bytes, is taken with
 * cudaMallocAsync on `stream` and released on it.  No written
 * buffer may overlap another buffer.  Errors as la_forward.
 */
LA_API la_status_t la_forward_gated(const void *q, const void *k, const void *v,
                                    const float *a, void *o, float *S, float *z, int B,
                                    int H, int N, int D, int Dv, float eps,
                                    la_dtype_t dtype, void *stream);

/*
 * Which form la_forward_gated runs for these arguments: 1 = tensor cores
 * (bf16, D = Dv = 128, B*H >= 8, with or without the final state, which
 * want_state no longer changes: q and k scaled per
 * 128-token chunk by gate suffix products, then the 128-token causal kernel
 * with its state rescaled by each chunk's gate products; a call whose gates
 * forget harder than 2^-93 within some chunk and feature falls back at run
 * time to the CUDA-core form, which a device flag selects), 0 = the fp32
 * CUDA-core form, or a negative la_status_t (negated) for invalid sizes.
 * Host-only.
 */
LA_API int la_gated_kernel(int B, int H, int N, int D, int Dv, la_dtype_t dtype, int want_state);

/*
 * One gated decode step, in place: first
 *   S <- diag(a) S + phi(k) v^T,  z <- a (.) z + phi(k),
 * then  o = phi(q)^T S / (phi(q) . z + eps)  with the updated state (the
 * recurrence of la_forward_gated for one token).  q, k: [B][H][D]; v, o:
 * [B][H][Dv] (dtype); a: [B][H][D] fp32 gates in [0, 1] (device); S:
 * [B][H][D][Dv] fp32 and z: [B][H][D] fp32 are read and rewritten.  No
 * written buffer (S, z, o) may overlap any other buffer.  Errors as
 * la_decode_step.
 */
LA_API la_status_t la_decode_gated(const void *q, const void *k, const void *v,
                                   const float *a, float *S, float *z, void *o, int B,
                                   int H, int D, int Dv, float eps, la_dtype_t dtype,
                                   void *stream);

/*
 * Performer random-feature map: for every row x of x [rows][D],
 *   phi(x) = r^(-1/2) [exp(w_1 . x - |x|^2/2), ..., exp(w_r . x - |x|^2/2)]
 * with the directions w_j the rows of W [r][D] (drawn by the caller: iid
 * N(0, 1), or block-orthogonal rows for positive orthogonal random features).
 * "Linear Attention Mechanisms" (dileepadev.github.io), "Choosing the Feature
 * Map": Random Fourier Features (Performer) and FAVOR+.  The -|x|^2/2 term is
 * the reading under which that passage's E[phi(q) . phi(k)] = exp(q . k)
 * holds for w ~ N(0, I).
 * x, W and phi [rows][r] (written) are DEVICE arrays of `dtype`; D and r in
 * {64, 128}.  LA_BF16 runs a tcgen05 GEMM with the exponential in its
 * epilogue (exact bf16 products, fp32 sums, phi rounded to bf16); LA_F32 runs
 * in fp32 on CUDA cores.  exp overflows fp32 where w_j . x - |x|^2/2 > 88.
 * phi may not overlap x or W.
 */
LA_API la_status_t la_favor_features(const void *x, const void *W, void *phi, int rows, int D,
                                     int r, la_dtype_t dtype, void *stream);

/*
 * Performer attention: la_favor_features on q and on k, then linear
 * attention over those r-dimensional features, o_i = phi(q_i)^T S_i /
 * (phi(q_i)^T z_i + eps), causal (S_i, z_i over j <= i, decayed by
 * gamma[h]^(i-j)) or non-causal (every j; gamma must be NULL or all 1).  The
 * attention runs on the same kernels as la_forward with the features in place
 * of phi(q), phi(k) (tensor cores for LA_BF16).  q, k: [B][H][N][D]; v, o:
 * [B][H][N][Dv]; W: [r][D]; all of `dtype`; D, Dv and r in {64, 128}.  The
 * features take a stream-ordered workspace of 2*B*H*N*r elements of `dtype`
 * (cudaMallocAsync on `stream`), plus the attention kernel's own.  o may not
 * overlap q, k, v or W.  Errors as la_forward.
 */
LA_API la_status_t la_forward_favor(const void *q, const void *k, const void *v, const void *W,
                                    void *o, int B, int H, int N, int D, int Dv, int r,
                                    int causal, const float *gamma, float eps,
                                    la_dtype_t dtype, void *stream);

/*
 * Backward pass of the causal form (with the per-head decay): given the
 * upstream gradient dO = dL/do of o = la_forward(q, k, v, causal = 1, gamma,
 * eps), writes dq = dL/dq, dk = dL/dk, dv = dL/dv.  With
 * w_ij = gamma^(i-j) phi(q_i).phi(k_j) (j <= i), d_i = sum_j w_ij + eps,
 * gt_i = dO_i / d_i and c_i = gt_i . o_i, the chain rule through
 * o_i = sum_j w_ij v_j / d_i gives dL/dw_ij = gt_i . v_j - c_i, and
 *   dv_j = sum_(i>=j) w_ij gt_i,
 *   dq_i = phi'(q_i) * sum_(j<=i) gamma^(i-j) (dL/dw_ij) phi(k_j),
 *   dk_j = phi'(k_j) * sum_(i>=j) gamma^(i-j) (dL/dw_ij) phi(q_i),
 * phi'(x) = 1 for x > 0, exp(x) otherwise.  The "parallel training" half
 * of the duality on "Linear Attention Mechanisms" (dileepadev.github.io),
 * "Recurrent Reformulation"; the forward it differentiates is la_forward's.
 * The library recomputes o and d itself (the caller keeps no forward
 * state).  q, k, dq, dk: [B][H][N][D]; v, dO, dv: [B][H][N][Dv]; all of
 * `dtype`.  For LA_BF16 with Dv = 64 and every gamma >= 0.35 the sums run on
 * tcgen05 tensor cores (la_backward_kernel = 1): the forward's undivided
 * numerators and normalisers, then three decayed causal products with bf16
 * operands and fp32 accumulation (dq forward, dk and dv over token-reversed
 * operands), in a stream-ordered workspace of about B*H*N*(8 D + 1412)
 * bytes.  Otherwise fp32 arithmetic on CUDA cores in a stream-ordered
 * workspace of B*H*N*(4D + 6Dv + 16)*4 bytes plus the per-part states of the
 * sequence split.  Workspaces are taken with cudaMallocAsync on `stream`.
 * No gradient may overlap an input or another gradient.  Errors as
 * la_forward.
 */
LA_API la_status_t la_backward(const void *q, const void *k, const void *v, const void *dO,
                               void *dq, void *dk, void *dv, int B, int H, int N, int D,
                               int Dv, const float *gamma, float eps, la_dtype_t dtype,
                               void *stream);

/*
 * Which kernels la_backward runs for these arguments: 1 = tcgen05 tensor
 * cores (bf16, Dv = 64, D in {64, 128}, every gamma >= 0.35), 0 = fp32 CUDA
 * cores, or a negative la_status_t (negated) for invalid arguments.  gamma
 * as in la_backward (host array or NULL).  Host-only apart from reading the
 * current device's SM count.
 */
LA_API int la_backward_kernel(int B, int H, int N, int D, int Dv, const float *gamma,
                              la_dtype_t dtype);

/*
 * Number of kernels one la_backward call with these arguments launches (on
 * CUDA cores it depends on how the sequence is split across the current
 * device's SMs), 0 for an empty call, or a negative la_status_t (negated)
 * for invalid arguments.  Host-only apart from reading the current device's
 * SM count.
 */
LA_API int la_backward_launches(int B, int H, int N, int D, int Dv, const float *gamma,
                                la_dtype_t dtype);

/*
 * Which kernel la_forward would run for a causal call with these arguments:
 * 2 = the tcgen05 tensor-core kernel with 128-token chunks (bf16,
 * D = Dv = 128, every gamma >= 0.61), 1 = the tcgen05 tensor-core kernel with
 * 64-token chunks (bf16, D and Dv in {64, 128}, every gamma >= 0.35),
 * 0 = the fp32 CUDA-core kernel (fp32 inputs, or stronger decays, whose
 * gamma^-63 operand scale would leave the bf16 range), or a negative
 * la_status_t (negated) if the arguments are invalid.
 * Host-only; touches no device.
 */
LA_API int la_causal_kernel(int B, int H, int N, int D, int Dv,
                            const float *gamma, la_dtype_t dtype);

/*
 * Number of bounded device-side waits that gave up on the current device since
 * the library was loaded (or since the last reset).  The tensor-core kernels
 * bound every wait on another warp's progress; a nonzero count means some
 * kernel abandoned its work and the outputs of that call are invalid.  Reads
 * device memory with a blocking copy, so call it after synchronising the
 * streams that ran the kernels.  reset != 0 sets the counter back to zero.
 * Returns -1 if the counter cannot be read.
 */
LA_API int la_device_wait_timeouts(int reset);

/*
 * Diagnostic of the failure path above, without a fault: runs the kernels'
 * own bounded mbarrier wait, with a limit of `cycles` SM clock cycles (1 to
 * 4e9; about 0.5 ms per 1e6 cycles at 2 GHz), on a barrier that nothing
 * arrives on.  The wait gives up, adds one to the counter that
 * la_device_wait_timeouts reads, and *gave_up (host) becomes 1; the context
 * stays usable.  Launches one warp on the legacy default stream of the
 * current device and synchronises the device.  LA_ERR_INVALID_ARG for a
 * null gave_up or cycles out of range.
 */
LA_API la_status_t la_wait_selftest(long long cycles, int *gave_up);

/*
 * Non-causal forward without any device allocation.  No counterpart on the
 * pages: it computes exactly what la_forward(..., causal = 0, gamma = NULL,
 * ...) computes, but keeps its scratch (per-head S, z and the partial sums of
 * the split reduction) in a fixed array inside the library instead of taking
 * a workspace with cudaMallocAsync.  For callers that cannot let a library
 * allocate: applications that reserve device memory up front in their own
 * allocator and forbid third-party allocations, and latency-critical loops
 * where an allocation could stall or fail on a full memory pool.
 *   - The scratch is la_forward_noncausal_static_limit() bytes (32 MiB) on
 *     every GPU that loads the library, held until the process exits.  Calls
 *     whose per-head state alone, B*H*(D*Dv + D)*4 bytes, exceeds it return
 *     LA_ERR_UNSUPPORTED; below that the reduction uses as many sequence
 *     splits as fit.
 *   - The first call on each device queries the device address of the
 *     scratch (one runtime call, with that device current); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the one scratch array.  Calls whose work
 *     overlaps on the GPU (for example on two streams with no ordering
 *     between them) race on it and corrupt each other's results: order them.
 *     Each call writes every scratch word before reading it, so nothing needs
 *     clearing between calls.
 * Arguments, layouts and errors otherwise as la_forward (gamma is implicitly
 * 1; D, Dv in {64, 128}).
 */
LA_API la_status_t la_forward_noncausal_static(const void *q, const void *k, const void *v,
                                               void *o, int B, int H, int N, int D, int Dv,
                                               float eps, la_dtype_t dtype, void *stream);

/* Size in bytes of the per-device scratch used by la_forward_noncausal_static. */
LA_API size_t la_forward_noncausal_static_limit(void);

/* Static, NUL-terminated description of a status code. */
LA_API const char *la_status_string(la_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
