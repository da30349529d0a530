/*
 * vla.h -- C ABI of libvla, the GB300 (sm_103a) forward recurrence of
 * Variational Linear Attention (VLA).
 *
 * Operation (per batch b, head h, token t = 1..T; d = d_h):
 *   k_hat_t = k_t / max(|k_t|, eps)                         section 2.3 (unit key)
 *   z_t     = A_{t-1} u_t
 *   A_t     = A_{t-1} - z_t z_t^T / (1 + u_t^T z_t)        sections 2.2, 2.3 step 1
 *   alpha_t = A_t k_hat_t / max(|A_t k_hat_t|, eps)         section 2.3 step 2
 *   S_t     = S_{t-1} + (v_t - S_{t-1} k_hat_t) alpha_t^T   section 2.3 step 3
 *   n_t     = n_{t-1} + phi(k_hat_t),  phi(x) = ELU(x) + 1
 *   o_t     = S_t phi(q_t) / (phi(q_t)^T n_t + eps)          section 2.3 (readout)
 * with eps = 1e-6.  Sections are those of "Variational Linear Attention:
 * Stable Associative Memory for Long-Context Transformers" (web summaries);
 * z_t = A_{t-1} u_t, A_0 = I / lambda0, the readout denominator and eps are
 * this library's readings of what those pages leave open.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or synchronises inside vla_forward.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).
 *   - Device pointers must be 16-byte aligned (bulk-copy requirement).
 *   - Layouts are C-contiguous: q, k, v, u, o are [B, H, T, d];
 *     S, A are [B, H, d, d] fp32 row-major, S[i][j] maps key coordinate j
 *     to value coordinate i, A symmetric; n is [B, H, d] fp32.
 *   - Return value 0 is success; negative values are VLA_ERR_* codes.  No
 *     C++ exception crosses this boundary.
 */
#ifndef VLA_H
#define VLA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define VLA_OK 0
#define VLA_ERR_ARG (-1)             /* null required pointer, negative size, bad lambda0/dtype/kernel */
#define VLA_ERR_UNSUPPORTED_DIM (-2) /* d_h not in {32, 64, 128} */
#define VLA_ERR_ALIGN (-3)           /* a pointer is not 16-byte aligned */
#define VLA_ERR_WORKSPACE (-4)       /* workspace missing or smaller than vla_workspace_bytes() */
#define VLA_ERR_CUDA (-5)            /* a CUDA runtime call failed; see vla_last_cuda_error() */
#define VLA_ERR_TIMEOUT (-6)         /* a bounded device-side wait gave up (vla_device_status) */
#define VLA_ERR_SCRATCH_LIMIT (-7)   /* vla_forward_noalloc: problem exceeds its built-in scratch */

/* I/O element types of q, k, v, u and o */
#define VLA_F32 0
#define VLA_BF16 1

/* kernel selection */
#define VLA_KERNEL_AUTO 0  /* pick by shape */
#define VLA_KERNEL_SEQ 1   /* one CTA per (b, h), token-sequential, no workspace */
#define VLA_KERNEL_CHUNK 2 /* chunk-parallel over T, needs workspace */
#define VLA_KERNEL_DECODE 3 /* a few tokens per call (decode step), state streamed from HBM */
#define VLA_KERNEL_CHUNK_TC 4 /* VLA_KERNEL_CHUNK with the gates and the state passes on the
                               * tcgen05 tensor cores (block Woodbury, UT transform): d_h = 64
                               * with bf16 I/O and chunks a multiple of 64 tokens, and d_h = 128
                               * with bf16 I/O and one chunk per (b, h) unit (the default
                               * chunk length there when B*H >= 128); other shapes run exactly
                               * as VLA_KERNEL_CHUNK.  Workspace from vla_workspace_bytes */

/*
 * vla_forward -- run the recurrence over T tokens for all B*H units.
 *
 * q, k, v, u   [B,H,T,d] io_dtype, read only.  Required when B*H*T > 0.
 * io_dtype     VLA_F32 or VLA_BF16.
 * lambda0      > 0 and finite; A_0 = I / lambda0 when A0 is NULL.
 * B, H, T      >= 0.  T = 0 copies the initial state to the outputs.
 * d_h          32, 64 or 128.
 * S0, A0, n0   optional initial state ([B,H,d,d], [B,H,d,d], [B,H,d] fp32);
 *              NULL means 0, I/lambda0 and 0.  S0 == S_T, A0 == A_T and
 *              n0 == n_T are allowed (in-place streaming); other overlaps
 *              between inputs and outputs are not.
 * o            [B,H,T,d] io_dtype, written.
 * S_T, A_T     [B,H,d,d] fp32, written (required).
 * n_T          [B,H,d] fp32, written when non-NULL.
 * kernel       VLA_KERNEL_AUTO / _SEQ / _CHUNK / _CHUNK_TC / _DECODE.  AUTO takes DECODE for
 *              T <= 4; CHUNK_TC at d_h = 128 with bf16 I/O when B*H >= 128 and T >= 256,
 *              and for any d_h when B*H < 304 and T >= 1024; SEQ otherwise.
 * chunk        chunk length for VLA_KERNEL_CHUNK and _CHUNK_TC (0 = library default).
 * workspace    device scratch of at least vla_workspace_bytes(...) bytes
 *              (may be NULL when that is 0).  Contents on entry are ignored.
 * stream       cudaStream_t as void*.
 * Returns VLA_OK or a VLA_ERR_* code; on error nothing has been launched.
 */
int vla_forward(const void *q, const void *k, const void *v, const void *u, int io_dtype,
                float lambda0, int B, int H, int T, int d_h, const float *S0, const float *A0,
                const float *n0, void *o, float *S_T, float *A_T, float *n_T, int kernel,
                int chunk, void *workspace, size_t ws_bytes, void *stream);

/*
 * vla_forward_host -- vla_forward for inputs and outputs in host memory, with
 * the uploads overlapped with the first passes.
 *
 * The recurrence reads u and k in its first passes (the chunk Grams, their
 * prefix and the gates of sections 2.2-2.3 of "Variational Linear Attention:
 * Stable Associative Memory for Long-Context Transformers") and q and v only
 * from the state pass on, and every pass works per (b, h) unit.  On the
 * tensor-core path (two or more units) the call therefore runs the passes in
 * ranges of units as their inputs land: u and k go to the device on
 * copy_stream in two halves of the units, each followed on `stream` by its
 * Grams, prefix and gates; then q and v in two or three ranges, each
 * followed by its state pass, chain and output pass.  The o of every range
 * but the last comes back on copy_stream once all uploads are queued; the
 * last range's o (and the final state for the non-NULL host pointers among
 * hS_T, hA_T, hn_T) comes back on `stream`, which finally waits for
 * copy_stream: everything the call queued is complete once `stream` is.  At
 * d_h = 128 with one chunk per unit the ranges are waves of at most 152 units
 * (up to four): u and k range by range, each followed by its gates; then q
 * and v range by range, each followed by its state pass and, on `stream`,
 * the download of its o.  The sequential kernel (two or more units, T > 0) is
 * staged the same way: q, k, v, u of at most four ranges of units in turn, each
 * followed by the kernel over the range and, on `stream`, its o.  With a
 * download_stream, on every staged path every
 * range's o comes back on it as soon as the range's passes are done, beside
 * the later uploads and passes (the link carries both directions at once),
 * and `stream` finally waits for it.  On the other paths u and k go first, the kernels wait for them before the
 * first launch and for q and v before the first pass that reads them, and
 * all outputs come back on `stream`.  ev_uk and ev_qv carry these
 * dependencies (each is recorded more than once).  The uploads start after
 * the work queued on `stream` before the call.  The results are those of
 * vla_forward on the same data, bit for bit.
 *
 * hq, hk, hv, hu  host [B,H,T,d] io_dtype, read; page-locked memory lets the
 *                 copies run asynchronously (pageable memory still works).
 * ho              host [B,H,T,d] io_dtype, written.
 * hS_T, hA_T, hn_T  optional host copies of S_T, A_T, n_T (hn_T needs n_T).
 * q, k, v, u, o   device staging buffers owned by the caller, as in
 *                 vla_forward; q, k, v, u are overwritten by the uploads.
 * S0 .. ws_bytes  as in vla_forward.
 * stream          the compute stream; copy_stream a second stream (cudaStream_t
 *                 as void*; the same stream works, without overlap).
 * download_stream optional third stream for the downloads of o on the staged
 *                 paths (NULL: as described above; ignored on the other paths).
 * ev_uk, ev_qv    two cudaEvent_t (as void*) the call records; required.
 * Asynchronous: the host buffers must stay valid until `stream` has passed
 * the call's work.  Returns as vla_forward; on an argument error nothing is
 * queued.  On VLA_ERR_CUDA (a failed copy, record or launch) the work queued
 * before the failure may still run on every stream given: synchronise them before
 * reusing the buffers.
 */
int vla_forward_host(const void *hq, const void *hk, const void *hv, const void *hu, int io_dtype,
                     float lambda0, int B, int H, int T, int d_h, const float *S0, const float *A0,
                     const float *n0, void *q, void *k, void *v, void *u, void *o, void *ho, float *S_T,
                     float *A_T, float *n_T, float *hS_T, float *hA_T, float *hn_T, int kernel, int chunk,
                     void *workspace, size_t ws_bytes, void *stream, void *copy_stream, void *ev_uk,
                     void *ev_qv, void *download_stream);

/* Workspace bytes for these arguments, enough for vla_forward and for
 * vla_forward_host (0 for the sequential kernel).  On the tensor-core path at
 * d_h = 64 with bf16 I/O the host entry runs the two halves of the units as
 * problems of their own, side by side in the workspace (vla_host_ranges), which
 * can take a little more than vla_forward alone.  Returns 0 for invalid
 * arguments as well. */
size_t vla_workspace_bytes(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk);

/* The chunk lengths vla_forward uses on the chunked paths for these
 * arguments: S-chunks of *C tokens (the state pass, the chain along the chunks,
 * the readout) and A-chunks of *CA tokens (the Grams and the gates; CA divides
 * C).  Both 0 when the call does not take a chunked path.  Returns VLA_OK, or
 * the argument checks' VLA_ERR_* code (C and CA untouched). */
int vla_chunk_lengths(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk, int *C, int *CA);

/* The ranges of units vla_forward_host stages on the tensor-core path at
 * d_h = 64 with bf16 I/O: *n ranges (2 or 3: half the units, then the rest in
 * one or two), range r from unit lo[r] (lo[n] = B * H), with S- and A-chunk
 * lengths C[r] = CA[r].  The two halves are problems of their own, each with
 * chunk when given; else the first half takes vla_forward's default S-chunk
 * length for the whole problem, and the second half the S-chunk length of a
 * lone pass over its last range when that is at least 512 tokens (the passes
 * over that range, which run after the last upload, then fill the GPU for
 * fewer sub-blocks), otherwise the first half's.  A range's results are those
 * of vla_forward on its units with chunk = C[r].
 * *n = 0 when the call does not
 * stage this way.  lo holds at least 4 entries, C and CA at least 3.  Returns
 * VLA_OK or the argument checks' VLA_ERR_* code. */
int vla_host_ranges(int B, int H, int T, int d_h, int io_dtype, int kernel, int chunk, int *n, int *lo, int *C,
                    int *CA);

/* Which kernel VLA_KERNEL_AUTO resolves to for this shape and I/O type
 * (VLA_KERNEL_SEQ, VLA_KERNEL_CHUNK_TC or VLA_KERNEL_DECODE), or a VLA_ERR_*
 * code for invalid arguments. */
int vla_select_kernel(int B, int H, int T, int d_h, int io_dtype);

/* Static, human-readable text for a status code. */
const char *vla_status_str(int status);

/* The cudaError_t value of the last failed CUDA call on this host thread
 * (0 if none). */
int vla_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the device error word that
 * bounded waits set on expiry.  Returns VLA_OK, VLA_ERR_TIMEOUT, or
 * VLA_ERR_CUDA. */
int vla_device_status(void *stream);

/* Test hook for the failure path: mode 1 makes the next vla_forward launches
 * of the sequential kernel wait for an input tile that is never requested,
 * and the gates jobs of the tensor-core queue launches (d_h = 64 and 128)
 * leave their flags unset, so that the bounded waits (limit `wait_limit_ns`,
 * clamped to [1e5, 1e10]) expire and set the device error word; the waiting
 * state passes are then skipped and the launch ends.  Mode 0 restores normal
 * operation and the default one-second limit.  Host state only; returns
 * VLA_OK or VLA_ERR_ARG. */
int vla_debug_inject(int mode, long long wait_limit_ns);

/* Measurement hook.  With n > 0, every later vla_forward (or
 * vla_forward_host) call records events[0] on its stream before its first
 * kernel and events[i] right after its i-th kernel, for i < n, so that a
 * caller can time each launch with cudaEventElapsedTime on the launching
 * stream (on the host entry the first record follows the wait for the first
 * uploads).  events are cudaEvent_t handles (as void*) created and owned by the
 * caller.  n = 0 or events = NULL turns recording off.  Process-wide host
 * state; returns VLA_OK, or VLA_ERR_ARG when n is negative or above 64. */
int vla_set_launch_events(void *const *events, int n);

/* Number of kernels the last successful vla_forward call on this host
 * thread launched: 1 for the sequential and decode paths and for the
 * tensor-core path at d_h = 128; 6 for the chunked one, or 5 on the
 * tensor-core path at d_h = 64 when its gates and state pass run as one queue
 * launch; one more for the inverse of A0, when given, on the chunked path and
 * the tensor-core path at d_h = 64. */
int vla_last_launch_count(void);

/*
 * vla_backward -- gradients of the recurrence (reverse mode).
 *
 * Loss L = sum_t <dO_t, o_t> + <dS_T, S_T> + <dA_T, A_T> + <dn_T, n_T>, with
 * o, S_T, A_T, n_T the outputs of vla_forward on the same inputs and initial
 * state.  The transition of S, J_t = I - alpha_t k_hat_t^T, is the one of
 * section 3.1 (Proposition 2); at |k| <= eps or |A_t k_hat| <= eps the
 * max(., eps) guards pass the gradient of their constant branch.
 *
 * q, k, v, u, dO  [B,H,T,d] io_dtype (dO: upstream gradient of o).
 * S0, A0, n0      initial state as in vla_forward (NULL = defaults).
 * dS_T, dA_T, dn_T upstream gradients of the final state, or NULL (= 0).
 * dq, dk, dv, du  [B,H,T,d] fp32, written when non-NULL.
 * dS0, dA0, dn0   gradients of the initial state ([B,H,d,d], [B,H,d,d],
 *                 [B,H,d] fp32), written when non-NULL.  dA0 is the full,
 *                 unsymmetrised adjoint of A_0.
 * d_h             32, 64 or 128 (VLA_ERR_UNSUPPORTED_DIM otherwise).
 * workspace       at least vla_backward_workspace_bytes(B, H, T, d_h) bytes.
 * At d_h = 32 and 64, when the stream spans two or more chunks of the chunked forward
 * (vla_forward's default chunk length), the call runs that forward for the
 * chunk-start states and then works on all chunks in parallel: over a chunk
 * the adjoint of S is an affine map with one d x d product (the chunk's
 * transitions of section 3.1), the symmetric part of the adjoint of A (the
 * only part that feeds back) a two-sided one, and the adjoint of n a sum, so
 * short chains along the chunks give every chunk its end adjoints.  Shorter
 * streams run one CTA per (b, h), which reruns the forward (records and a
 * state checkpoint every 64 tokens) and sweeps the tokens in reverse.  At
 * d_h = 128 every stream takes that sequential form, with S and its adjoint
 * in shared memory (A and its adjoint in registers).
 * Asynchronous on stream; returns VLA_OK or a VLA_ERR_* code.
 */
int vla_backward(const void *q, const void *k, const void *v, const void *u, const void *dO,
                 int io_dtype, float lambda0, int B, int H, int T, int d_h, const float *S0,
                 const float *A0, const float *n0, const float *dS_T, const float *dA_T,
                 const float *dn_T, float *dq, float *dk, float *dv, float *du, float *dS0,
                 float *dA0, float *dn0, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes of vla_backward (0 for invalid arguments). */
size_t vla_backward_workspace_bytes(int B, int H, int T, int d_h);

/* Size of the device scratch array built into the library for
 * vla_forward_noalloc.  It is a static device array: each GPU holds its
 * 64 MiB from the moment the library's code is loaded on that GPU until the
 * process exits.  Under CUDA's default lazy module loading that moment is
 * the entry point's set-up (its first call on the GPU), not library load. */
#define VLA_NOALLOC_SCRATCH_BYTES (64ull << 20)

/*
 * vla_forward_noalloc -- the chunk-parallel path of vla_forward, with its
 * workspace taken from a scratch array compiled into the library instead of
 * from the caller.  The pages have no counterpart: this is an integration
 * entry point, not part of the method.
 *
 * Who it is for: hosts that own all device memory themselves and never let
 * a component call cudaMalloc, for example a serving runtime that reserves
 * its whole memory budget at start-up so that a long stream can never fail
 * mid-sequence on an allocation and the request path never stalls in the
 * allocator, or a plugin loaded into such a runtime that is handed only its
 * input and output buffers.  Such callers cannot allocate a workspace to
 * pass to vla_forward.
 *
 * Arguments and results are those of vla_forward with kernel =
 * VLA_KERNEL_CHUNK (chunk: chunk length, 0 = library default); inputs and
 * outputs are still the caller's device buffers.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Set-up: the array's device address is looked up (cudaGetSymbolAddress,
 * with the device current) by the first call on each device, and again by
 * the first call in a different driver context of that device (after a
 * cudaDeviceReset, say); the address is kept per device together with the
 * id of the context it belongs to.  Make that first call before any stream
 * capture begins.  A call with B = 0 (every pointer may then be NULL) does
 * the set-up and nothing else: a host that takes its memory budget at
 * start-up should make it first, so that the 64 MiB are already held.
 *
 * Limits and sharing:
 *   - Problems whose chunked workspace (vla_workspace_bytes with
 *     VLA_KERNEL_CHUNK and the same chunk) exceeds VLA_NOALLOC_SCRATCH_BYTES
 *     are rejected with VLA_ERR_SCRATCH_LIMIT before anything is launched.
 *   - The array is a single static device allocation per GPU that every
 *     call on that GPU shares, and it keeps the previous call's contents.
 *     Nothing in it needs to start at zero: every word a call reads from it
 *     is written earlier in the same call.  Calls that overlap on the GPU
 *     (different streams, or different host threads without ordering)
 *     race on the array and produce garbage; serialise them.
 * Returns VLA_OK or a VLA_ERR_* code.
 */
int vla_forward_noalloc(const void *q, const void *k, const void *v, const void *u, int io_dtype,
                        float lambda0, int B, int H, int T, int d_h, const float *S0,
                        const float *A0, const float *n0, void *o, float *S_T, float *A_T,
                        float *n_T, int chunk, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int vla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VLA_H */
