/*
 * m3scan.h -- C ABI of the B300 (sm_103a) Mamba-3 scan library, libm3scan.so.
 *
 * The scan (Mamba-3, "Improved Sequence Modeling using State Space
 * Principles"): per batch row b and head h,
 *
 *   h_t = alpha_t R_t h_{t-1} + beta_t R_t B_{t-1} x_{t-1}^T + gamma_t B_t x_t^T
 *   y_t = C_t^T h_t
 *
 *   alpha_t = exp(Delta_t A),  beta_t = (1 - lambda_t) Delta_t alpha_t,  gamma_t = lambda_t Delta_t
 *       -- exponential-trapezoidal discretisation, [A] sec. 4.1, Prop. 1
 *   R_t = block-diagonal 2x2 rotations [[cos,-sin],[sin,cos]] by Delta_t theta[t,k] on state
 *         rows (2k, 2k+1)  -- complex-valued state, [A] sec. 4.2 (Prop. 2/3);
 *         rotation matrix from [X] sec. 2.2
 *   B_t = B[b,t,g] + B_bias[h] (N x R), C_t = C[b,t,g] + C_bias[h], x_t (P x R)
 *       -- MIMO rank R, [N] sec. 3; head-specific B/C bias, [N] sec. 4
 *
 * Sources (web pages on the method), cited by letter with the page's section:
 *   [A] "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc)
 *   [N] "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)
 *   [X] "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog)
 *   [U] "Mamba-3: Improved Sequence Modeling using State Space Principles" (bud-325 notes)
 *   g = h / (H / G): heads are split into G equal groups that share B, C and theta.
 *   h_{-1} = 0 and B_{-1} x_{-1} = 0 for prefill.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers to row-major, contiguous arrays
 *     (any CUDA allocation, including managed memory). The caller owns every
 *     buffer; the library keeps no allocation between calls.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream). A call returns once the work is enqueued.
 *   - Arguments are validated on the host before anything is enqueued. An
 *     invalid or unsupported call returns a non-zero status and touches no
 *     output. A failed launch returns M3_ERR_CUDA.
 *   - Kernels never trap or assert. A bounded device-side wait that expires
 *     records a flag that m3_device_status() reports as M3_ERR_TIMEOUT; the
 *     outputs of that call (and decode's state) are then unspecified.
 *   - Outputs must not alias inputs (decode's `state` is updated in place).
 *   - The library runs on compute capability 10.3 (B300) only; elsewhere the
 *     compute entry points return M3_ERR_UNSUPPORTED.
 *   - Fault injection for tests: the environment variable M3_FAULT, read at
 *     every call, makes a valid compute call return M3_ERR_INVALID_ARG before
 *     any device work ("arg"), return M3_ERR_CUDA in place of its launches
 *     ("launch") or of the library's own scratch allocation ("alloc"), or run
 *     a kernel whose bounded device wait expires after 1 ms in place of the
 *     work ("timeout"; m3_device_status then reports M3_ERR_TIMEOUT). Outputs
 *     and state are left untouched in every mode.
 */
#ifndef M3SCAN_H_
#define M3SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  M3_OK = 0,
  M3_ERR_INVALID_ARG = 1, /* null pointer, negative size, odd N, G not dividing H, ... */
  M3_ERR_UNSUPPORTED = 2, /* valid but not implemented: dtype, shape, device arch      */
  M3_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed                      */
  M3_ERR_TIMEOUT = 4      /* a bounded device-side wait expired (see m3_device_status) */
} m3_status;

typedef enum {
  M3_F32 = 0, /* x, B, C, B_prev, x_prev, out are float32 (the fp32 precision mode) */
  M3_BF16 = 1 /* ... are bfloat16; dt, lambda, theta, A, biases and state stay fp32 */
} m3_dtype;

/*
 * m3_dims.flags. Any other bit set is M3_ERR_INVALID_ARG.
 *
 * M3_FLAG_BC_NORM: B and C arrive un-normalised, and the prefill applies
 * BCNorm to them itself, fused into its prologue: every (b, t, g, r) vector
 * of B (and of C) over the N state rows is divided by its root mean square,
 *   B[b,t,g,:,r] / sqrt(mean_n B[b,t,g,n,r]^2 + 1e-6),
 * with no learned weight, before the per-head bias and the rotation
 * ([N] sec. 4, BC normalisation and B/C bias; [U] Key claims). Supported by m3_scan_fwd and m3_scan_fwd_noalloc on the tensor-core
 * path (bf16, P = 64, N in {64, 128}, chunk * R = 64, the alignments given
 * there); every other call with it returns M3_ERR_UNSUPPORTED, as do
 * m3_scan_fwd_state, the decode calls and m3_scan_bwd (normalise B and C
 * before calling those).
 */
#define M3_FLAG_BC_NORM 1

typedef struct {
  int64_t batch;   /* b  >= 0                                             */
  int64_t seqlen;  /* L  >= 0 (prefill); K (multi-token decode); ignored by decode */
  int64_t heads;   /* H  >= 1                                             */
  int64_t groups;  /* G  >= 1, divides H                                  */
  int64_t headdim; /* P  >= 1                                             */
  int64_t dstate;  /* N  >= 2, even (N/2 rotating pairs)                  */
  int32_t act_dtype;  /* an m3_dtype                                      */
  int32_t flags;      /* 0, or M3_FLAG_BC_NORM (prefill only, see below)  */
  const float* B_bias; /* [H, N, R] fp32 device pointer, or NULL (zero bias) */
  const float* C_bias; /* [H, N, R] fp32 device pointer, or NULL            */
  void* workspace;        /* device scratch for long sequences, or NULL     */
  size_t workspace_bytes; /* its size; see m3_scan_workspace_bytes()        */
} m3_dims;

/*
 * Prefill: the whole scan over L tokens (chunked SSD algorithm).
 *
 * Layouts (R = MIMO rank, N = dstate, P = headdim):
 *   x, out       [b, L, H, P, R]   act_dtype
 *   dt, lambda   [b, L, H]         fp32, dt > 0, lambda in [0, 1]
 *   A            [H]               fp32 (A < 0 decays; A = 0 allowed)
 *   B, C         [b, L, G, N, R]   act_dtype
 *   theta        [b, L, G, N/2]    fp32 (rotation rate per state pair; angle = dt * theta)
 *   final_state  [b, H, N, P]      fp32, or NULL. h_{L-1} in the explicit
 *                (unrotated) frame. It does not include the next token's
 *                beta term; m3_decode_step adds that from B_prev/x_prev.
 * `chunk` is the chunk length Q in tokens (>= 1); the chunked algorithm is
 * exact up to rounding for any Q. The tensor-core bf16 path needs Q * R = 64
 * with P = 64 and N in {64, 128}; other bf16 shapes and every fp32 shape run
 * on the CUDA-core path (still on the GPU). Out-of-range chunk sizes return
 * M3_ERR_UNSUPPORTED.
 * Scratch: on the tensor-core path, when there are fewer (b, h) sequences
 * than SMs, each sequence is cut into segments that run in parallel (a
 * state-only pass, an ordered combine of the segment states, and the full
 * pass); that needs m3_scan_workspace_bytes() bytes of device scratch. Pass it
 * in dims->workspace (16-byte aligned, at least that size, else
 * M3_ERR_INVALID_ARG), or NULL and the library allocates and frees it on
 * `stream` (cudaMallocAsync / cudaFreeAsync). Calls that need none ignore it.
 * L = 0 writes zeros to final_state (if given) and nothing else.
 */
m3_status m3_scan_fwd(const void* x, const float* dt, const float* A, const float* lambda,
                      const void* B, const void* C, const float* theta, const m3_dims* dims,
                      int R, int chunk, void* out, float* final_state, void* stream);

/*
 * Prefill that continues a sequence (chunked prefill): the same computation,
 * arguments and layouts as m3_scan_fwd over the block of L tokens, started
 * from `state` instead of zero, with the state updated in place:
 *
 *   state   [b, H, N, P] fp32: h before the block on entry (explicit frame, as
 *           returned by m3_scan_fwd's final_state, m3_decode_step or this
 *           call), h after the block on return.
 *   B_prev  [b, G, N, R] raw B and
 *   x_prev  [b, H, P, R] x of the token before the block (act_dtype); both
 *           NULL when the block starts the sequence (then the call equals
 *           m3_scan_fwd from a zero state when `state` is zero). One NULL and
 *           one non-NULL is M3_ERR_INVALID_ARG.
 * Calling m3_scan_fwd on tokens [0, L1) and then this on [L1, L1 + L2) with
 * the first call's final state and its last token as B_prev / x_prev gives
 * the outputs and final state of one m3_scan_fwd over [0, L1 + L2). R must
 * be 1, 2 or 4 (else M3_ERR_UNSUPPORTED). L = 0 leaves the state unchanged.
 * The state must not alias any other argument. Scratch as for m3_scan_fwd.
 */
m3_status m3_scan_fwd_state(const void* x, const float* dt, const float* A, const float* lambda,
                            const void* B, const void* C, const float* theta,
                            const void* B_prev, const void* x_prev, const m3_dims* dims, int R,
                            int chunk, void* out, float* state, void* stream);

/*
 * Backward pass of a prefill that starts from a zero state: the gradients of
 * the scalar <y, dy> + <h_final, d_final> with respect to every input
 * (training). Same inputs and layouts as m3_scan_fwd, plus
 *   dy        [b, L, H, P, R]  act_dtype, the gradient of the outputs
 *   d_final   [b, H, N, P]     fp32 (16-byte aligned), the gradient of the final
 *                              state, or NULL for zero
 * and fp32 gradients: dx [b,L,H,P,R], ddt and dlambda [b,L,H], dA [H],
 * dB and dC [b,L,G,N,R] (summed over the heads of a group), dtheta
 * [b,L,G,N/2], dB_bias and dC_bias [H,N,R] (each may be NULL: not computed).
 * R in {1, 2, 4}, P a multiple of 4 with P/4 dividing 32, N/2 * P/4 <= 1024;
 * other shapes return M3_ERR_UNSUPPORTED. bf16 shapes with P = 64 and
 * N in {64, 128} (x, dy, dB, dC 16-byte aligned) run a chunked backward on
 * the tensor cores (chunks of 64 / R tokens); the others a CUDA-core kernel
 * that walks each sequence forward to store a state checkpoint every 64
 * tokens, then backward chunk by chunk. Gradients shared by heads, batch rows
 * or tokens are accumulated with atomics, so their last bits can vary from
 * run to run. Scratch: dims->workspace, at least
 * m3_scan_bwd_workspace_bytes(dims, R) bytes and 16-byte aligned (smaller or
 * misaligned: M3_ERR_INVALID_ARG), or NULL, in which case the library
 * allocates and frees it on `stream` (cudaMallocAsync / cudaFreeAsync).
 */
m3_status m3_scan_bwd(const void* x, const float* dt, const float* A, const float* lambda,
                      const void* B, const void* C, const float* theta, const void* dy,
                      const float* d_final, const m3_dims* dims, int R, float* dx, float* ddt,
                      float* dA, float* dlambda, float* dB, float* dC, float* dtheta,
                      float* dB_bias, float* dC_bias, void* stream);

/*
 * Decode: one token of the recurrence for every (b, h), state updated in place.
 *
 *   state   [b, H, N, P]  fp32, h_{t-1} on entry, h_t on return (explicit frame)
 *   x, out  [b, H, P, R]  act_dtype
 *   dt, lambda [b, H] fp32;  A [H] fp32
 *   B, C    [b, G, N, R]  act_dtype (raw: the kernel adds the bias)
 *   theta   [b, G, N/2]   fp32
 *   B_prev  [b, G, N, R]  raw B of the previous token, and
 *   x_prev  [b, H, P, R]  x of the previous token; both NULL for the first
 *           token of a sequence (then B_{t-1} x_{t-1}^T = 0). One NULL and
 *           one non-NULL is M3_ERR_INVALID_ARG.
 * dims->seqlen, workspace and workspace_bytes are ignored. The product
 * B_prev x_prev^T is formed on the fly (passing N x P products per head would
 * double the step's memory traffic). bf16 at R = 4, P = 64, N a multiple of
 * 16 up to 128 (all pointers 16-byte aligned, b H a multiple of 4) forms the
 * rank-8 update on the tensor cores (mma.sync, U in bf16 high and low parts);
 * every other shape runs on the CUDA cores.
 */
m3_status m3_decode_step(float* state, const void* x, const float* dt, const float* A,
                         const float* lambda, const void* B_prev, const void* x_prev,
                         const void* B, const void* C, const float* theta, const m3_dims* dims,
                         int R, void* out, void* stream);

/*
 * Multi-token decode: K consecutive tokens of the recurrence for every (b, h)
 * in one call, state updated in place; the result equals K calls of
 * m3_decode_step in token order, token t's B_prev / x_prev being token t-1's
 * raw B and x. The state is read once and written once per call (it stays on
 * chip between the K tokens), so the state traffic per token falls by K --
 * for a block of tokens that is known in advance (speculative drafts, a
 * prompt's tail, several tokens per request).
 *
 *   state   [b, H, N, P]     fp32, h before the block on entry, after it on return
 *   x, out  [b, K, H, P, R]  act_dtype
 *   dt, lambda [b, K, H] fp32;  A [H] fp32
 *   B, C    [b, K, G, N, R]  act_dtype (raw: the kernel adds the bias)
 *   theta   [b, K, G, N/2]   fp32
 *   B_prev  [b, G, N, R]     raw B, and
 *   x_prev  [b, H, P, R]     x of the token before the block; both NULL when
 *           the block starts a sequence. One NULL and one non-NULL is
 *           M3_ERR_INVALID_ARG.
 * K = dims->seqlen (1 ... 4096; K = 0 with b H > 0 is a no-op); workspace and
 * workspace_bytes are ignored. Supported shapes: R in {1, 2, 4}, P a multiple
 * of 4 with P/4 dividing 32, N/2 * P/4 <= 1024 (a state of at most 32 KB per
 * head), every per-token block of x, B, C, theta and the biases a multiple of
 * 16 bytes and 16-byte aligned, and the block's activations within 200 KB of
 * shared memory; other valid shapes return M3_ERR_UNSUPPORTED (use
 * m3_decode_step per token). bf16 at R = 4, P = 64, N a multiple of 16 up to
 * 128 runs the tokens' updates on the tensor cores (mma.sync) when the
 * block's activations fit its shared-memory layout (about 20 tokens at
 * N = 128); other shapes run on the CUDA cores.
 */
m3_status m3_decode_tokens(float* state, const void* x, const float* dt, const float* A,
                           const float* lambda, const void* B_prev, const void* x_prev,
                           const void* B, const void* C, const float* theta,
                           const m3_dims* dims, int R, void* out, void* stream);

/*
 * Prefill that allocates no device memory: the same computation, arguments
 * and layouts as m3_scan_fwd, for callers that cannot let a library allocate
 * GPU memory -- an application or framework whose own allocator owns all of
 * the device's memory, or a latency-critical caller for which a device
 * allocation (which may block, or fail under memory pressure) is not
 * acceptable. (The paper has no counterpart; this is a library interface.)
 *
 * The scratch a call needs (m3_scan_workspace_bytes) is taken from a fixed
 * 32 MiB array of this library in device memory, held on every GPU that loads
 * the library until the process exits; dims->workspace is ignored. A call
 * that needs more than 32 MiB returns M3_ERR_UNSUPPORTED without launching
 * anything (use m3_scan_fwd with a caller workspace for those). Every call
 * looks up the current device's address of the array (a host-side runtime
 * query, no allocation), so the address stays right if the device's context
 * is destroyed and created again; the first call on a device also loads the
 * library's device code there, so make that first call before any stream
 * capture. All calls share the one array, so calls that can overlap on the
 * GPU (different streams, or different host threads, on the same device)
 * race on it; serialise them. The scan writes every scratch byte it reads, so
 * the previous call's leftovers need no clearing.
 */
m3_status m3_scan_fwd_noalloc(const void* x, const float* dt, const float* A, const float* lambda,
                              const void* B, const void* C, const float* theta,
                              const m3_dims* dims, int R, int chunk, void* out,
                              float* final_state, void* stream);

/* Bytes of device scratch m3_scan_fwd wants for these arguments when its
 * pointers are 16-byte aligned (0 if none); (size_t)-1 if the arguments are
 * invalid. Host function: reads the current device's SM count when a device
 * is present (assumes 148, a B300, otherwise); launches nothing. */
size_t m3_scan_workspace_bytes(const m3_dims* dims, int R, int chunk);

/*
 * The device scratch (bytes) m3_scan_bwd needs for these dims and R, whichever
 * of its two kernels runs (0 when there is nothing to compute); (size_t)-1
 * for invalid dims. Callers that run the backward pass repeatedly pass it
 * once allocated in dims->workspace.
 */
size_t m3_scan_bwd_workspace_bytes(const m3_dims* dims, int R);

/* Static, human-readable name of a status. Pure host function. */
const char* m3_status_string(m3_status status);

/* Synchronises `stream`, then reads and clears this device's flag of expired
 * device-side waits: M3_OK if none expired since the last call,
 * M3_ERR_TIMEOUT otherwise, M3_ERR_CUDA if the synchronisation failed. */
m3_status m3_device_status(void* stream);

/* Library version as major*10000 + minor*100 + patch. Pure host function. */
int m3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_H_ */
