/*
 * s4.h -- C ABI of libs4: forward pass of the S4 structured state-space layer
 * on one NVIDIA GB300 (sm_103a).
 *
 * Model (page "Recurrent, LSTM, and structured state-space models", sections on
 * the complex SISO state-space model and "DPLR structured state-space
 * parameterization"):  per channel h,
 *     A = Lambda - P Q^*          (Lambda diagonal N x N, P, Q in C^{N x r})
 *     Abar = (I - Delta A/2)^{-1} (I + Delta A/2),  Bbar = (I - Delta A/2)^{-1} Delta B
 *     K_j  = C^* Abar^j Bbar,  0 <= j < L          (length-L convolution kernel)
 *     y_t  = sum_{j<=t} K_j u_{t-j} + D u_t         (causal convolution + skip term)
 * The kernel is generated from the truncated output vector
 *     C~ = (I - Abar^M)^* C,   M = least power of two >= L,
 * which the filter procedure receives as given data.
 *
 * Conventions for every entry point
 *  - Complex numbers are s4_c32 = {re, im} fp32 pairs (the memory layout of
 *    torch.complex64 / std::complex<float>).  All arrays are dense row-major.
 *  - Every array pointer is a DEVICE pointer owned by the caller.  The library
 *    allocates no device memory and keeps no state between calls other than
 *    per-device kernel attributes (and the fixed scratch array of
 *    s4_conv_fwd_noalloc).  `ws` is caller-owned device scratch of at
 *    least s4_workspace_bytes(...) bytes, 256-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *    enqueued asynchronously on it; no entry point synchronises the host
 *    except s4_get_status.
 *  - Argument errors are detected on the host before anything is enqueued
 *    and returned synchronously.  Conditions that depend on device data
 *    (resonances, non-finite values, a bad step size) are recorded in a
 *    status block at the start of `ws` and read with s4_get_status; when one
 *    is recorded, the affected output (K, or y) is written as all zeros.
 *    The block holds the flags, the generation they were set under and the
 *    generation of the last call.  Called on a stream that is not being
 *    captured, s4_kernel_gen, s4_conv_fwd, s4_conv_fwd_real and
 *    s4_layer_fwd tag their flags with a fresh generation instead of
 *    clearing the block, so such a call is kernels only and chains to the
 *    kernel before it on the stream.  Captured into a CUDA graph (a captured
 *    call would replay its generation), and for s4_ctilde and
 *    s4_recurrent_fwd, a call clears the block first (an enqueued memset).
 *    Either way s4_get_status reports the last call only, whatever `ws` held
 *    before.
 *  - Concurrent calls that share one `ws` race; give each stream its own.
 *
 * Supported sizes: 1 <= H, 1 <= N <= 65536, 1 <= r <= 4, 1 <= L <= 65536,
 * 1 <= batch.  Arrays u, y, K must be 16-byte aligned; others 8-byte aligned.
 */
#ifndef S4_H_
#define S4_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct { float re, im; } s4_c32;

typedef enum {
    S4_OK = 0,
    S4_ERR_INVALID_ARG = 1,          /* null pointer, size out of range, misaligned */
    S4_ERR_WORKSPACE = 2,            /* ws missing, misaligned or too small */
    S4_ERR_RESONANT_DIAGONAL = 3,    /* s(z_k) - lambda_j == 0 in fp32 at some root */
    S4_ERR_RESONANT_CORRECTION = 4,  /* I_r + Q^* R(z_k) P singular at some root */
    S4_ERR_NONFINITE = 5,            /* a root value or spectrum entry is inf/nan */
    S4_ERR_INVALID_STEP = 6,         /* some Delta_h <= 0 or not finite */
    S4_ERR_CUDA = 7,                 /* a CUDA runtime call or launch failed */
    S4_ERR_SINGULAR_BILINEAR = 8,    /* G = I - (Delta/2) A not solved: I_r + (Delta/2) Q^* D^{-1} P is
                                        exactly singular; or, where some d_j = 1 - (Delta/2) lambda_j is
                                        exactly 0, more such d_j than r, or a singular bordered matrix */
    S4_ERR_TIMEOUT = 9               /* a kernel's bounded wait for an asynchronous copy into shared
                                        memory ran out (the affected output is zeros) */
} s4_status;

/* Bytes of scratch that s4_kernel_gen, s4_conv_fwd and s4_layer_fwd need for
 * these sizes (the same number serves all three).  Returns 0 if the sizes are
 * outside the supported range. */
size_t s4_workspace_bytes(int H, int N, int r, int L, int batch);

/*
 * s4_kernel_gen -- the S4 filter: length-L kernel K from (Lambda, P, Q, B, C~, Delta).
 * Page "Recurrent, LSTM, and structured state-space models", section "DPLR
 * structured state-space parameterization", filter mode: with
 * s(z) = (2/Delta)(1-z)/(1+z), R(z) = diag(1/(s(z) - lambda_j)),
 * W(z) = I_r + Q^* R(z) P, the root values
 *     H(z) = 2/(1+z) (C~^* R B - C~^* R P W^{-1} Q^* R B)
 * at the M roots z_k = exp(-2 pi i k/M) (z = -1 by its finite value
 * (Delta/2) C~^* B), followed by the inverse radix-two transform; K is its
 * first L coefficients.  The resolvent sums are evaluated directly over the N
 * poles in fp32 (the (r+1)^2 Cauchy sums of that section).
 *   Lambda [H][N]    diagonal entries lambda_j per channel
 *   P, Q   [H][N][r] low-rank factors (A = Lambda - P Q^*)
 *   B      [H][N]    input vector
 *   Ctilde [H][N]    truncated output vector C~_M
 *   dt     [H]       step sizes Delta_h (fp32, must be > 0 and finite; checked on the device)
 *   K      [H][L]    output kernel
 * Device-detected statuses: S4_ERR_RESONANT_DIAGONAL, S4_ERR_RESONANT_CORRECTION,
 * S4_ERR_NONFINITE, S4_ERR_INVALID_STEP (then K is all zeros).
 */
s4_status s4_kernel_gen(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q,
                        const s4_c32* B, const s4_c32* Ctilde, const float* dt,
                        int H, int N, int r, int L, s4_c32* K,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * s4_conv_fwd -- causal convolution plus skip term for a batch of sequences.
 * Page "Recurrent, LSTM, and structured state-space models": y_t = sum_{j<=t}
 * K_j u_{t-j} + D u_t (direct term added separately); section "Roots-of-unity
 * orthogonality and radix-two FFT cost": polynomial products by zero-padding
 * to a radix-two length >= 2L-1.  Computed per row with FFTs of length 2M.
 *   u [batch][H][L] real fp32 inputs
 *   K [H][L]        kernel (complex)
 *   D [H]           skip coefficients
 *   y [batch][H][L] complex outputs
 * Device-detected status: S4_ERR_NONFINITE (a non-finite kernel spectrum; y is zeros).
 */
s4_status s4_conv_fwd(const float* u, const s4_c32* K, const float* D,
                      int batch, int H, int L, s4_c32* y,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * s4_conv_fwd_real -- real-output variant: y = Re(K) * u + D u with real y.
 * The pages take no real part (K and y are complex); this variant serves the
 * common layer convention that keeps only the real part of the kernel.  Its
 * kernel spectrum is Hermitian, so two batch rows share one complex forward
 * and one complex inverse transform, and y takes 4 bytes per sample.
 *   u [batch][H][L] real inputs; K [H][L] complex (its real part is used);
 *   D [H]; y [batch][H][L] real fp32 outputs.  ws as for s4_conv_fwd.
 * Device-detected status: S4_ERR_NONFINITE (y zeros).
 */
s4_status s4_conv_fwd_real(const float* u, const s4_c32* K, const float* D,
                           int batch, int H, int L, float* y,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * s4_layer_fwd -- s4_kernel_gen followed by s4_conv_fwd on the same stream.
 * K [H][L] receives the generated kernel (caller-owned; it is also an input of
 * the convolution).  Statuses as for the two steps; a device-detected status
 * from kernel generation makes both K and y all zeros.
 */
s4_status s4_layer_fwd(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q,
                       const s4_c32* B, const s4_c32* Ctilde, const float* dt,
                       const float* D, const float* u,
                       int batch, int H, int N, int r, int L,
                       s4_c32* K, s4_c32* y,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * s4_conv_fwd_noalloc -- s4_conv_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a service entry point of the library.
 * Some callers cannot call cudaMalloc: a host program that owns all device
 * memory through its own pool and forbids allocations by the libraries it
 * loads, or a latency-critical loop where an allocation (which can
 * synchronise the device) is not acceptable.  They cannot provide `ws`, so
 * this variant keeps its scratch (the status word and the kernel spectrum)
 * in a fixed array of S4_NOALLOC_SCRATCH_BYTES compiled into the library;
 * every device that loads the library holds that array until the process exits.
 *   Arguments, layouts and results as for s4_conv_fwd; no ws, no ws_bytes.
 *   Limit: 256 + 16 * H * M bytes of scratch (M = least power of two >= L)
 *   must fit S4_NOALLOC_SCRATCH_BYTES (8 MiB; e.g. H * M <= 524272), else
 *   S4_ERR_WORKSPACE is returned before anything is enqueued.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.
 *   All calls share the one array: calls that can overlap on the GPU (work
 *   on streams not ordered with each other) race and must not be issued.
 *   A non-finite kernel spectrum writes y as zeros; no status block is exposed.
 *   Allocates nothing: no cudaMalloc/cudaFree and no allocating library call.
 */
#define S4_NOALLOC_SCRATCH_BYTES (8u << 20)
s4_status s4_conv_fwd_noalloc(const float* u, const s4_c32* K, const float* D,
                              int batch, int H, int L, s4_c32* y, void* stream);

/*
 * s4_ctilde -- form the truncated output vector from a conventional C.
 * Page "Recurrent, LSTM, and structured state-space models": for a filter of
 * transform length M (least power of two >= L) the output vector is
 * C~ = (I - Abar^M)^* C; the filter procedure receives it as given data, and
 * this entry point forms it.  Computed as C - (Abar^*)^M C, Abar^* w =
 * 2 G^{-*} w - w (G = I - (Delta/2) A) being a diagonal plus a rank-r term
 * (the Woodbury form of G^{-*}); the kernel squares that form to Abar^{*p}
 * (diagonal plus rank p r) and takes M/p steps of it.  A channel with an
 * exactly zero d_j = 1 - (Delta/2) lambda_j takes M single steps instead, each
 * solving G^* by the conjugated bordered system of s4_recurrent_fwd.
 *   Lambda, P, Q, dt as for s4_kernel_gen; C [H][N] (input); Ctilde [H][N] (output).
 *   N <= 256.  ws: at least 256 bytes (the status block; see s4_get_status).
 * Device-detected statuses: S4_ERR_SINGULAR_BILINEAR, S4_ERR_INVALID_STEP (Ctilde zeros).
 */
s4_status s4_ctilde(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const float* dt,
                    const s4_c32* C, int H, int N, int r, int L, s4_c32* Ctilde,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * s4_recurrent_fwd -- the recurrent mode over L steps, for streaming inference.
 * Page "Recurrent, LSTM, and structured state-space models", section "DPLR
 * structured state-space parameterization", recurrent mode:
 *     b_t = (I + (Delta/2) A) x_{t-1} + Delta B u_t,   G x_t = b_t,   y_t = C^* x_t + D u_t,
 * G solved by the Woodbury inverse with D = diag(1 - (Delta/2) lambda_j); in a
 * channel where some of those d_j are exactly 0 in fp32 (the set Z, s = |Z| <= r),
 * by the pages' bordered system of size r + s for (Q^* x, x_Z), with
 * x_J = D_J^{-1}(b_J - (Delta/2) P_J Q^* x) on the other states.
 *   Lambda, P, Q, B, dt, D as for s4_layer_fwd; C [H][N] is the conventional
 *   output vector (not C~).  u [batch][H][L] inputs; y [batch][H][L] outputs.
 *   x [batch][H][N]: the state x_{-1} on entry and x_{L-1} on return, so
 *   consecutive calls continue one sequence (zeros for a fresh sequence).
 *   N <= 256.  ws: at least 256 bytes (the status block).
 * Device-detected statuses: S4_ERR_SINGULAR_BILINEAR, S4_ERR_INVALID_STEP (y and x zeros).
 */
s4_status s4_recurrent_fwd(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q,
                           const s4_c32* B, const s4_c32* C, const float* dt, const float* D,
                           const float* u, int batch, int H, int N, int r, int L,
                           s4_c32* x, s4_c32* y, void* ws, size_t ws_bytes, void* stream);

/*
 * s4_hippo_dplr -- HiPPO state matrix in DPLR form (host routine, float64).
 * Page "Recurrent, LSTM, and structured state-space models", the paragraph on
 * the HiPPO generators and the DPLR / NPLR definitions:
 *   kind S4_HIPPO_LEGS: G_nk = -sqrt((2n+1)(2k+1)) (n > k), -(n+1) (n = k), 0 (n < k)
 *   kind S4_HIPPO_LEGT: G_nk = -(2n+1)(-1)^(n-k)/theta (n >= k), -(2n+1)/theta (n < k),
 *                       taken through the similarity S_0 = diag(sqrt(2n+1)) diag((-1)^n)
 *   kind S4_HIPPO_LAGT: G_nk = -1 (n >= k), 0 (n < k)
 * The (similar) generator is split as H - U U^T with H normal and U of rank
 * r = 1 (LegS, LagT) or 2 (LegT); a unitary W with H = W diag(Lambda) W^*
 * (eigenvectors of a Hermitian matrix, by cyclic Jacobi rotations) gives
 *     W^* S^{-1} G S W = diag(Lambda) - P P^*,   P = W^* U,
 * i.e. the DPLR form with Q = P, and the state change x = S W x~ maps the
 * input and output vectors to B~ = W^* S^{-1} B and C~ = W^* S^* C.
 *   N: 1 .. 512.  theta: window of LegT (> 0, finite; ignored otherwise).
 *   B, C: optional inputs [N] complex (interleaved re, im doubles; NULL = none).
 *   Lambda [N] complex, P [N][r] complex (caller allocates room for [N][2]),
 *   Bt, Ct [N] complex (required when B, C are given), *rank = r: outputs.
 * All pointers are HOST pointers.  Runs synchronously on the calling thread,
 * uses no GPU and allocates only host scratch.  Eigenvalues are returned in
 * ascending order of Im Lambda; eigenvector phases (and so P, B~, C~) are
 * one valid choice among many, while Lambda - P P^* is unique up to the
 * unitary freedom of W and the kernel C^* Abar^j Bbar is unique.
 * Returns S4_ERR_INVALID_ARG on bad arguments; S4_ERR_NONFINITE if the
 * eigen-iteration does not converge.
 */
typedef enum { S4_HIPPO_LEGS = 0, S4_HIPPO_LEGT = 1, S4_HIPPO_LAGT = 2 } s4_hippo_kind;
s4_status s4_hippo_dplr(int kind, int N, double theta, const double* B, const double* C,
                        double* Lambda, double* P, double* Bt, double* Ct, int* rank);

/* Synchronises `stream`, then returns the device-detected status recorded in
 * `ws` by the last entry point that used it (S4_OK if none), or
 * S4_ERR_CUDA if the synchronisation or the read fails. */
s4_status s4_get_status(const void* ws, void* stream);

/* A static, human-readable name for a status value. */
const char* s4_status_str(s4_status st);

/* Optional per-kernel timing: when enabled, every kernel launch of the
 * library is bracketed by CUDA events recorded on its launch stream.
 * s4_timing_read syncs those events and returns, for the kernel family
 * `name` ("cauchy", "ifft", "spectrum", "kspec", "conv", "conv_real",
 * "recurrent", "ctilde", "bordered"), the number of launches and their summed duration
 * in milliseconds since the last reset.  Timing state is per process; it is
 * meant for benchmarks, not for use from several host threads at once. */
void s4_timing_enable(int on);
void s4_timing_reset(void);
int  s4_timing_read(const char* name, int* launches, double* total_ms);

/* Fault-detection test hook, outside the method: the number of polls a
 * kernel's bounded wait on an asynchronous copy into shared memory makes
 * before it gives up and records S4_ERR_TIMEOUT (default 4194304; polls < 0
 * restores the default, 0 makes every such wait give up at once).  Only the
 * staged kernels wait this way: the convolution of rows of 2M = 8192 points
 * and the layer's kernel spectrum for M <= 1024.  A kernel whose wait gave up
 * issues no further copies, reads the data from global memory instead, waits
 * for the copy in flight once more (default limit) before it exits, and
 * writes its output as zeros.  Library-wide and read at launch time; meant
 * for tests of that path, not for concurrent use.  Returns S4_OK. */
s4_status s4_set_wait_limit(int polls);

/* Test aid, outside the method: in a library built with -DS4_BOUNDS_CHECK
 * (a separate build for tests), every global and shared-memory index of the
 * instrumented kernels is compared with its buffer's extent, and an index outside
 * it is counted and its access skipped (nothing traps).  Returns the number counted
 * since the library was loaded (after synchronising the device), -2 if the counters
 * cannot be read, and -1 in the normal build, which has no checks. */
long long s4_bounds_violations(void);

/* Measurement aid, outside the method: an FP32 issue-rate probe.  Launches
 * `blocks` CTAs of 256 threads on `stream`; every thread runs `iters`
 * iterations (rounded up to a multiple of 8) of 8 independent fused
 * multiply-adds, 16 flop each, so one launch executes
 * blocks x 256 x iters x 16 flop, and each thread writes one float to `out`
 * (device memory, blocks x 256 floats, caller-owned) so that nothing is
 * elided.  The caller times the launch (CUDA events on `stream`) to compare
 * the FP32 peak derived from unit counts and clocks with the rate the SMs
 * sustain.  Asynchronous; S4_ERR_INVALID_ARG for a null `out`, blocks < 1 or
 * iters < 1; S4_ERR_CUDA if the launch fails. */
s4_status s4_fp32_probe(float* out, int blocks, int iters, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* S4_H_ */
