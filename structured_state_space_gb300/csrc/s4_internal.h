// Internal host-side interfaces between the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace s4impl {

// The device status of one call: `w` points to the workspace's status block of
// three 32-bit words [flags, generation of the flags, generation of the last
// call]; `gen` is this call's generation.  Flags carrying another generation are
// stale and read as clear, so a call need not reset the block before its
// kernels run (gen 0: the block was zeroed by a memset before the call).
struct St {
  unsigned* w;
  unsigned gen;
};

#ifdef S4_BOUNDS_CHECK
// Out-of-extent indices counted by each translation unit's kernels (checked build).
unsigned long long oob_rows();
unsigned long long oob_cluster();
unsigned long long oob_fourstep();
unsigned long long oob_cauchy();
unsigned long long oob_recurrent();
unsigned long long oob_bordered();
#endif

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Polls a kernel's bounded wait on an asynchronous copy makes before it gives
// up (library-wide; s4_set_wait_limit changes it, for tests of that path).
int wait_limit();

// Optional event bracketing of kernel launches (see s4_timing_* in s4.h).
// Construct right before a launch and let it go out of scope right after.
class TimedLaunch {
 public:
  TimedLaunch(const char* name, cudaStream_t s);
  ~TimedLaunch();
  TimedLaunch(const TimedLaunch&) = delete;
  TimedLaunch& operator=(const TimedLaunch&) = delete;

 private:
  static void record(cudaEvent_t e, cudaStream_t s);
  int slot_;
  cudaStream_t s_;
};

// Longest rows (log2 of the length) that one CTA transforms in shared
// memory: the inverse transform of the root values holds one row, the
// convolution two (a pair of batch rows) and so stops one size earlier.
constexpr int kMaxLogRowCta = 14;
constexpr int kMaxLogConvRow = 13;

// log2 of the cluster size that splits a longer row of 2^logn points:
// 2^14 uses 2 CTAs of 2^13 (convolution only); 2^15 uses 4 of 2^13; 2^16
// uses 8 of 2^13; 2^17 uses 8 of 2^14.  Spectra of split rows are stored in
// blocked order.
__host__ __device__ constexpr int cluster_log(int logn) {
  return logn <= 13 ? 0 : (logn == 14 ? 1 : (logn == 15 ? 2 : 3));
}
// Blocked layout of the root values (inverse transform of length 2^logM).
__host__ __device__ constexpr int khat_cluster_log(int logM) {
  return logM <= kMaxLogRowCta ? 0 : cluster_log(logM);
}

// Far-field constants of the root-value sums, per channel: the centre c and
// radius R of the poles and the moments of the (r+1)^2 weight vectors, kFarTerms
// of each; kFarStride complex values per channel (room for rank 4).
constexpr int kFarTerms = 42;
constexpr int kFarStride = 2 + 25 * kFarTerms;
// Second level (rank 1, N <= kFarPermMax): the poles ranked by imaginary part and
// split into kFarGroups groups of consecutive ranks, each with its own centre,
// radius and kFarTerms moments of the 4 weight vectors (kFarGStride complex
// values), then the permutation (pole index by rank, 32-bit).  Per channel:
// kFarChannel complex values in all.
constexpr int kFarGroups = 4;
constexpr int kFarGStride = 2 + 4 * kFarTerms;
constexpr int kFarPermMax = 512;
constexpr int kFarChannel = kFarStride + kFarGroups * kFarGStride + kFarPermMax / 2;

// Root values Khat[h][p] for every channel, in the blocked root order
// (position p -> root (p mod M/C) C + p div M/C, C = 2^logC), after the far-field
// constants of every channel (into `mom`, H kFarStride complex values).  Two
// launches; the first records the call's generation (it is a call's first
// kernel); `pdl`: launch it as a programmatic dependent of the previous kernel on
// the stream, which it waits for before any memory access.
cudaError_t launch_cauchy(const float2* Lambda, const float2* P, const float2* Q, const float2* B,
                          const float2* Ct, const float* dt, float2* Khat, float2* mom, int H, int N, int r,
                          int M, int logC, St status, cudaStream_t s, bool pdl = false);

// Single-CTA row transforms (log sizes up to kMaxLogRowCta).
cudaError_t launch_ifft_rows(int logM, const float2* Khat, float2* K, int H, int L,
                             St st, cudaStream_t s);
// realk: the spectrum of Re K (real-output convolution), scaled by 1/n
// instead of 1/(2n).  The spectrum kernels are a convolution call's first
// kernel: they record the call's generation; `pdl`: launch as a programmatic
// dependent of the previous kernel on the stream (waited for before any access).
cudaError_t launch_spectrum_rows(int logn, const float2* K, float2* K2, int H, int L, St st,
                                 cudaStream_t s, bool realk = false, bool pdl = false);
// Full (unpadded) forward transforms of `rows` rows of 2^logn points (logn =
// 10..13), natural order, times `scale`; records the call's generation.
cudaError_t launch_spectrum_rows_full(int logn, const float2* X, float2* K2, int rows, float scale, St st,
                                      cudaStream_t s);
// Layer path: inverse transform of the root values and the kernel spectrum in
// one launch (rows of M = 2^logM with 2M <= 2^13; see kspec_supported),
// launched as a programmatic dependent of the root-value kernel.
bool kspec_supported(int logM);
cudaError_t launch_kspec_rows(int logM, const float2* Khat, float2* K, float2* K2, int H, int L,
                              St st, cudaStream_t s);
// (the row kernels pair batch rows; K2 from launch_spectrum_rows is scaled by 1/(2n))
// `pdl`: launch as a programmatic dependent of the previous kernel (layer path).
cudaError_t launch_conv_rows(int logn, const float* u, const float2* K2, const float* D, float2* y,
                             int batch, int H, int L, St st, cudaStream_t s,
                             bool pdl = false);

// Long-row convolution by a four-step split through global memory (2M =
// 2^14 .. 2^17 points; K2 in the blocked order of the cluster spectrum
// kernels): three launches, scratch of fs_scratch_bytes(logn, batch, H) bytes
// (two complex rows of 2M points per pair of batch rows), 16-byte aligned.
constexpr int kMinLogFourStep = 14;
constexpr int kMaxLogFourStep = 17;
// Across-column radix 2^fs_log_radix(logn) of the four-step split: 16 up to
// 2^16 points, 32 at 2^17 (columns of 4096 points).
constexpr int fs_log_radix(int logn) { return logn >= 17 ? 5 : 4; }
// K2 in the blocked order of 2^k2_logC (fs_log_radix(logn): column order from
// the four-step spectrum; cluster_log(logn): from the cluster spectrum
// kernels), stored as the spectrum times n k2_scale.
size_t fs_scratch_bytes(int logn, int batch, int H);
// K2o != nullptr: the spectrum in two halves (see launch_kspec_fourstep_half),
// the even bins in K2 and the odd bins in K2o (stored as the spectrum times n
// k2o_scale), each H x n/2 in the blocked order of 2^k2_logC over n/2 bins.
cudaError_t launch_conv_fourstep(int logn, const float* u, const float2* K2, int k2_logC, float k2_scale,
                                 const float* D, float2* y, int batch, int H, int L, float2* scratch, St st,
                                 cudaStream_t s, const float2* K2o = nullptr, float k2o_scale = 0.f);
// The four-step kernel spectrum (2M = 2^logn, 2^14..2^17) of K [H][L], in
// column order (k2_logC = fs_log_radix(logn)) scaled 8/(2M) (k2_scale = 1/8);
// scratch of fs_spec_scratch_bytes(logn, H) bytes.  Records the call's generation.
constexpr float kFsSpecScale = 0.125f;
size_t fs_spec_scratch_bytes(int logn, int H);
cudaError_t launch_spectrum_fourstep(int logn, const float2* K, float2* K2, int H, int L, float2* scratch, St st,
                                     cudaStream_t s, bool realk = false);
// Layer path, M = 2^13 .. 2^16: root values in column order (the root-value
// kernel with logC = 4) -> K (out) and its 2M spectrum as above; G: H M and X:
// H 2M complex scratch.
cudaError_t launch_kspec_fourstep(int logM, const float2* Khat, float2* K, float2* K2, int H, int L, float2* G,
                                  float2* X, St st, cudaStream_t s);
// Layer path with L = M (M = 2^13 .. 2^16): the 2M spectrum's even bins are the
// root values themselves, so only its odd bins T (H x M, scaled 8/(2M)) are
// formed, from the root values in column order of C = 2^(fs_log_radix(logM + 1) - 1)
// (the root-value kernel with logC = log C); K written out; G and X: H M complex
// scratch each.  The convolution then takes (K2 = root values, scale 1/(2M);
// K2o = T, scale 1/8; k2_logC = log C).
cudaError_t launch_kspec_fourstep_half(int logM, const float2* Khat, float2* K, float2* T, int H, int L,
                                       float2* G, float2* X, St st, cudaStream_t s);

// Cluster row transforms for longer rows (rows split over C = 2..8 CTAs).
cudaError_t launch_ifft_cluster(int logM, const float2* Khat, float2* K, int H, int L,
                                St st, cudaStream_t s);
cudaError_t launch_spectrum_cluster(int logn, const float2* K, float2* K2, int H, int L,
                                    St st, cudaStream_t s, bool realk = false);
cudaError_t launch_conv_cluster(int logn, const float* u, const float2* K2, const float* D,
                                float2* y, int rows, int H, int L, St st,
                                cudaStream_t s);

// Recurrent mode over L steps from the state x (in/out), one warp per
// (batch row, channel); N <= 256.
cudaError_t launch_recurrent(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                             const float2* C, const float* dt, const float* D, const float* u,
                             int batch, int H, int N, int r, int L, float2* x, float2* y,
                             St st, cudaStream_t s);
// The bordered branch (channels with an exactly zero d_j = 1 - (Delta/2) lambda_j):
// launched after launch_recurrent's / launch_ctilde's own kernel, which leave
// those channels to it; one warp per sequence, N <= 256.
cudaError_t launch_recurrent_bordered(int r, const float2* Lam, const float2* P, const float2* Q,
                                      const float2* B, const float2* C, const float* dt, const float* D,
                                      const float* u, int batch, int H, int N, int L, float2* x, float2* y,
                                      St st, cudaStream_t s);
cudaError_t launch_ctilde_bordered(int r, const float2* Lam, const float2* P, const float2* Q,
                                   const float* dt, const float2* C, int H, int N, int M, float2* Ct,
                                   St st, cudaStream_t s);
// C~ = (I - Abar^M)^* C, one warp per channel; N <= 256.
cudaError_t launch_ctilde(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                          const float2* C, int H, int N, int r, int M, float2* Ct, St st,
                          cudaStream_t s);

// Real-output convolution y = Re(K) * u + D u (real y), two batch rows per
// complex transform; K2 from the spectrum launchers with realk = true.
cudaError_t launch_conv_real_rows(int logn, const float* u, const float2* K2, const float* D, float* y,
                                  int batch, int H, int L, St st, cudaStream_t s, bool pdl = false);
cudaError_t launch_conv_real_cluster(int logn, const float* u, const float2* K2, const float* D,
                                     float* y, int batch, int H, int L, St st,
                                     cudaStream_t s);

}  // namespace s4impl
