// Internal host-side interfaces between the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace s4impl {

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Optional event bracketing of kernel launches (see s4_timing_* in s4.h).
// Construct right before a launch and let it go out of scope right after.
class TimedLaunch {
 public:
  TimedLaunch(const char* name, cudaStream_t s);
  ~TimedLaunch();
  TimedLaunch(const TimedLaunch&) = delete;
  TimedLaunch& operator=(const TimedLaunch&) = delete;

 private:
  int slot_;
  cudaStream_t s_;
};

// Largest row that one CTA transforms in shared memory (log2 of the length).
constexpr int kMaxLogRowCta = 14;

// log2 of the cluster size that splits a row of 2^logn points: rows of up to
// 2^14 points stay in one CTA; 2^15 uses 4 CTAs of 2^13; 2^16 uses 8 of 2^13;
// 2^17 uses 8 of 2^14.  Spectra of split rows are stored in blocked order.
__host__ __device__ constexpr int cluster_log(int logn) {
  return logn <= kMaxLogRowCta ? 0 : (logn == 15 ? 2 : 3);
}

// tan(pi k / M) for every root k, as an fp32 (hi, lo) pair, stored in the
// blocked root order used for Khat (position p -> root (p mod M/C) C + p div M/C).
cudaError_t launch_tau(float2* tau, int M, int logC, cudaStream_t s);

// Root values Khat[h][p] (blocked order) for every channel.
cudaError_t launch_cauchy(const float2* Lambda, const float2* P, const float2* Q, const float2* B,
                          const float2* Ct, const float* dt, const float2* tau, float2* Khat, int H,
                          int N, int r, int M, int logC, unsigned* status, cudaStream_t s);

// Single-CTA row transforms (log sizes up to kMaxLogRowCta).
cudaError_t launch_ifft_rows(int logM, const float2* Khat, float2* K, int H, int L,
                             const unsigned* st, cudaStream_t s);
cudaError_t launch_spectrum_rows(int logn, const float2* K, float2* K2, int H, int L, unsigned* st,
                                 cudaStream_t s);
cudaError_t launch_conv_rows(int logn, const float* u, const float2* K2, const float* D, float2* y,
                             int rows, int H, int L, const unsigned* st, cudaStream_t s);

// Cluster row transforms for longer rows (rows split over C = 2..8 CTAs).
cudaError_t launch_ifft_cluster(int logM, const float2* Khat, float2* K, int H, int L,
                                const unsigned* st, cudaStream_t s);
cudaError_t launch_spectrum_cluster(int logn, const float2* K, float2* K2, int H, int L,
                                    unsigned* st, cudaStream_t s);
cudaError_t launch_conv_cluster(int logn, const float* u, const float2* K2, const float* D,
                                float2* y, int rows, int H, int L, const unsigned* st,
                                cudaStream_t s);

}  // namespace s4impl
