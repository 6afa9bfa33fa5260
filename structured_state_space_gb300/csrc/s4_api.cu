// C ABI of libs4 (declared in include/s4.h): argument checks, workspace
// layout, the order of kernel launches on the caller's stream, the device
// status word and optional launch timing.
#include <limits.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "s4.h"
#include "s4_dev.cuh"
#include "s4_internal.h"

// Build-time tuning: on long rows with L = M, form only the odd half of the
// kernel spectrum (1) or all of it (0).
#ifndef S4_HALF_SPECTRUM
#define S4_HALF_SPECTRUM 1
#endif

namespace {

constexpr int kMaxL = 65536;
constexpr int kMaxN = 65536;
constexpr int kMaxR = 4;

int ilog2_ceil(int v) {
  int lg = 0;
  while ((1 << lg) < v) ++lg;
  return lg;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

// Workspace: [status word | far-field constants of the root values (H
// kFarChannel) | root values (H M) | kernel spectra (H 2M) | long-row convolution
// scratch (two rows of 2M points per pair of batch rows, only when 2M >= 2^14)].
// `gen_total` is what kernel generation alone needs.
struct Layout {
  size_t mom, khat, k2, fs, gen_total, total;
};

Layout layout_for(int H, int L, int batch) {
  const size_t M = (size_t)1 << ilog2_ceil(L);
  Layout l;
  l.mom = 256;
  l.khat = l.mom + round256(sizeof(float2) * (size_t)s4impl::kFarChannel * (size_t)H);
  l.k2 = l.khat + round256(sizeof(float2) * M * (size_t)H);
  l.fs = l.k2 + round256(sizeof(float2) * 2 * M * (size_t)H);
  l.gen_total = l.fs;
  l.total = l.fs + round256(s4impl::fs_scratch_bytes(ilog2_ceil(L) + 1, batch, H));
  return l;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool sizes_ok(int H, int N, int r, int L, int batch) {
  if (H < 1 || N < 1 || N > kMaxN || r < 1 || r > kMaxR || L < 1 || L > kMaxL || batch < 1)
    return false;
  if ((long long)batch * H > INT_MAX) return false;
  if ((long long)H * N > INT_MAX / kMaxR) return false;
  return true;
}

// batch = 0: kernel generation only (no convolution scratch)
s4_status check_ws(const void* ws, size_t ws_bytes, int H, int L, int batch) {
  if (ws == nullptr || !aligned(ws, 256)) return S4_ERR_WORKSPACE;
  const Layout l = layout_for(H, L, batch > 0 ? batch : 1);
  if (ws_bytes < (batch > 0 ? l.total : l.gen_total)) return S4_ERR_WORKSPACE;
  return S4_OK;
}

s4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? S4_OK : S4_ERR_CUDA; }

// The status block at the start of the workspace (see s4impl::St).
s4impl::St status_of(void* ws, unsigned gen) { return s4impl::St{static_cast<unsigned*>(ws), gen}; }
constexpr size_t kStatusBlockBytes = 3 * sizeof(unsigned);

// Generations of calls: 1, 2, ... (0 marks a status block reset by a memset).
unsigned next_generation() {
  static std::atomic<unsigned> g_gen{0};
  unsigned g;
  do {
    g = g_gen.fetch_add(1u) + 1u;
  } while (g == 0u);
  return g;
}

// The status of a call on `s`: a fresh generation, with no reset of the block
// and the call's first kernel chained to the previous kernel (`chain`) -- unless
// `s` is being captured into a graph.  A captured call would replay its
// generation every time the graph runs, so flags a replay sets would read as
// current in the next replay; captured calls therefore reset the block with a
// memset (generation 0) each time they run, and their first kernel is launched
// normally.  Returns false if the memset cannot be enqueued.
bool call_status(void* ws, cudaStream_t s, s4impl::St* st, bool* chain) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return false;
  if (cs != cudaStreamCaptureStatusNone) {
    *st = status_of(ws, 0u);
    *chain = false;
    return cudaMemsetAsync(ws, 0, kStatusBlockBytes, s) == cudaSuccess;
  }
  *st = status_of(ws, next_generation());
  *chain = true;
  return true;
}

// Root values in the blocked order of 2^logC (logC < 0: the order the inverse
// transform of s4_kernel_gen reads, khat_cluster_log).
cudaError_t cauchy_impl(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const s4_c32* B,
                        const s4_c32* Ct, const float* dt, int H, int N, int r, int L, void* ws,
                        s4impl::St st, bool pdl, cudaStream_t s, int logC = -1) {
  using namespace s4impl;
  const int logM = ilog2_ceil(L);
  char* w = static_cast<char*>(ws);
  return launch_cauchy(reinterpret_cast<const float2*>(Lambda), reinterpret_cast<const float2*>(P),
                       reinterpret_cast<const float2*>(Q), reinterpret_cast<const float2*>(B),
                       reinterpret_cast<const float2*>(Ct), dt,
                       reinterpret_cast<float2*>(w + layout_for(H, L, 1).khat),
                       reinterpret_cast<float2*>(w + layout_for(H, L, 1).mom), H, N, r, 1 << logM,
                       logC >= 0 ? logC : khat_cluster_log(logM), st, s, pdl);
}

s4_status gen_impl(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const s4_c32* B,
                   const s4_c32* Ct, const float* dt, int H, int N, int r, int L, s4_c32* K,
                   void* ws, s4impl::St st, bool pdl, cudaStream_t s) {
  using namespace s4impl;
  const int logM = ilog2_ceil(L);
  const Layout lay = layout_for(H, L, 1);
  char* w = static_cast<char*>(ws);
  float2* khat = reinterpret_cast<float2*>(w + lay.khat);
  cudaError_t e = cauchy_impl(Lambda, P, Q, B, Ct, dt, H, N, r, L, ws, st, pdl, s);
  if (e == cudaSuccess)
    e = logM <= kMaxLogRowCta
            ? launch_ifft_rows(logM, khat, reinterpret_cast<float2*>(K), H, L, st, s)
            : launch_ifft_cluster(logM, khat, reinterpret_cast<float2*>(K), H, L, st, s);
  return cuda_status(e);
}

s4_status conv_impl(const float* u, const s4_c32* K, const float* D, int batch, int H, int L,
                    s4_c32* y, void* ws, s4impl::St st, bool chain, cudaStream_t s) {
  using namespace s4impl;
  const int logn = ilog2_ceil(L) + 1;
  const Layout lay = layout_for(H, L, batch);
  char* w = static_cast<char*>(ws);
  float2* k2 = reinterpret_cast<float2*>(w + lay.k2);
  const float2* Kf = reinterpret_cast<const float2*>(K);
  float2* yf = reinterpret_cast<float2*>(y);
  cudaError_t e;
  if (logn <= kMaxLogConvRow) {
    e = launch_spectrum_rows(logn, Kf, k2, H, L, st, s, false, /*pdl=*/chain);
    // programmatic dependent: the convolution transforms its input rows while
    // the spectrum kernel finishes, and waits for it before reading K2
    if (e == cudaSuccess) e = launch_conv_rows(logn, u, k2, D, yf, batch, H, L, st, s, /*pdl=*/true);
  } else {
    // long rows: the four-step spectrum (column order; its scratch is the start
    // of the convolution's, free again before the convolution writes it)
    float2* fs = reinterpret_cast<float2*>(w + lay.fs);
    e = launch_spectrum_fourstep(logn, Kf, k2, H, L, fs, st, s);
    if (e == cudaSuccess)
      e = launch_conv_fourstep(logn, u, k2, fs_log_radix(logn), kFsSpecScale, D, yf, batch, H, L, fs, st, s);
  }
  return cuda_status(e);
}

// ---- launch timing --------------------------------------------------------------
struct TimingRec {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_tmu;
bool g_timing = false;
std::vector<TimingRec> g_recs;
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_pool;
size_t g_used = 0;

}  // namespace

namespace s4impl {

namespace {
std::atomic<int> g_wait_limit{s4dev::kMbarWaitLimit};
}  // namespace

int wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) v = 148;
    cache[dev] = v;
  }
  return cache[dev];
}

TimedLaunch::TimedLaunch(const char* name, cudaStream_t s) : slot_(-1), s_(s) {
  std::lock_guard<std::mutex> lk(g_tmu);
  if (!g_timing) return;
  if (g_used == g_pool.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return;
    }
    g_pool.push_back({a, b});
  }
  const auto pr = g_pool[g_used];
  slot_ = (int)g_recs.size();
  g_recs.push_back({name, pr.first, pr.second});
  ++g_used;
  record(pr.first, s);
}

// Inside a stream capture the events become event-record nodes of the graph.
void TimedLaunch::record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

TimedLaunch::~TimedLaunch() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  record(g_recs[slot_].stop, s_);
}

// FP32 issue-rate probe (a measurement aid): 8 independent FMA chains per
// thread, the iteration loop unrolled by 8 so that loop control is ~5 % of
// the issued instructions.
__global__ void __launch_bounds__(256) fp32_probe_kernel(float* __restrict__ out, int iters8) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = (float)(t & 255) * 1e-6f + (float)k * 1e-3f;
  const float m = 0.99999988f, c = 1e-7f;  // a -> c / (1 - m): bounded, never denormal
  for (int i = 0; i < iters8; ++i) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = fmaf(a[k], m, c);
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += a[k];
  out[t] = sum;
}

}  // namespace s4impl

extern "C" {

s4_status s4_fp32_probe(float* out, int blocks, int iters, void* stream) {
  if (!out || blocks < 1 || iters < 1) return S4_ERR_INVALID_ARG;
  s4impl::fp32_probe_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(out, (iters + 7) / 8);
  return cudaGetLastError() == cudaSuccess ? S4_OK : S4_ERR_CUDA;
}

long long s4_bounds_violations(void) {
#ifdef S4_BOUNDS_CHECK
  if (cudaDeviceSynchronize() != cudaSuccess) return -2;
  const unsigned long long c[] = {s4impl::oob_rows(), s4impl::oob_cluster(), s4impl::oob_fourstep(),
                                  s4impl::oob_cauchy(), s4impl::oob_recurrent(), s4impl::oob_bordered()};
  unsigned long long t = 0;
  for (unsigned long long v : c) {
    if (v == ~0ull) return -2;
    t += v;
  }
  return (long long)t;
#else
  return -1;
#endif
}

s4_status s4_set_wait_limit(int polls) {
  s4impl::g_wait_limit.store(polls >= 0 ? polls : s4dev::kMbarWaitLimit, std::memory_order_relaxed);
  return S4_OK;
}

size_t s4_workspace_bytes(int H, int N, int r, int L, int batch) {
  if (!sizes_ok(H, N, r, L, batch)) return 0;
  return layout_for(H, L, batch).total;
}

s4_status s4_kernel_gen(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const s4_c32* B,
                        const s4_c32* Ctilde, const float* dt, int H, int N, int r, int L,
                        s4_c32* K, void* ws, size_t ws_bytes, void* stream) {
  if (!Lambda || !P || !Q || !B || !Ctilde || !dt || !K) return S4_ERR_INVALID_ARG;
  if (!sizes_ok(H, N, r, L, 1)) return S4_ERR_INVALID_ARG;
  if (!aligned(Lambda, 8) || !aligned(P, 8) || !aligned(Q, 8) || !aligned(B, 8) ||
      !aligned(Ctilde, 8) || !aligned(dt, 4) || !aligned(K, 16))
    return S4_ERR_INVALID_ARG;
  const s4_status wst = check_ws(ws, ws_bytes, H, L, 0);
  if (wst != S4_OK) return wst;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  s4impl::St st;
  bool chain;
  if (!call_status(ws, s, &st, &chain)) return S4_ERR_CUDA;
  return gen_impl(Lambda, P, Q, B, Ctilde, dt, H, N, r, L, K, ws, st, chain, s);
}

s4_status s4_conv_fwd(const float* u, const s4_c32* K, const float* D, int batch, int H, int L,
                      s4_c32* y, void* ws, size_t ws_bytes, void* stream) {
  if (!u || !K || !D || !y) return S4_ERR_INVALID_ARG;
  if (!sizes_ok(H, 1, 1, L, batch)) return S4_ERR_INVALID_ARG;
  if (!aligned(u, 16) || !aligned(K, 16) || !aligned(D, 4) || !aligned(y, 16))
    return S4_ERR_INVALID_ARG;
  const s4_status wst = check_ws(ws, ws_bytes, H, L, batch);
  if (wst != S4_OK) return wst;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  s4impl::St st;
  bool chain;
  if (!call_status(ws, s, &st, &chain)) return S4_ERR_CUDA;
  return conv_impl(u, K, D, batch, H, L, y, ws, st, chain, s);
}

s4_status s4_conv_fwd_real(const float* u, const s4_c32* K, const float* D, int batch, int H, int L,
                           float* y, void* ws, size_t ws_bytes, void* stream) {
  if (!u || !K || !D || !y) return S4_ERR_INVALID_ARG;
  if (!sizes_ok(H, 1, 1, L, batch)) return S4_ERR_INVALID_ARG;
  if (!aligned(u, 16) || !aligned(K, 16) || !aligned(D, 4) || !aligned(y, 16)) return S4_ERR_INVALID_ARG;
  const s4_status wst = check_ws(ws, ws_bytes, H, L, 0);
  if (wst != S4_OK) return wst;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  using namespace s4impl;
  const int logn = ilog2_ceil(L) + 1;
  char* w = static_cast<char*>(ws);
  St st;
  bool chain;
  if (!call_status(ws, s, &st, &chain)) return S4_ERR_CUDA;
  float2* k2 = reinterpret_cast<float2*>(w + layout_for(H, L, 1).k2);
  const float2* Kf = reinterpret_cast<const float2*>(K);
  cudaError_t e;
  if (logn <= kMaxLogConvRow) {
    e = launch_spectrum_rows(logn, Kf, k2, H, L, st, s, /*realk=*/true, /*pdl=*/chain);
    if (e == cudaSuccess) e = launch_conv_real_rows(logn, u, k2, D, y, batch, H, L, st, s, /*pdl=*/true);
  } else {
    e = launch_spectrum_cluster(logn, Kf, k2, H, L, st, s, /*realk=*/true);
    if (e == cudaSuccess) e = launch_conv_real_cluster(logn, u, k2, D, y, batch, H, L, st, s);
  }
  return cuda_status(e);
}

s4_status s4_layer_fwd(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const s4_c32* B,
                       const s4_c32* Ctilde, const float* dt, const float* D, const float* u,
                       int batch, int H, int N, int r, int L, s4_c32* K, s4_c32* y, void* ws,
                       size_t ws_bytes, void* stream) {
  if (!Lambda || !P || !Q || !B || !Ctilde || !dt || !D || !u || !K || !y)
    return S4_ERR_INVALID_ARG;
  if (!sizes_ok(H, N, r, L, batch)) return S4_ERR_INVALID_ARG;
  if (!aligned(Lambda, 8) || !aligned(P, 8) || !aligned(Q, 8) || !aligned(B, 8) ||
      !aligned(Ctilde, 8) || !aligned(dt, 4) || !aligned(D, 4) || !aligned(u, 16) ||
      !aligned(K, 16) || !aligned(y, 16))
    return S4_ERR_INVALID_ARG;
  const s4_status wst = check_ws(ws, ws_bytes, H, L, batch);
  if (wst != S4_OK) return wst;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // No reset of the status block: this call's flags carry a fresh generation,
  // so the call is kernels only and its first kernel (root values) can be a
  // programmatic dependent of whatever kernel precedes it on the stream.
  s4impl::St st;
  bool chain;
  if (!call_status(ws, s, &st, &chain)) return S4_ERR_CUDA;
  const int logM = ilog2_ceil(L);
  if (s4impl::kspec_supported(logM) && logM + 1 <= s4impl::kMaxLogConvRow) {
    // root values -> (K, kernel spectrum) in one launch -> convolution
    const Layout lay = layout_for(H, L, batch);
    char* w = static_cast<char*>(ws);
    float2* khat = reinterpret_cast<float2*>(w + lay.khat);
    float2* k2 = reinterpret_cast<float2*>(w + lay.k2);
    cudaError_t e = cauchy_impl(Lambda, P, Q, B, Ctilde, dt, H, N, r, L, ws, st, chain, s);
    if (e == cudaSuccess)
      e = s4impl::launch_kspec_rows(logM, khat, reinterpret_cast<float2*>(K), k2, H, L, st, s);
    if (e == cudaSuccess)
      e = s4impl::launch_conv_rows(logM + 1, u, k2, D, reinterpret_cast<float2*>(y), batch, H, L, st, s,
                                   /*pdl=*/true);
    return cuda_status(e);
  }
  if (logM + 1 >= s4impl::kMinLogFourStep) {
    // long rows: root values in column order -> column inverse transforms -> K
    // (out) and the across-column step of its spectrum -> column spectra ->
    // four-step convolution.  The spectrum's scratch (H M + 2 H M values) lies
    // in the convolution's, which is written only after it is consumed; the root
    // values stay in their own region until the convolution has read them.
    const Layout lay = layout_for(H, L, batch);
    char* w = static_cast<char*>(ws);
    float2* khat = reinterpret_cast<float2*>(w + lay.khat);
    float2* k2 = reinterpret_cast<float2*>(w + lay.k2);
    float2* fs = reinterpret_cast<float2*>(w + lay.fs);
    if (S4_HALF_SPECTRUM && L == (1 << logM)) {
      // L = M: the spectrum's even bins are the root values; only its odd bins are
      // formed (into the spectrum's region), and the convolution reads both halves
      const int logC = s4impl::fs_log_radix(logM + 1) - 1;
      cudaError_t e = cauchy_impl(Lambda, P, Q, B, Ctilde, dt, H, N, r, L, ws, st, chain, s, logC);
      if (e == cudaSuccess)
        e = s4impl::launch_kspec_fourstep_half(logM, khat, reinterpret_cast<float2*>(K), k2, H, L, fs,
                                               fs + ((size_t)H << logM), st, s);
      if (e == cudaSuccess)
        e = s4impl::launch_conv_fourstep(logM + 1, u, khat, logC, 1.f / (float)(2 << logM), D,
                                         reinterpret_cast<float2*>(y), batch, H, L, fs, st, s, k2,
                                         s4impl::kFsSpecScale);
      return cuda_status(e);
    }
    cudaError_t e = cauchy_impl(Lambda, P, Q, B, Ctilde, dt, H, N, r, L, ws, st, chain, s, /*logC=*/4);
    if (e == cudaSuccess)
      e = s4impl::launch_kspec_fourstep(logM, khat, reinterpret_cast<float2*>(K), k2, H, L, fs,
                                        fs + ((size_t)H << logM), st, s);
    if (e == cudaSuccess)
      e = s4impl::launch_conv_fourstep(logM + 1, u, k2, s4impl::fs_log_radix(logM + 1), s4impl::kFsSpecScale, D,
                                       reinterpret_cast<float2*>(y), batch, H, L, fs, st, s);
    return cuda_status(e);
  }
  const s4_status g = gen_impl(Lambda, P, Q, B, Ctilde, dt, H, N, r, L, K, ws, st, chain, s);
  if (g != S4_OK) return g;
  return conv_impl(u, K, D, batch, H, L, y, ws, st, /*chain=*/true, s);
}

s4_status s4_ctilde(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const float* dt,
                    const s4_c32* C, int H, int N, int r, int L, s4_c32* Ctilde, void* ws,
                    size_t ws_bytes, void* stream) {
  if (!Lambda || !P || !Q || !dt || !C || !Ctilde) return S4_ERR_INVALID_ARG;
  if (!sizes_ok(H, N, r, L, 1) || N > 256) return S4_ERR_INVALID_ARG;
  if (!aligned(Lambda, 8) || !aligned(P, 8) || !aligned(Q, 8) || !aligned(C, 8) || !aligned(Ctilde, 8) ||
      !aligned(dt, 4))
    return S4_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < 256) return S4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kStatusBlockBytes, s) != cudaSuccess) return S4_ERR_CUDA;
  return cuda_status(s4impl::launch_ctilde(
      reinterpret_cast<const float2*>(Lambda), reinterpret_cast<const float2*>(P),
      reinterpret_cast<const float2*>(Q), dt, reinterpret_cast<const float2*>(C), H, N, r,
      1 << ilog2_ceil(L), reinterpret_cast<float2*>(Ctilde), status_of(ws, 0u), s));
}

s4_status s4_recurrent_fwd(const s4_c32* Lambda, const s4_c32* P, const s4_c32* Q, const s4_c32* B,
                           const s4_c32* C, const float* dt, const float* D, const float* u,
                           int batch, int H, int N, int r, int L, s4_c32* x, s4_c32* y, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!Lambda || !P || !Q || !B || !C || !dt || !D || !u || !x || !y) return S4_ERR_INVALID_ARG;
  if (H < 1 || N < 1 || N > 256 || r < 1 || r > kMaxR || L < 1 || batch < 1) return S4_ERR_INVALID_ARG;
  if ((long long)batch * H > INT_MAX / 32) return S4_ERR_INVALID_ARG;
  if (!aligned(Lambda, 8) || !aligned(P, 8) || !aligned(Q, 8) || !aligned(B, 8) || !aligned(C, 8) ||
      !aligned(x, 8) || !aligned(y, 8) || !aligned(dt, 4) || !aligned(D, 4) || !aligned(u, 4))
    return S4_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < 256) return S4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kStatusBlockBytes, s) != cudaSuccess) return S4_ERR_CUDA;
  return cuda_status(s4impl::launch_recurrent(
      reinterpret_cast<const float2*>(Lambda), reinterpret_cast<const float2*>(P),
      reinterpret_cast<const float2*>(Q), reinterpret_cast<const float2*>(B),
      reinterpret_cast<const float2*>(C), dt, D, u, batch, H, N, r, L, reinterpret_cast<float2*>(x),
      reinterpret_cast<float2*>(y), status_of(ws, 0u), s));
}

s4_status s4_get_status(const void* ws, void* stream) {
  if (ws == nullptr) return S4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return S4_ERR_CUDA;
  unsigned blk[3] = {0u, 0u, 0u};  // flags, their generation, the last call's generation
  if (cudaMemcpy(blk, ws, sizeof(blk), cudaMemcpyDeviceToHost) != cudaSuccess) return S4_ERR_CUDA;
  const unsigned word = blk[1] == blk[2] ? blk[0] : 0u;  // older flags are stale
  if (word & s4dev::ST_STALL) return S4_ERR_TIMEOUT;
  if (word & s4dev::ST_BAD_STEP) return S4_ERR_INVALID_STEP;
  if (word & s4dev::ST_RES_DIAG) return S4_ERR_RESONANT_DIAGONAL;
  if (word & s4dev::ST_RES_CORR) return S4_ERR_RESONANT_CORRECTION;
  if (word & s4dev::ST_SINGULAR) return S4_ERR_SINGULAR_BILINEAR;
  if (word & s4dev::ST_NONFINITE) return S4_ERR_NONFINITE;
  return S4_OK;
}

const char* s4_status_str(s4_status st) {
  switch (st) {
    case S4_OK: return "ok";
    case S4_ERR_INVALID_ARG: return "invalid argument";
    case S4_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case S4_ERR_RESONANT_DIAGONAL: return "resonant-diagonal";
    case S4_ERR_RESONANT_CORRECTION: return "resonant-correction";
    case S4_ERR_NONFINITE: return "non-finite value";
    case S4_ERR_INVALID_STEP: return "step size not positive and finite";
    case S4_ERR_CUDA: return "CUDA error";
    case S4_ERR_SINGULAR_BILINEAR: return "singular-bilinear-matrix";
    case S4_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

void s4_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_tmu);
  g_timing = on != 0;
}

void s4_timing_reset(void) {
  std::lock_guard<std::mutex> lk(g_tmu);
  g_recs.clear();
  g_used = 0;
}

int s4_timing_read(const char* name, int* launches, double* total_ms) {
  std::lock_guard<std::mutex> lk(g_tmu);
  int n = 0;
  double ms = 0.0;
  for (const TimingRec& r : g_recs) {
    if (name && strcmp(name, r.name) != 0) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) return -1;
    ms += t;
    ++n;
  }
  if (launches) *launches = n;
  if (total_ms) *total_ms = ms;
  return 0;
}

}  // extern "C"
