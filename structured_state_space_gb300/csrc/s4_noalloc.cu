// s4_conv_fwd_noalloc: the causal convolution for callers that cannot
// allocate device memory.
//
// Who needs it: a host program that owns all device memory through its own
// pool and forbids allocations from libraries it loads (a plugin, an engine
// with a fixed memory budget), or a latency-critical loop where cudaMalloc
// is not acceptable because it can synchronise the device.  Such a caller
// cannot hand s4_conv_fwd a workspace of its own, so this variant keeps its
// scratch -- the status word and the kernel spectrum -- in a fixed array
// compiled into the library.  That array exists on every device that loads
// the library and stays there until the process exits.
//
// The same kernels as s4_conv_fwd run (spectrum, then fused convolution),
// after a memset of the status word and without programmatic dependent launch,
// so the convolution does not overlap the spectrum kernel as it does there.
#include <stdint.h>

#include <mutex>

#include "s4.h"
#include "s4_internal.h"

namespace {

// Scratch: [status word, 256 B | kernel spectra K2 [H][2M] complex64].
static __device__ __align__(256) unsigned char g_noalloc_scratch[S4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array for the current device, looked up
// once per device.  (In host code the array's name is only a host-side
// stand-in; kernels must be given this address.)
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

int log2_ceil(int v) {
  int lg = 0;
  while ((1 << lg) < v) ++lg;
  return lg;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" s4_status s4_conv_fwd_noalloc(const float* u, const s4_c32* K, const float* D, int batch,
                                         int H, int L, s4_c32* y, void* stream) {
  if (!u || !K || !D || !y) return S4_ERR_INVALID_ARG;
  if (H < 1 || L < 1 || L > 65536 || batch < 1 || (long long)batch * H > 0x7fffffffLL)
    return S4_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(K) || !aligned16(y) || ((uintptr_t)D & 3u) != 0)
    return S4_ERR_INVALID_ARG;
  const int logn = log2_ceil(L) + 1;  // transform length 2M
  const size_t need = 256 + sizeof(float2) * ((size_t)1 << logn) * (size_t)H;
  if (need > (size_t)S4_NOALLOC_SCRATCH_BYTES) return S4_ERR_WORKSPACE;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return S4_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const s4impl::St st{static_cast<unsigned*>(base), 0u};
  float2* k2 = reinterpret_cast<float2*>(static_cast<char*>(base) + 256);
  // the status block starts at zero (generation 0); the spectrum is fully overwritten
  if (cudaMemsetAsync(base, 0, 3 * sizeof(unsigned), s) != cudaSuccess) return S4_ERR_CUDA;
  const float2* Kf = reinterpret_cast<const float2*>(K);
  float2* yf = reinterpret_cast<float2*>(y);
  const int rows = batch * H;
  cudaError_t e;
  if (logn <= s4impl::kMaxLogConvRow) {
    e = s4impl::launch_spectrum_rows(logn, Kf, k2, H, L, st, s);
    if (e == cudaSuccess) e = s4impl::launch_conv_rows(logn, u, k2, D, yf, batch, H, L, st, s);
  } else {
    e = s4impl::launch_spectrum_cluster(logn, Kf, k2, H, L, st, s);
    if (e == cudaSuccess) e = s4impl::launch_conv_cluster(logn, u, k2, D, yf, rows, H, L, st, s);
  }
  return e == cudaSuccess ? S4_OK : S4_ERR_CUDA;
}
