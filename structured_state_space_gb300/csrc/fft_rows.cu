// Row FFT kernels whose rows fit one CTA's shared memory (length <= 16384):
//   ifft_kernel      K = first L of (1/M) iFFT_M(Khat)             (kernel generation)
//   spectrum_kernel  K2 = FFT_{2M}(K zero-padded to 2M)            (kernel spectrum)
//   conv_kernel      y = first L of iFFT_{2M}(FFT_{2M}(u) * K2) + D u (fused convolution)
//
// "Recurrent, LSTM, and structured state-space models": filter mode returns
// the first L coefficients of the inverse radix-two transform of the root
// values; "Roots-of-unity orthogonality and radix-two FFT cost": a product of
// two length-n polynomials by zero-padding to a radix-two length >= 2n - 1.
// Here both factors have length L <= M and the transforms have length 2M.
#include "s4_internal.h"
#include "s4_plan.cuh"

namespace s4dev {

// ----------------------------------------------------------------------------
// Rows of length <= 16: one thread per row, the whole transform in registers.
// ----------------------------------------------------------------------------
template <int LOGN>
__global__ void __launch_bounds__(128) ifft_small_kernel(const float2* __restrict__ Khat,
                                                         float2* __restrict__ K, int H, int L,
                                                         const unsigned* __restrict__ status) {
  constexpr int n = 1 << LOGN;
  const int h = blockIdx.x * 128 + threadIdx.x;
  if (h >= H) return;
  const bool zero = *((volatile const unsigned*)status) != 0u;
  float2 a[n];
#pragma unroll
  for (int q = 0; q < n; ++q) a[q] = Khat[(size_t)h * n + q];
  dft<n, true>(a);
  const float sc = 1.f / n;
#pragma unroll
  for (int q = 0; q < n; ++q)
    if (q < L) K[(size_t)h * L + q] = zero ? make_float2(0.f, 0.f) : cscale(a[q], sc);
}

template <int LOGN>
__global__ void __launch_bounds__(128) spectrum_small_kernel(const float2* __restrict__ K,
                                                             float2* __restrict__ K2, int H, int L,
                                                             unsigned* __restrict__ status) {
  constexpr int n = 1 << LOGN;  // n = 2M >= 2
  const int h = blockIdx.x * 128 + threadIdx.x;
  if (h >= H) return;
  float2 a[n];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) a[q] = q < L ? K[(size_t)h * L + q] : make_float2(0.f, 0.f);
  dft<n, false, true>(a);
  bool fin = true;
#pragma unroll
  for (int q = 0; q < n; ++q) {
    fin = fin && cfinite(a[q]);
    K2[(size_t)h * n + q] = a[q];
  }
  if (!fin) atomicOr(status, ST_NONFINITE);
}

template <int LOGN>
__global__ void __launch_bounds__(128) conv_small_kernel(const float* __restrict__ u,
                                                         const float2* __restrict__ K2,
                                                         const float* __restrict__ D,
                                                         float2* __restrict__ y, int rows, int H,
                                                         int L, const unsigned* __restrict__ status) {
  constexpr int n = 1 << LOGN;  // n = 2M >= 2
  const int row = blockIdx.x * 128 + threadIdx.x;
  if (row >= rows) return;
  const int h = row % H;
  const bool zero = *((volatile const unsigned*)status) != 0u;
  float uv[n / 2];
  float2 a[n];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    uv[q] = q < L ? u[(size_t)row * L + q] : 0.f;
    a[q] = make_float2(uv[q], 0.f);
  }
  dft<n, false, true>(a);
#pragma unroll
  for (int q = 0; q < n; ++q) a[q] = cmul(a[q], K2[(size_t)h * n + q]);
  dft<n, true, false, true>(a);
  const float sc = 1.f / n, d = D[h];
#pragma unroll
  for (int q = 0; q < n / 2; ++q)
    if (q < L)
      y[(size_t)row * L + q] =
          zero ? make_float2(0.f, 0.f) : make_float2(fmaf(a[q].x, sc, d * uv[q]), a[q].y * sc);
}

// ----------------------------------------------------------------------------
// Rows of length 32 .. 16384: Stockham passes over padded shared memory.
// ----------------------------------------------------------------------------
template <int LOGN>
struct RowCfg {
  static constexpr int n = 1 << LOGN;
  static constexpr int T = row_threads(LOGN);
  static constexpr int ROWS = rows_per_cta(LOGN);
  static constexpr int THREADS = T * ROWS;
  static constexpr int NP = plan_npass(LOGN);
  static constexpr int RA = plan_radix(LOGN, 0, false);       // first forward radix
  static constexpr int RB = plan_radix(LOGN, NP - 1, false);  // last forward radix
  static constexpr int TWF = plan_tw_size(LOGN, false);
  static constexpr int TWI = plan_tw_size(LOGN, true);
  static constexpr int PADN = padded_len(n);
};

// Inverse transform of each channel's root values, first L outputs scaled 1/M.
template <int LOGN>
__global__ void __launch_bounds__(RowCfg<LOGN>::THREADS) ifft_kernel(
    const float2* __restrict__ Khat, float2* __restrict__ K, int H, int L,
    const unsigned* __restrict__ status) {
  using C = RowCfg<LOGN>;
  constexpr int n = C::n, T = C::T, NP = C::NP;
  constexpr int R0 = plan_radix(LOGN, 0, true), RL = plan_radix(LOGN, NP - 1, true);
  constexpr int NB0 = n / R0, PER0 = NB0 / T, NBL = n / RL, PERL = NBL / T;
  extern __shared__ float2 smem[];
  float2* tw = smem;
  float2* data = smem + C::TWI;
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = data + slot * C::PADN;
  fill_plan_twiddles<LOGN, true>(tw, threadIdx.x, C::THREADS);
  const bool zero = *((volatile const unsigned*)status) != 0u;
  __syncthreads();
  const float sc = 1.f / n;
  for (int h0 = blockIdx.x * C::ROWS; h0 < H; h0 += gridDim.x * C::ROWS) {
    const int h = h0 + slot;
    const bool act = h < H;
    {  // inverse pass 0 (P = 1): global -> registers -> shared
      float2 a[PER0][R0];
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
#pragma unroll
        for (int q = 0; q < R0; ++q)
          a[s][q] = act ? Khat[(size_t)h * n + i + q * NB0] : make_float2(0.f, 0.f);
        dft<R0, true>(a[s]);
#pragma unroll
        for (int q = 0; q < R0; ++q) buf[pad(i * R0 + q)] = a[s][q];
      }
      __syncthreads();
    }
    run_passes<LOGN, true, 1, NP - 2, T>(buf, tw, lt);
    {  // last inverse pass (P = n / RL): shared -> registers -> global
      const float2* twl = tw + plan_tw_off(LOGN, NP - 1, true);
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
        float2 a[RL];
#pragma unroll
        for (int q = 0; q < RL; ++q) a[q] = buf[pad(i + q * NBL)];
        float2 w = twl[i];
        w.y = -w.y;
        apply_twiddles<RL>(a, w);
        dft<RL, true>(a);
#pragma unroll
        for (int q = 0; q < RL; ++q) {
          const int t = i + q * NBL;
          if (act && t < L) K[(size_t)h * L + t] = zero ? make_float2(0.f, 0.f) : cscale(a[q], sc);
        }
      }
      __syncthreads();
    }
  }
}

// Spectrum of each channel's kernel zero-padded to n = 2M (natural order).
template <int LOGN>
__global__ void __launch_bounds__(RowCfg<LOGN>::THREADS) spectrum_kernel(
    const float2* __restrict__ K, float2* __restrict__ K2, int H, int L,
    unsigned* __restrict__ status) {
  using C = RowCfg<LOGN>;
  constexpr int n = C::n, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  extern __shared__ float2 smem[];
  float2* tw = smem;
  float2* data = smem + C::TWF;
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = data + slot * C::PADN;
  fill_plan_twiddles<LOGN, false>(tw, threadIdx.x, C::THREADS);
  __syncthreads();
  bool fin = true;
  for (int h0 = blockIdx.x * C::ROWS; h0 < H; h0 += gridDim.x * C::ROWS) {
    const int h = h0 + slot;
    const bool act = h < H;
    {  // forward pass 0 (P = 1), upper half of the input is the zero padding
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
        float2 a[RA];
#pragma unroll
        for (int q = 0; q < RA / 2; ++q) {
          const int t = i + q * NB0;
          a[q] = (act && t < L) ? K[(size_t)h * L + t] : make_float2(0.f, 0.f);
        }
        dft<RA, false, true>(a);
#pragma unroll
        for (int q = 0; q < RA; ++q) buf[pad(i * RA + q)] = a[q];
      }
      __syncthreads();
    }
    run_passes<LOGN, false, 1, NP - 2, T>(buf, tw, lt);
    {  // last forward pass: shared -> registers -> global
      const float2* twl = tw + plan_tw_off(LOGN, NP - 1, false);
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
        float2 a[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) a[q] = buf[pad(i + q * NBL)];
        apply_twiddles<RB>(a, twl[i]);
        dft<RB, false>(a);
        if (act) {
#pragma unroll
          for (int q = 0; q < RB; ++q) {
            fin = fin && cfinite(a[q]);
            K2[(size_t)h * n + i + q * NBL] = a[q];
          }
        }
      }
      __syncthreads();
    }
  }
  if (!fin) atomicOr(status, ST_NONFINITE);
}

// Fused causal convolution of real rows u[row] (row = b H + h) with the
// channel spectrum K2[h]: pad -> FFT -> product -> iFFT -> first L -> + D u.
template <int LOGN>
__global__ void __launch_bounds__(RowCfg<LOGN>::THREADS) conv_kernel(
    const float* __restrict__ u, const float2* __restrict__ K2, const float* __restrict__ D,
    float2* __restrict__ y, int rows, int H, int L, const unsigned* __restrict__ status) {
  using C = RowCfg<LOGN>;
  constexpr int n = C::n, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  extern __shared__ float2 smem[];
  float2* twf = smem;
  float2* twi = smem + C::TWF;
  float2* data = twi + C::TWI;
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = data + slot * C::PADN;
  fill_plan_twiddles<LOGN, false>(twf, threadIdx.x, C::THREADS);
  fill_plan_twiddles<LOGN, true>(twi, threadIdx.x, C::THREADS);
  const bool zero = *((volatile const unsigned*)status) != 0u;
  __syncthreads();
  const float sc = 1.f / n;
  for (int r0 = blockIdx.x * C::ROWS; r0 < rows; r0 += gridDim.x * C::ROWS) {
    const int row = r0 + slot;
    const bool act = row < rows;
    const int h = act ? row % H : 0;
    const float d = act ? D[h] : 0.f;
    float uv[PER0][RA / 2];
    {  // forward pass 0: u (real, zero-padded) -> registers -> shared
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
        float2 a[RA];
#pragma unroll
        for (int q = 0; q < RA / 2; ++q) {
          const int t = i + q * NB0;
          uv[s][q] = (act && t < L) ? u[(size_t)row * L + t] : 0.f;
          a[q] = make_float2(uv[s][q], 0.f);
        }
        dft<RA, false, true>(a);
#pragma unroll
        for (int q = 0; q < RA; ++q) buf[pad(i * RA + q)] = a[q];
      }
      __syncthreads();
    }
    run_passes<LOGN, false, 1, NP - 2, T>(buf, twf, lt);
    {  // last forward pass, product with K2, first inverse pass: all in registers
      const float2* twl = twf + plan_tw_off(LOGN, NP - 1, false);
      float2 a[PERL][RB];
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
        float2 kv[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) kv[q] = K2[(size_t)h * n + i + q * NBL];
#pragma unroll
        for (int q = 0; q < RB; ++q) a[s][q] = buf[pad(i + q * NBL)];
        apply_twiddles<RB>(a[s], twl[i]);
        dft<RB, false>(a[s]);
#pragma unroll
        for (int q = 0; q < RB; ++q) a[s][q] = cmul(a[s][q], kv[q]);
        dft<RB, true>(a[s]);
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
#pragma unroll
        for (int q = 0; q < RB; ++q) buf[pad(i * RB + q)] = a[s][q];
      }
      __syncthreads();
    }
    run_passes<LOGN, true, 1, NP - 2, T>(buf, twi, lt);
    {  // last inverse pass: shared -> registers -> first L outputs + D u
      const float2* twl = twi + plan_tw_off(LOGN, NP - 1, true);
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
        float2 a[RA];
#pragma unroll
        for (int q = 0; q < RA; ++q) a[q] = buf[pad(i + q * NB0)];
        float2 w = twl[i];
        w.y = -w.y;
        apply_twiddles<RA>(a, w);
        dft<RA, true, false, true>(a);
#pragma unroll
        for (int q = 0; q < RA / 2; ++q) {
          const int t = i + q * NB0;
          if (act && t < L)
            y[(size_t)row * L + t] = zero ? make_float2(0.f, 0.f)
                                          : make_float2(fmaf(a[q].x, sc, d * uv[s][q]), a[q].y * sc);
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace s4dev

// ----------------------------------------------------------------------------
// Host launchers
// ----------------------------------------------------------------------------
namespace s4impl {
using namespace s4dev;

template <typename KernelT>
static cudaError_t prepare(KernelT k, size_t smem) {
  if (smem > 48 * 1024)
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return cudaSuccess;
}

template <typename KernelT>
static int grid_for(KernelT k, int threads, size_t smem, int ctas_needed) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int cap = per_sm * num_sms();
  return ctas_needed < cap ? ctas_needed : cap;
}

template <int LOGN>
static cudaError_t ifft_launch(const float2* Khat, float2* K, int H, int L, const unsigned* st,
                               cudaStream_t s) {
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("ifft", s);
    ifft_small_kernel<LOGN><<<(H + 127) / 128, 128, 0, s>>>(Khat, K, H, L, st);
  } else {
    using C = RowCfg<LOGN>;
    const size_t smem = sizeof(float2) * (C::TWI + (size_t)C::ROWS * C::PADN);
    auto k = ifft_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (H + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("ifft", s);
    k<<<grid, C::THREADS, smem, s>>>(Khat, K, H, L, st);
  }
  return cudaGetLastError();
}

template <int LOGN>
static cudaError_t spectrum_launch(const float2* K, float2* K2, int H, int L, unsigned* st,
                                   cudaStream_t s) {
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("spectrum", s);
    spectrum_small_kernel<LOGN><<<(H + 127) / 128, 128, 0, s>>>(K, K2, H, L, st);
  } else {
    using C = RowCfg<LOGN>;
    const size_t smem = sizeof(float2) * (C::TWF + (size_t)C::ROWS * C::PADN);
    auto k = spectrum_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (H + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("spectrum", s);
    k<<<grid, C::THREADS, smem, s>>>(K, K2, H, L, st);
  }
  return cudaGetLastError();
}

template <int LOGN>
static cudaError_t conv_launch(const float* u, const float2* K2, const float* D, float2* y, int rows,
                               int H, int L, const unsigned* st, cudaStream_t s) {
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("conv", s);
    conv_small_kernel<LOGN><<<(rows + 127) / 128, 128, 0, s>>>(u, K2, D, y, rows, H, L, st);
  } else {
    using C = RowCfg<LOGN>;
    const size_t smem = sizeof(float2) * (C::TWF + C::TWI + (size_t)C::ROWS * C::PADN);
    auto k = conv_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (rows + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("conv", s);
    k<<<grid, C::THREADS, smem, s>>>(u, K2, D, y, rows, H, L, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_ifft_rows(int logM, const float2* Khat, float2* K, int H, int L,
                             const unsigned* st, cudaStream_t s) {
  switch (logM) {
#define S4_CASE(X) \
  case X:          \
    return ifft_launch<X>(Khat, K, H, L, st, s);
    S4_CASE(0) S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13) S4_CASE(14)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_spectrum_rows(int logn, const float2* K, float2* K2, int H, int L, unsigned* st,
                                 cudaStream_t s) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return spectrum_launch<X>(K, K2, H, L, st, s);
    S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13) S4_CASE(14)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_conv_rows(int logn, const float* u, const float2* K2, const float* D, float2* y,
                             int rows, int H, int L, const unsigned* st, cudaStream_t s) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return conv_launch<X>(u, K2, D, y, rows, H, L, st, s);
    S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13) S4_CASE(14)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
