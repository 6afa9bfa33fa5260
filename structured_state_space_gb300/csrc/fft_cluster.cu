// Row FFT kernels for rows longer than one CTA's shared memory holds
// (length 2^15 .. 2^17).  A row of n = C m points is split over a thread-block
// cluster of C CTAs by the four-step factorisation n = C x m:
//   forward:  b_c[i] = w_n^{i c} * sum_q x[i + q m] w_C^{q c}     (cross-CTA, through DSMEM)
//             X[c + C k] = sum_i b_c[i] w_m^{i k}                (local m-point FFT in CTA c)
//   inverse:  g_c[i] = sum_k Y[c + C k] w_m^{-i k}               (local inverse in CTA c)
//             y[i + q m] = (1/n) sum_c g_c[i] w_n^{-i c} w_C^{-q c} (cross-CTA)
// Spectra therefore live in "blocked" order: CTA c owns bins c, c + C, ...
// stored contiguously; the kernel spectrum and the root values of kernel
// generation use the same layout, so no reordering pass is needed.
// Remote shared-memory traffic uses plain DSMEM loads and stores.
#include <cooperative_groups.h>

#include "s4_fft.cuh"
#include "s4_internal.h"

namespace cg = cooperative_groups;

namespace s4dev {

template <int LOGN, bool PAIR = false>
struct ClusterCfg {
  static constexpr int LOGC = s4impl::cluster_log(LOGN);
  static constexpr int C = 1 << LOGC;
  static constexpr int LOGM = LOGN - LOGC;
  static constexpr int n = 1 << LOGN, m = 1 << LOGM;
  // the paired convolution keeps two rows per thread in its inverse passes:
  // one radix-16 butterfly per thread (conv_row_threads) measured 20 % faster
  // than two at 2M = 2^15
  static constexpr int T = PAIR ? conv_row_threads(LOGM) : row_threads(LOGM);
  static constexpr int NP = plan_npass(LOGM);
  static constexpr int MI = m / C;   // cross-step indices owned by one CTA
  static constexpr int PI = MI / T;  // ... per thread
  static constexpr int PADM = padded_len(m);
  static_assert(PI >= 1 && MI % T == 0, "cluster split");
};

// w_n^i for the indices i = c MI + il owned by CTA c.
__device__ __forceinline__ void fill_cross_twiddles(float2* tw1, int c, int MI, int n, int tid, int nth) {
  for (int il = tid; il < MI; il += nth) {
    float s, co;
    sincospif(2.0f * (float)(c * MI + il) / (float)n, &s, &co);
    tw1[il] = make_float2(co, -s);
  }
}

// Forward cross step for one row: x[i + q m] (q < C/2 from `load`, the rest zero
// padding) -> radix-C DFT -> twiddle -> CTA q'.
template <int LOGN, bool PAIR = false, typename LoadF>
__device__ __forceinline__ void cross_forward(cg::cluster_group& cl, float2* buf, const float2* tw1,
                                              int c, int lt, LoadF load) {
  using Cf = ClusterCfg<LOGN, PAIR>;
  constexpr int C = Cf::C, MI = Cf::MI, T = Cf::T, m = Cf::m;
#pragma unroll
  for (int s = 0; s < Cf::PI; ++s) {
    const int il = lt + s * T;
    const int i = c * MI + il;
    float2 x[C];
#pragma unroll
    for (int q = 0; q < C / 2; ++q) x[q] = load(s, q, i + q * m);
    dft<C, false, true>(x);
    apply_twiddles<C>(x, tw1[il]);
#pragma unroll
    for (int q = 0; q < C; ++q) {
      float2* dst = cl.map_shared_rank(buf, q);
      st_chk(dst, pad(i), Cf::PADM, x[q]);
    }
  }
}

// Inverse cross step: gather g_c[i] from every CTA, twiddle, inverse radix-C DFT.
template <int LOGN, bool HALF, bool PAIR = false, typename StoreF>
__device__ __forceinline__ void cross_inverse(cg::cluster_group& cl, float2* buf, const float2* tw1,
                                              int c, int lt, StoreF store) {
  using Cf = ClusterCfg<LOGN, PAIR>;
  constexpr int C = Cf::C, MI = Cf::MI, T = Cf::T, m = Cf::m;
#pragma unroll
  for (int s = 0; s < Cf::PI; ++s) {
    const int il = lt + s * T;
    const int i = c * MI + il;
    float2 x[C];
#pragma unroll
    for (int q = 0; q < C; ++q) {
      const float2* src = cl.map_shared_rank(buf, q);
      x[q] = ld_chk(src, pad(i), Cf::PADM);
    }
    float2 w = tw1[il];
    w.y = -w.y;
    apply_twiddles<C>(x, w);
    dft<C, true, false, HALF>(x);
#pragma unroll
    for (int q = 0; q < (HALF ? C / 2 : C); ++q) store(s, q, i + q * m, x[q]);
  }
}

// Kernel spectrum of n = 2M points per channel, blocked output order.
template <int LOGN>
__global__ void __launch_bounds__(ClusterCfg<LOGN>::T) spectrum_cluster_kernel(
    const float2* __restrict__ K, float2* __restrict__ K2, int H, int L, int realk,
    St status) {
  using Cf = ClusterCfg<LOGN>;
  constexpr int n = Cf::n, m = Cf::m, T = Cf::T, NP = Cf::NP, LOGM = Cf::LOGM;
  constexpr int RB = plan_radix(LOGM, NP - 1, false), NBL = m / RB, PERL = NBL / T;
  using IXL = PassIdx<m, RB, m / RB>;
  using TWL = PassTw<LOGM, NP - 1, false>;
  cg::cluster_group cl = cg::this_cluster();
  const int c = (int)cl.block_rank();
  extern __shared__ float2 smem[];
  float2* tw1 = smem;
  float2* buf = tw1 + Cf::MI;
  float2* const bufs[1] = {buf};
  const int lt = threadIdx.x;
  st_record_gen(status);  // the first kernel of a convolution call (launched normally)
  fill_cross_twiddles(tw1, c, Cf::MI, n, lt, T);
  __syncthreads();
  cl.sync();
  bool fin = true;
  const int ncl = gridDim.x / Cf::C;
  for (int h = blockIdx.x / Cf::C; h < H; h += ncl) {
    cross_forward<LOGN>(cl, buf, tw1, c, lt, [&](int, int, int t) {
      float2 v = (t < L && S4_IN((long long)h * L + t, (long long)H * L)) ? K[(size_t)h * L + t] : make_float2(0.f, 0.f);
      if (realk) v.y = 0.f;
      return v;
    });
    cl.sync();
    passes_rows<LOGM, false, 0, NP - 2, T, 1>(bufs, lt);
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
      float2 a[RB], w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) a[q] = buf[IXL::rd(i, q)];
      TWL::load(w, i);
      TWL::apply(a, w);
      dft<RB, false>(a);
#pragma unroll
      for (int q = 0; q < RB; ++q) {
        fin = fin && cfinite(a[q]);
        st_chk(K2, (long long)h * n + (long long)c * m + i + q * NBL, (long long)H * n, a[q]);
      }
    }
    cl.sync();
  }
  if (!fin) st_flag(status, ST_NONFINITE);
}

// Inverse transform of M = n root values per channel (blocked input order),
// first L outputs scaled by 1/M.
template <int LOGN>
__global__ void __launch_bounds__(ClusterCfg<LOGN>::T) ifft_cluster_kernel(
    const float2* __restrict__ Khat, float2* __restrict__ K, int H, int L,
    St status) {
  using Cf = ClusterCfg<LOGN>;
  constexpr int n = Cf::n, m = Cf::m, T = Cf::T, NP = Cf::NP, LOGM = Cf::LOGM;
  constexpr int R0 = plan_radix(LOGM, 0, true), NB0 = m / R0, PER0 = NB0 / T;
  using IX0 = PassIdx<m, R0, 1>;
  cg::cluster_group cl = cg::this_cluster();
  const int c = (int)cl.block_rank();
  extern __shared__ float2 smem[];
  float2* tw1 = smem;
  float2* buf = tw1 + Cf::MI;
  float2* const bufs[1] = {buf};
  const int lt = threadIdx.x;
  fill_cross_twiddles(tw1, c, Cf::MI, n, lt, T);
  const bool zero = st_bad(status);
  __syncthreads();
  cl.sync();
  const float sc = 1.f / n;
  const int ncl = gridDim.x / Cf::C;
  for (int h = blockIdx.x / Cf::C; h < H; h += ncl) {
#pragma unroll
    for (int s = 0; s < PER0; ++s) {
      const int i = lt + s * T;
      float2 a[R0];
#pragma unroll
      for (int q = 0; q < R0; ++q) a[q] = ld_chk(Khat, (long long)h * n + (long long)c * m + i + q * NB0, (long long)H * n);
      dft<R0, true>(a);
#pragma unroll
      for (int q = 0; q < R0; ++q) buf[IX0::wr(i, q)] = a[q];
    }
    __syncthreads();
    passes_rows<LOGM, true, 1, NP - 1, T, 1>(bufs, lt);
    cl.sync();
    cross_inverse<LOGN, false>(cl, buf, tw1, c, lt, [&](int, int, int t, float2 v) {
      if (t < L) st_chk(K, (long long)h * L + t, (long long)H * L, zero ? make_float2(0.f, 0.f) : cscale(v, sc));
    });
    cl.sync();
  }
}

// Fused causal convolution for rows of n = 2M > 16384 points.  The skip term
// enters as D added to every kernel-spectrum bin (the spectrum of D times the
// unit impulse), so no input value stays live across the transforms.
template <int LOGN>
__global__ void __launch_bounds__(ClusterCfg<LOGN>::T) conv_cluster_kernel(
    const float* __restrict__ u, const float2* __restrict__ K2, const float* __restrict__ D,
    float2* __restrict__ y, int rows, int H, int L, St status) {
  using Cf = ClusterCfg<LOGN>;
  constexpr int n = Cf::n, m = Cf::m, T = Cf::T, NP = Cf::NP, LOGM = Cf::LOGM, C = Cf::C;
  constexpr int RB = plan_radix(LOGM, NP - 1, false), NBL = m / RB, PERL = NBL / T;
  using IXL = PassIdx<m, RB, m / RB>;
  using IXI0 = PassIdx<m, RB, 1>;
  using TWL = PassTw<LOGM, NP - 1, false>;
  cg::cluster_group cl = cg::this_cluster();
  const int c = (int)cl.block_rank();
  extern __shared__ float2 smem[];
  float2* tw1 = smem;
  float2* buf = tw1 + Cf::MI;
  float2* const bufs[1] = {buf};
  const int lt = threadIdx.x;
  fill_cross_twiddles(tw1, c, Cf::MI, n, lt, T);
  const bool zero = st_bad(status);
  __syncthreads();
  cl.sync();
  const float sc = 1.f / n;
  const int ncl = gridDim.x / C;
  const int batch = rows / H;
  for (int idx = blockIdx.x / C; idx < rows; idx += ncl) {
    // channel-major order: the batch rows of one channel run on neighbouring
    // clusters at about the same time and share its spectrum through L2
    const int h = idx / batch, row = (idx % batch) * H + h;
    {  // this CTA's slice of the channel spectrum into L2 during the forward transform
      const char* k2 = reinterpret_cast<const char*>(K2 + (size_t)h * n + (size_t)c * m);
      for (int o = lt * 128; o < m * (int)sizeof(float2); o += T * 128) prefetch_l2(k2 + o);
    }
    const float d = D[h];
    cross_forward<LOGN>(cl, buf, tw1, c, lt, [&](int, int, int t) {
      return make_float2((t < L && S4_IN((long long)row * L + t, (long long)rows * L)) ? u[(size_t)row * L + t] : 0.f, 0.f);
    });
    cl.sync();
    passes_rows<LOGM, false, 0, NP - 2, T, 1>(bufs, lt);
    {
      float2 a[PERL][RB];
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
        float2 kv[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          kv[q] = ld_chk(K2, (long long)h * n + (long long)c * m + i + q * NBL, (long long)H * n);
          kv[q].x += d;
        }
        float2 w[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) a[s][q] = buf[IXL::rd(i, q)];
        TWL::load(w, i);
        TWL::apply(a[s], w);
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
        for (int q = 0; q < RB; ++q) buf[IXI0::wr(i, q)] = a[s][q];
      }
      __syncthreads();
    }
    passes_rows<LOGM, true, 1, NP - 1, T, 1>(bufs, lt);
    cl.sync();
    cross_inverse<LOGN, true>(cl, buf, tw1, c, lt, [&](int, int, int t, float2 v) {
      if (t < L) st_chk(y, (long long)row * L + t, (long long)rows * L, zero ? make_float2(0.f, 0.f) : cscale(v, sc));
    });
    cl.sync();
  }
}

// Fused causal convolution for long rows, two batch rows per complex row
// (2M = 2^14 .. 2^16, where two row buffers fit in one CTA's shared memory).
// With z = u_b + i u_{b+1} one forward transform serves both rows; the two
// spectra are split from Z[g] and Z[n-g] (split_mul), where bin n - g of
// CTA c's bin g = c + C k lives in CTA (C - c) mod C at local index
// m - 1 - k (c != 0) or (m - k) mod m (c = 0), read through DSMEM.  The skip
// term enters as D added to every kernel-spectrum bin (the spectrum of D times
// the unit impulse), and the 1/2 of the split and the 1/n of the inverse are
// applied to the outputs.
template <int LOGN>
__global__ void __launch_bounds__(ClusterCfg<LOGN, true>::T) conv_cluster_pair_kernel(
    const float* __restrict__ u, const float2* __restrict__ K2, const float* __restrict__ D,
    float2* __restrict__ y, int batch, int H, int L, St status) {
  using Cf = ClusterCfg<LOGN, true>;
  constexpr int n = Cf::n, m = Cf::m, T = Cf::T, NP = Cf::NP, LOGM = Cf::LOGM, C = Cf::C;
  constexpr int RB = plan_radix(LOGM, NP - 1, false), NBL = m / RB, PERL = NBL / T;
  using IXL = PassIdx<m, RB, m / RB>;
  using IXI0 = PassIdx<m, RB, 1>;
  using TWL = PassTw<LOGM, NP - 1, false>;
  cg::cluster_group cl = cg::this_cluster();
  const int c = (int)cl.block_rank();
  extern __shared__ float2 smem[];
  float2* tw1 = smem;
  float2* bufA = tw1 + Cf::MI;
  float2* bufB = bufA + Cf::PADM;
  float2* const buf1[1] = {bufA};
  float2* const buf2[2] = {bufA, bufB};
  const int lt = threadIdx.x;
  fill_cross_twiddles(tw1, c, Cf::MI, n, lt, T);
  const bool zero = st_bad(status);
  __syncthreads();
  cl.sync();
  const float sc = 0.5f / n;
  const int ncl = gridDim.x / C;
  const int pb = (batch + 1) / 2, pairs = pb * H;
  const float2* zpart = cl.map_shared_rank(bufA, (C - c) & (C - 1));
  for (int p = blockIdx.x / C; p < pairs; p += ncl) {
    // channel-major order (see conv_cluster_kernel)
    const int h = p / pb, b0 = 2 * (p % pb);
    const float2* K2c = K2 + (size_t)h * n + (size_t)c * m;
    {
      const char* k2 = reinterpret_cast<const char*>(K2c);
      for (int o = lt * 128; o < m * (int)sizeof(float2); o += T * 128) prefetch_l2(k2 + o);
    }
    const bool has1 = b0 + 1 < batch;
    const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
    const float d = D[h];
    cross_forward<LOGN, true>(cl, bufA, tw1, c, lt, [&](int, int, int t) {
      return make_float2(t < L ? u[row0 * L + t] : 0.f, (has1 && t < L) ? u[row1 * L + t] : 0.f);
    });
    cl.sync();
    passes_rows<LOGM, false, 0, NP - 2, T, 1>(buf1, lt);
    // last local forward pass: Z at local bins k = i + q NBL, in registers
    float2 z[PERL][RB];
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
      float2 w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) z[s][q] = bufA[IXL::rd(i, q)];
      TWL::load(w, i);
      TWL::apply(z[s], w);
      dft<RB, false>(z[s]);
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < PERL; ++s)
#pragma unroll
      for (int q = 0; q < RB; ++q) bufA[pad(lt + s * T + q * NBL)] = z[s][q];
    cl.sync();  // every CTA's Z is in place for its partner
    // split, product with K2 + D, first inverse pass in registers; row b+1
    // goes to bufB at once, row b (replacing Z) after the partner has read it
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
      float2 a1[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) {
        const int k = i + q * NBL;
        const int km = c == 0 ? ((m - k) & (m - 1)) : (m - 1 - k);
        float2 kv = K2c[k];
        kv.x += d;
        split_mul(z[s][q], ld_chk(zpart, pad(km), Cf::PADM), kv, z[s][q], a1[q]);
      }
      dft<RB, true>(z[s]);
      dft<RB, true>(a1);
#pragma unroll
      for (int q = 0; q < RB; ++q) bufB[IXI0::wr(i, q)] = a1[q];
    }
    cl.sync();
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
#pragma unroll
      for (int q = 0; q < RB; ++q) bufA[IXI0::wr(i, q)] = z[s][q];
    }
    __syncthreads();
    passes_rows<LOGM, true, 1, NP - 1, T, 2>(buf2, lt);
    cl.sync();
    cross_inverse<LOGN, true, true>(cl, bufA, tw1, c, lt, [&](int, int, int t, float2 v) {
      if (t < L) y[row0 * L + t] = zero ? make_float2(0.f, 0.f) : cscale(v, sc);
    });
    if (has1)
      cross_inverse<LOGN, true, true>(cl, bufB, tw1, c, lt, [&](int, int, int t, float2 v) {
        if (t < L) y[row1 * L + t] = zero ? make_float2(0.f, 0.f) : cscale(v, sc);
      });
    cl.sync();
  }
}

// Real-output convolution for long rows: two batch rows b, b+1 are the real
// and imaginary parts of one complex row; with the spectrum of Re K (Hermitian)
// the inverse transform gives y_b + i y_{b+1} directly.
template <int LOGN>
__global__ void __launch_bounds__(ClusterCfg<LOGN>::T) conv_cluster_real_kernel(
    const float* __restrict__ u, const float2* __restrict__ K2, const float* __restrict__ D,
    float* __restrict__ y, int batch, int H, int L, St status) {
  using Cf = ClusterCfg<LOGN>;
  constexpr int n = Cf::n, m = Cf::m, T = Cf::T, NP = Cf::NP, LOGM = Cf::LOGM, C = Cf::C;
  constexpr int RB = plan_radix(LOGM, NP - 1, false), NBL = m / RB, PERL = NBL / T;
  using IXL = PassIdx<m, RB, m / RB>;
  using IXI0 = PassIdx<m, RB, 1>;
  using TWL = PassTw<LOGM, NP - 1, false>;
  cg::cluster_group cl = cg::this_cluster();
  const int c = (int)cl.block_rank();
  extern __shared__ float2 smem[];
  float2* tw1 = smem;
  float2* buf = tw1 + Cf::MI;
  float2* const bufs[1] = {buf};
  const int lt = threadIdx.x;
  fill_cross_twiddles(tw1, c, Cf::MI, n, lt, T);
  const bool zero = st_bad(status);
  __syncthreads();
  cl.sync();
  const float sc = 1.f / n;
  const int ncl = gridDim.x / C;
  const int pairs = ((batch + 1) / 2) * H;
  const int pb = (batch + 1) / 2;
  for (int p = blockIdx.x / C; p < pairs; p += ncl) {
    // channel-major order (see conv_cluster_kernel)
    const int h = p / pb, b0 = 2 * (p % pb);
    {
      const char* k2 = reinterpret_cast<const char*>(K2 + (size_t)h * n + (size_t)c * m);
      for (int o = lt * 128; o < m * (int)sizeof(float2); o += T * 128) prefetch_l2(k2 + o);
    }
    const bool has1 = b0 + 1 < batch;
    const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
    const float d = D[h];
    float u0[Cf::PI][C / 2], u1[Cf::PI][C / 2];
    cross_forward<LOGN>(cl, buf, tw1, c, lt, [&](int s, int q, int t) {
      const float v0 = t < L ? u[row0 * L + t] : 0.f;
      const float v1 = (has1 && t < L) ? u[row1 * L + t] : 0.f;
      u0[s][q] = v0;
      u1[s][q] = v1;
      return make_float2(v0, v1);
    });
    cl.sync();
    passes_rows<LOGM, false, 0, NP - 2, T, 1>(bufs, lt);
    {
      float2 a[PERL][RB];
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
        float2 w[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) a[s][q] = buf[IXL::rd(i, q)];
        TWL::load(w, i);
        TWL::apply(a[s], w);
        dft<RB, false>(a[s]);
#pragma unroll
        for (int q = 0; q < RB; ++q) a[s][q] = cmul(a[s][q], K2[(size_t)h * n + (size_t)c * m + i + q * NBL]);
        dft<RB, true>(a[s]);
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < PERL; ++s) {
        const int i = lt + s * T;
#pragma unroll
        for (int q = 0; q < RB; ++q) buf[IXI0::wr(i, q)] = a[s][q];
      }
      __syncthreads();
    }
    passes_rows<LOGM, true, 1, NP - 1, T, 1>(bufs, lt);
    cl.sync();
    cross_inverse<LOGN, true>(cl, buf, tw1, c, lt, [&](int s, int q, int t, float2 v) {
      if (t < L) {
        y[row0 * L + t] = zero ? 0.f : fmaf(v.x, sc, d * u0[s][q]);
        if (has1) y[row1 * L + t] = zero ? 0.f : fmaf(v.y, sc, d * u1[s][q]);
      }
    });
    cl.sync();
  }
}

}  // namespace s4dev

namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_cluster)
#endif

template <typename... KArgs, typename... Args>
static cudaError_t launch_clustered(void (*kern)(KArgs...), int C, int threads, size_t smem,
                                    int rows, const char* name, cudaStream_t s, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(C * rows);
  int maxc = 0;
  if (cudaOccupancyMaxActiveClusters(&maxc, kern, &cfg) != cudaSuccess || maxc < 1) {
    (void)cudaGetLastError();
    maxc = 1;
  }
  const int ncl = rows < maxc ? rows : maxc;
  cfg.gridDim = dim3(C * ncl);
  TimedLaunch tl(name, s);
  e = cudaLaunchKernelEx(&cfg, kern, args...);
  return e;
}

template <int LOGN>
static cudaError_t ifft_cl(const float2* Khat, float2* K, int H, int L, St st,
                           cudaStream_t s) {
  using Cf = ClusterCfg<LOGN>;
  const size_t smem = sizeof(float2) * (Cf::MI + (size_t)Cf::PADM);
  return launch_clustered(ifft_cluster_kernel<LOGN>, Cf::C, Cf::T, smem, H, "ifft", s, Khat, K, H, L, st);
}

template <int LOGN>
static cudaError_t spectrum_cl(const float2* K, float2* K2, int H, int L, St st, cudaStream_t s,
                               bool realk) {
  using Cf = ClusterCfg<LOGN>;
  const size_t smem = sizeof(float2) * (Cf::MI + (size_t)Cf::PADM);
  return launch_clustered(spectrum_cluster_kernel<LOGN>, Cf::C, Cf::T, smem, H, "spectrum", s, K, K2,
                          H, L, realk ? 1 : 0, st);
}

template <int LOGN>
static cudaError_t conv_pair_cl(const float* u, const float2* K2, const float* D, float2* y, int batch,
                                int H, int L, St st, cudaStream_t s) {
  using Cf = ClusterCfg<LOGN, true>;
  const size_t smem = sizeof(float2) * (Cf::MI + 2 * (size_t)Cf::PADM);
  const int pairs = ((batch + 1) / 2) * H;
  return launch_clustered(conv_cluster_pair_kernel<LOGN>, Cf::C, Cf::T, smem, pairs, "conv", s, u, K2, D,
                          y, batch, H, L, st);
}

template <int LOGN>
static cudaError_t conv_real_cl(const float* u, const float2* K2, const float* D, float* y, int batch,
                                int H, int L, St st, cudaStream_t s) {
  using Cf = ClusterCfg<LOGN>;
  const size_t smem = sizeof(float2) * (Cf::MI + (size_t)Cf::PADM);
  const int pairs = ((batch + 1) / 2) * H;
  return launch_clustered(conv_cluster_real_kernel<LOGN>, Cf::C, Cf::T, smem, pairs, "conv_real", s, u,
                          K2, D, y, batch, H, L, st);
}

cudaError_t launch_conv_real_cluster(int logn, const float* u, const float2* K2, const float* D,
                                     float* y, int batch, int H, int L, St st,
                                     cudaStream_t s) {
  switch (logn) {
    case 14: return conv_real_cl<14>(u, K2, D, y, batch, H, L, st, s);
    case 15: return conv_real_cl<15>(u, K2, D, y, batch, H, L, st, s);
    case 16: return conv_real_cl<16>(u, K2, D, y, batch, H, L, st, s);
    case 17: return conv_real_cl<17>(u, K2, D, y, batch, H, L, st, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int LOGN>
static cudaError_t conv_cl(const float* u, const float2* K2, const float* D, float2* y, int rows, int H,
                           int L, St st, cudaStream_t s) {
  using Cf = ClusterCfg<LOGN>;
  const size_t smem = sizeof(float2) * (Cf::MI + (size_t)Cf::PADM);
  return launch_clustered(conv_cluster_kernel<LOGN>, Cf::C, Cf::T, smem, rows, "conv", s, u, K2, D, y,
                          rows, H, L, st);
}

cudaError_t launch_ifft_cluster(int logM, const float2* Khat, float2* K, int H, int L,
                                St st, cudaStream_t s) {
  switch (logM) {
    case 15: return ifft_cl<15>(Khat, K, H, L, st, s);
    case 16: return ifft_cl<16>(Khat, K, H, L, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_spectrum_cluster(int logn, const float2* K, float2* K2, int H, int L,
                                    St st, cudaStream_t s, bool realk) {
  switch (logn) {
    case 14: return spectrum_cl<14>(K, K2, H, L, st, s, realk);
    case 15: return spectrum_cl<15>(K, K2, H, L, st, s, realk);
    case 16: return spectrum_cl<16>(K, K2, H, L, st, s, realk);
    case 17: return spectrum_cl<17>(K, K2, H, L, st, s, realk);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_conv_cluster(int logn, const float* u, const float2* K2, const float* D,
                                float2* y, int rows, int H, int L, St st,
                                cudaStream_t s) {
  // two batch rows per complex row where two row buffers fit a CTA (2^14..2^16);
  // one row at a time at 2^17
  const int batch = rows / H;
  switch (logn) {
    case 14: return conv_pair_cl<14>(u, K2, D, y, batch, H, L, st, s);
    case 15: return conv_pair_cl<15>(u, K2, D, y, batch, H, L, st, s);
    case 16: return conv_pair_cl<16>(u, K2, D, y, batch, H, L, st, s);
    case 17: return conv_cl<17>(u, K2, D, y, rows, H, L, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
