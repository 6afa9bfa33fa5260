// Fused causal convolution for long rows (2M = 2^14 .. 2^17 points) by a
// four-step split through global memory, with ordinary CTAs (no clusters), so
// that every SM takes part.
//
// "Recurrent, LSTM, and structured state-space models": y_t = sum_{j<=t} K_j
// u_{t-j} + D u_t; section "Roots-of-unity orthogonality and radix-two FFT
// cost": the product of two length-M polynomials by zero-padding to n = 2M.
//
// Two batch rows b, b+1 of a channel are one complex row z = u_b + i u_{b+1}.
// With K^r and K^i the spectra of Re K and Im K (both Hermitian, formed from
// the spectrum K^ of K as K^r[k] = (K^[k] + conj K^[-k])/2 and K^i[k] =
// (K^[k] - conj K^[-k])/(2i)), the two inverse transforms
//     a = iFFT(Z (K^r + D)) = (Re K * u_b + D u_b) + i (Re K * u_{b+1} + D u_{b+1})
//     c = iFFT(Z K^i)       =  Im K * u_b + i Im K * u_{b+1}
// give y_b = Re a + i Re c and y_{b+1} = Im a + i Im c, with no mirror of Z
// (the skip term D u enters as D added to every bin of K^r: the spectrum of D
// times the unit impulse).
//
// Split n = R m, t = m t1 + t2, k = k1 + R k2 (t1, k1 < R; t2, k2 < m):
//     Z[k1 + R k2] = sum_{t2} w_m^{t2 k2} (w_n^{t2 k1} sum_{t1} z[m t1 + t2] w_R^{t1 k1}),
// w_n = exp(-2 pi i/n), with R = 16 up to n = 2^16 and R = 32 at n = 2^17
// (columns of 4096 points, which run two CTAs per SM).  Three kernels:
//   fs_forward_kernel  per (pair, t2): the R-point DFT over t1 (inputs t1 >= R/2
//                      are the zero padding) and the twiddle w_n^{t2 k1} -> X[pair][k1][t2]
//   fs_column_kernel   per (pair, k1): the m-point FFT over t2, the products with
//                      K^r + D and K^i (scaled 1/n), two m-point inverse FFTs over k2
//                      -> a and c in the (k1, t2) layout (a over X's storage)
//   fs_inverse_kernel  per (pair, t2): the twiddle w_n^{-t2 k1} and the R-point
//                      inverse over k1 for t1 < R/2 (t < M) -> y_b, y_{b+1}
// The spectrum K^ is read in a blocked order, bin k at (k mod C) n/C + k div C:
// C = R ("column order", K^[k1][k2]) when it comes from the four-step spectrum
// below, C = 2^cluster_log(log n) when it comes from the cluster spectrum kernels.
//
// The kernel spectrum itself, also in four steps:
//   fs_kfwd_kernel   per (channel, t2): the radix-R across-column step of the
//                    2M-point transform of K (zero-padded) -> X[h][k1][t2];
//                    the row spectrum kernel then transforms the R H columns of
//                    2M/R points (full transforms) -> K2 in column order, scaled 8/(2M).
// and, on the layer path, from the root values Khat in column order
// [k1][k2] (k = k1 + 16 k2 of the M-point grid):
//   the row inverse-transform kernel: the 16 H columns of M/16 points, 1/(M/16)
//   ks_cross_kernel  per (channel, t2 < M/16): the twiddle w_M^{-t2 k1} and the
//                    16-point inverse over k1 (1/16) -> K[h][t], t = (M/16) t1 + t2
//                    (written out), then the forward across-column step of the
//                    2M transform: with R = 16 for its two columns t2 and t2 + M/16,
//                    with R = 32 for its column t2 (whose nonzero inputs are exactly
//                    these 16 values) -> X[h][k1][.]
// When L = M the 2M-point spectrum needs only half of that: its even bins are the
// root values themselves (K^[2j] = sum_{t<M} K[t] w_M^{jt} = Khat[j], K being the
// whole inverse transform), and its odd bins are the M-point transform of the
// twisted kernel, K^[2j+1] = sum_t (K[t] w_2M^t) w_M^{jt}.  With the root values in
// column order of C = R/2 ([k1][k2], k = k1 + C k2 of the M-point grid):
//   the row inverse-transform kernel: the C H columns of M/C points, 1/(M/C)
//   ks_cross_half_kernel per (channel, t2 < M/C): the radix-C inverse -> K (written
//                    out), the twist w_2M^t and the radix-C forward across-column
//                    step of its M-point transform -> X[h][k1][t2]
//   the row spectrum kernel on the C H columns -> T = K^[odd] in column order of C.
// The column kernel then reads the spectrum's bin k = k1 + R k2 of its column from
// the root values (k1 even) or from T (k1 odd), at j = k div 2 = k1/2 + C k2: one
// contiguous column of either array.
// (light twiddle loads only in the passes of P >= 256 here; see s4_fft.cuh)
#ifndef S4_TW_LIGHT_MINP
#define S4_TW_LIGHT_MINP 256
#endif
#include "s4_fft.cuh"
#include "s4_internal.h"

namespace s4dev {

// Build-time tuning: the column kernel reads its input cached in L2 only (1), which
// keeps L1 for the twiddle tables (1140 -> 1098 us with the light loads on N=256
// H=1024 L=65536), or as streaming data (0).
#ifndef S4_FS_XCG
#define S4_FS_XCG 1
#endif

constexpr int kFsThreads = 256;  // threads per CTA of the across-column kernels
constexpr int kKsRadix = 16;     // across-column radix of the layer path's M-point inverse

// a[q] *= w^q, q = 1..R-1, each power the product of the w^(2^j) of its bits:
// few registers live beside a 32-point array (apply_twiddles keeps all powers).
template <int R>
__device__ __forceinline__ void apply_twiddles_bits(float2* a, float2 w) {
  constexpr int LR = R <= 1 ? 0 : R <= 2 ? 1 : R <= 4 ? 2 : R <= 8 ? 3 : R <= 16 ? 4 : 5;
  float2 b[LR > 0 ? LR : 1];
  b[0] = w;
#pragma unroll
  for (int j = 1; j < LR; ++j) b[j] = cmul(b[j - 1], b[j - 1]);
#pragma unroll
  for (int q = 1; q < R; ++q) {
    float2 t = make_float2(1.f, 0.f);
    bool first = true;
#pragma unroll
    for (int j = 0; j < LR; ++j)
      if ((q >> j) & 1) {
        t = first ? b[j] : cmul(t, b[j]);
        first = false;
      }
    a[q] = cmul(a[q], t);
  }
}
template <int R>
__device__ __forceinline__ void fs_twiddles(float2* a, float2 w) {
  if constexpr (R > 16) apply_twiddles_bits<R>(a, w);
  else apply_twiddles<R>(a, w);
}

// Rows of a pair: pair p = h pb + j (pb = ceil(batch / 2)) holds rows b0 = 2 j and b0 + 1.
struct FsPair {
  int h;
  size_t row0, row1;
  bool has1;
};
__device__ __forceinline__ FsPair fs_pair(int p, int pb, int batch, int H) {
  FsPair q;
  q.h = p / pb;
  const int b0 = 2 * (p % pb);
  q.row0 = (size_t)b0 * H + q.h;
  q.row1 = q.row0 + H;
  q.has1 = b0 + 1 < batch;
  return q;
}

// w_n^{t2} = exp(-2 pi i t2 / n)
__device__ __forceinline__ float2 fs_twiddle(int t2, int n) {
  float s, c;
  sincospif(2.0f * (float)t2 / (float)n, &s, &c);
  return make_float2(c, -s);
}

template <int LOGN>
__global__ void __launch_bounds__(kFsThreads) fs_forward_kernel(const float* __restrict__ u,
                                                                float2* __restrict__ X, int batch, int H,
                                                                int L, int pb) {
  constexpr int R = 1 << s4impl::fs_log_radix(LOGN), n = 1 << LOGN, m = n / R;
  const long long gid = (long long)blockIdx.x * kFsThreads + threadIdx.x;
  const int p = (int)(gid / m), t2 = (int)(gid % m);
  if (p >= pb * H) return;
  const FsPair q = fs_pair(p, pb, batch, H);
  float2 x[R];
#pragma unroll
  for (int t1 = 0; t1 < R; ++t1) {
    const int t = m * t1 + t2;
    const long long nu = (long long)batch * H * L;
    x[t1] = t1 >= R / 2 ? make_float2(0.f, 0.f)
          : make_float2((t < L && S4_IN(q.row0 * L + t, nu)) ? __ldcs(u + q.row0 * L + t) : 0.f,
                        (q.has1 && t < L && S4_IN(q.row1 * L + t, nu)) ? __ldcs(u + q.row1 * L + t) : 0.f);
  }
  dft<R, false, true>(x);
  fs_twiddles<R>(x, fs_twiddle(t2, n));
  const long long nx = (long long)pb * H * n;
#pragma unroll
  for (int k1 = 0; k1 < R; ++k1) st_chk(X, (long long)p * n + (long long)k1 * m + t2, nx, x[k1]);
}

// Forward across-column step of the 2M-point spectrum of a complex kernel K
// [H][L] (zero beyond L): X[h][k1][t2] = w_n^{t2 k1} sum_{t1 < R/2} K[m t1 + t2] w_R^{t1 k1}.
template <int LOGN>
__global__ void __launch_bounds__(kFsThreads) fs_kfwd_kernel(const float2* __restrict__ K,
                                                             float2* __restrict__ X, int H, int L,
                                                             int realk) {
  constexpr int R = 1 << s4impl::fs_log_radix(LOGN), n = 1 << LOGN, m = n / R;
  const long long gid = (long long)blockIdx.x * kFsThreads + threadIdx.x;
  const int h = (int)(gid / m), t2 = (int)(gid % m);
  if (h >= H) return;
  float2 x[R];
#pragma unroll
  for (int t1 = 0; t1 < R; ++t1) {
    const int t = m * t1 + t2;
    x[t1] = (t1 < R / 2 && t < L && S4_IN((long long)h * L + t, (long long)H * L)) ? __ldg(K + (size_t)h * L + t)
                                                                                  : make_float2(0.f, 0.f);
    if (realk) x[t1].y = 0.f;
  }
  dft<R, false, true>(x);
  fs_twiddles<R>(x, fs_twiddle(t2, n));
#pragma unroll
  for (int k1 = 0; k1 < R; ++k1)
    st_chk(X, (long long)h * n + (long long)k1 * m + t2, (long long)H * n, x[k1]);
}

// Layer path: K from the column inverse transforms G[h][k1][t2] (M/16 points
// each, already scaled 1/(M/16)), and the forward across-column step of its
// 2M-point spectrum.  A thread owns t2 < M/16: K[(M/16) t1 + t2] for all t1 < 16.
// With the 2M step's radix RO = 16 (columns of M/8 points) these are the 8
// nonzero inputs of its columns t2 (t1 even) and t2 + M/16 (t1 odd); with
// RO = 32 (columns of M/16 points) they are the 16 nonzero inputs of column t2.
template <int LOGM>
__global__ void __launch_bounds__(kFsThreads) ks_cross_kernel(const float2* __restrict__ G,
                                                              float2* __restrict__ K, float2* __restrict__ X,
                                                              int H, int L, St status) {
  constexpr int RI = kKsRadix, RO = 1 << s4impl::fs_log_radix(LOGM + 1);
  constexpr int M = 1 << LOGM, mi = M / RI, n = 2 * M, mf = n / RO;
  const long long gid = (long long)blockIdx.x * kFsThreads + threadIdx.x;
  const int h = (int)(gid / mi), t2 = (int)(gid % mi);
  if (h >= H) return;
  const bool zero = st_bad(status);
  float2 g[RI];
  const float2* gp = G + (size_t)h * M + t2;
#pragma unroll
  for (int k1 = 0; k1 < RI; ++k1)
    g[k1] = S4_IN((long long)h * M + (long long)k1 * mi + t2, (long long)H * M) ? __ldcs(gp + (size_t)k1 * mi)
                                                                               : make_float2(0.f, 0.f);
  float2 w = fs_twiddle(t2, M);
  w.y = -w.y;
  apply_twiddles<RI>(g, w);
  dft<RI, true>(g);
#pragma unroll
  for (int t1 = 0; t1 < RI; ++t1) {
    const int t = mi * t1 + t2;
    g[t1] = (zero || t >= L) ? make_float2(0.f, 0.f) : cscale(g[t1], 1.f / RI);
    if (t < L) st_chk(K, (long long)h * L + t, (long long)H * L, g[t1]);
  }
  if constexpr (RO == 2 * RI) {
    static_assert(mf == mi, "one 2M column per thread");
    float2 x[RO];
#pragma unroll
    for (int t1 = 0; t1 < RO; ++t1) x[t1] = t1 < RI ? g[t1] : make_float2(0.f, 0.f);
    dft<RO, false, true>(x);
    fs_twiddles<RO>(x, fs_twiddle(t2, n));
#pragma unroll
    for (int k1 = 0; k1 < RO; ++k1) st_chk(X, (long long)h * n + (long long)k1 * mf + t2, (long long)H * n, x[k1]);
  } else {
    static_assert(RO == RI && mf == 2 * mi, "two 2M columns per thread");
    float2 xa[RO], xb[RO];
#pragma unroll
    for (int t1 = 0; t1 < RO; ++t1) {
      xa[t1] = t1 < RO / 2 ? g[2 * t1] : make_float2(0.f, 0.f);
      xb[t1] = t1 < RO / 2 ? g[2 * t1 + 1] : make_float2(0.f, 0.f);
    }
    dft<RO, false, true>(xa);
    dft<RO, false, true>(xb);
    apply_twiddles<RO>(xa, fs_twiddle(t2, n));
    apply_twiddles<RO>(xb, fs_twiddle(t2 + mi, n));
#pragma unroll
    for (int k1 = 0; k1 < RO; ++k1) {
      st_chk(X, (long long)h * n + (long long)k1 * mf + t2, (long long)H * n, xa[k1]);
      st_chk(X, (long long)h * n + (long long)k1 * mf + mi + t2, (long long)H * n, xb[k1]);
    }
  }
}

// Layer path with L = M: K from the column inverse transforms G[h][k1][t2] (M/C
// points each, scaled 1/(M/C); C = R/2 for the 2M split's radix R), and the forward
// across-column step of the M-point transform of K[t] w_2M^t, whose bins are the
// odd bins of K's 2M-point spectrum.  A thread owns t2 < M/C and K[(M/C) t1 + t2]
// for all t1 < C; w_2M^t = w_{2C}^{t1} w_2M^{t2}, the second factor applied after
// the DFT over t1 together with the across-column twiddle w_M^{t2 k1}.
template <int LOGM>
__global__ void __launch_bounds__(kFsThreads) ks_cross_half_kernel(const float2* __restrict__ G,
                                                                   float2* __restrict__ K,
                                                                   float2* __restrict__ X, int H, int L,
                                                                   St status) {
  constexpr int C = 1 << (s4impl::fs_log_radix(LOGM + 1) - 1);
  constexpr int M = 1 << LOGM, mi = M / C, n = 2 * M;
  const long long gid = (long long)blockIdx.x * kFsThreads + threadIdx.x;
  if (gid / mi >= H) return;
  // channels in reverse order: the first read are the inverse transforms' last
  // writes (still in L2), the last written are the column spectra's first reads
  const int h = H - 1 - (int)(gid / mi), t2 = (int)(gid % mi);
  const bool zero = st_bad(status);
  float2 g[C];
  const float2* gp = G + (size_t)h * M + t2;
#pragma unroll
  for (int k1 = 0; k1 < C; ++k1)
    g[k1] = S4_IN((long long)h * M + (long long)k1 * mi + t2, (long long)H * M) ? __ldcs(gp + (size_t)k1 * mi)
                                                                              : make_float2(0.f, 0.f);
  float2 w = fs_twiddle(t2, M);
  w.y = -w.y;
  apply_twiddles<C>(g, w);
  dft<C, true>(g);
#pragma unroll
  for (int t1 = 0; t1 < C; ++t1) {
    const int t = mi * t1 + t2;
    g[t1] = (zero || t >= L) ? make_float2(0.f, 0.f) : cscale(g[t1], 1.f / C);
    if (t < L) st_chk(K, (long long)h * L + t, (long long)H * L, g[t1]);
    // w_{2C}^{t1} = exp(-2 pi i t1 / (2C)), in 32nds of a turn
    if (t1 > 0) g[t1] = cmul(g[t1], make_float2(cos32(t1 * (16 / C)), -sin32(t1 * (16 / C))));
  }
  dft<C, false>(g);
  // times w_2M^{t2 (2 k1 + 1)}: v = w_2M^{t2} on every output, then (v^2)^{k1}
  const float2 v = fs_twiddle(t2, n);
#pragma unroll
  for (int k1 = 0; k1 < C; ++k1) g[k1] = cmul(g[k1], v);
  apply_twiddles<C>(g, fs_twiddle(t2, M));
#pragma unroll
  for (int k1 = 0; k1 < C; ++k1) st_chk(X, (long long)h * M + (long long)k1 * mi + t2, (long long)H * M, g[k1]);
}

// Stores y_b[t] = (Re a_t, Re c_t) and y_{b+1}[t] = (Im a_t, Im c_t) for t < L.
__device__ __forceinline__ void fs_store_y(float2* __restrict__ y, const FsPair& q, int t, int L, long long ny,
                                           bool zero, float2 a, float2 c) {
  if (t >= L) return;
  if (S4_IN(q.row0 * L + t, ny)) __stcs(y + q.row0 * L + t, zero ? make_float2(0.f, 0.f) : make_float2(a.x, c.x));
  if (q.has1 && S4_IN(q.row1 * L + t, ny))
    __stcs(y + q.row1 * L + t, zero ? make_float2(0.f, 0.f) : make_float2(a.y, c.y));
}

// Inverse across-column step.  R = 16: one thread per (pair, t2).  R = 32: two
// lanes per (pair, t2), lanes l and l + 16 of a warp, the half h = l / 16 taking
// k1 = 2 j + h: with A' the twiddled column values, the outputs t1 < 16 are
//     sum_{k1} w_32^{-t1 k1} A'[k1] = E[t1] + w_32^{-t1} O[t1],
// E and O the 16-point inverse DFTs over j of A'[2 j] and A'[2 j + 1].  Half 0
// keeps t1 < 8 and half 1 keeps t1 >= 8, each taking the other half's 8 values
// by a shuffle (half the registers of a 32-point transform per thread).
template <int LOGN>
__global__ void __launch_bounds__(kFsThreads) fs_inverse_kernel(const float2* __restrict__ Ar,
                                                                const float2* __restrict__ Ci,
                                                                float2* __restrict__ y, int batch, int H,
                                                                int L, int pb, St status) {
  constexpr int R = 1 << s4impl::fs_log_radix(LOGN), n = 1 << LOGN, m = n / R;
  const long long gid = (long long)blockIdx.x * kFsThreads + threadIdx.x;
  const bool zero = st_bad(status);
  const long long nx = (long long)pb * H * n, ny = (long long)batch * H * L;
  if constexpr (R == 32) {
    constexpr int RH = R / 2;
    const int lane = threadIdx.x & 31, h = lane >> 4;
    const long long slot = (gid >> 5) * 16 + (lane & 15);
    const int p = (int)(slot / m), t2 = (int)(slot % m);
    const bool act = p < pb * H;  // no early return: the warp shuffles below
    const FsPair q = fs_pair(act ? p : 0, pb, batch, H);
    float2 a[RH], c[RH];
    const size_t base = (size_t)(act ? p : 0) * n + t2 + (size_t)h * m;
#pragma unroll
    for (int j = 0; j < RH; ++j) {
      const bool in = act && S4_IN((long long)base + (long long)(2 * j) * m, nx);
      a[j] = in ? __ldcs(Ar + base + (size_t)(2 * j) * m) : make_float2(0.f, 0.f);
      c[j] = in ? __ldcs(Ci + base + (size_t)(2 * j) * m) : make_float2(0.f, 0.f);
    }
    // twiddle w_n^{-t2 k1} = (w^2)^j w^h, w = w_n^{-t2}
    float2 w = fs_twiddle(t2, n);
    w.y = -w.y;
    const float2 w2 = cmul(w, w);
    if (h) {
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        a[j] = cmul(a[j], w);
        c[j] = cmul(c[j], w);
      }
    }
    apply_twiddles<RH>(a, w2);
    apply_twiddles<RH>(c, w2);
    dft<RH, true>(a);
    dft<RH, true>(c);
    if (h) {  // O[t1] w_32^{-t1}
#pragma unroll
      for (int t1 = 1; t1 < RH; ++t1) {
        const float2 r = make_float2(cos32(t1), sin32(t1));
        a[t1] = cmul(a[t1], r);
        c[t1] = cmul(c[t1], r);
      }
    }
#pragma unroll
    for (int j = 0; j < RH / 2; ++j) {
      // half 0 sends E[8 + j] and keeps E[j]; half 1 sends O'[j] and keeps O'[8 + j]
      const float2 sa = h ? a[j] : a[RH / 2 + j], sc = h ? c[j] : c[RH / 2 + j];
      const float2 ra = make_float2(__shfl_xor_sync(0xffffffffu, sa.x, 16), __shfl_xor_sync(0xffffffffu, sa.y, 16));
      const float2 rc = make_float2(__shfl_xor_sync(0xffffffffu, sc.x, 16), __shfl_xor_sync(0xffffffffu, sc.y, 16));
      const float2 ka = h ? a[RH / 2 + j] : a[j], kc = h ? c[RH / 2 + j] : c[j];
      if (act) fs_store_y(y, q, m * (h * (RH / 2) + j) + t2, L, ny, zero, cadd(ka, ra), cadd(kc, rc));
    }
  } else {
    const int p = (int)(gid / m), t2 = (int)(gid % m);
    if (p >= pb * H) return;
    const FsPair q = fs_pair(p, pb, batch, H);
    float2 a[R], c[R];
    const size_t base = (size_t)p * n + t2;
#pragma unroll
    for (int k1 = 0; k1 < R; ++k1) {
      const bool in = S4_IN((long long)base + (long long)k1 * m, nx);
      a[k1] = in ? __ldcs(Ar + base + (size_t)k1 * m) : make_float2(0.f, 0.f);
      c[k1] = in ? __ldcs(Ci + base + (size_t)k1 * m) : make_float2(0.f, 0.f);
    }
    float2 w = fs_twiddle(t2, n);
    w.y = -w.y;
    apply_twiddles<R>(a, w);
    apply_twiddles<R>(c, w);
    dft<R, true, false, true>(a);
    dft<R, true, false, true>(c);
#pragma unroll
    for (int t1 = 0; t1 < R / 2; ++t1) fs_store_y(y, q, m * t1 + t2, L, ny, zero, a[t1], c[t1]);
  }
}

// Column transforms: one column (pair p, k1) of m = 2^LOGM points per row group,
// n = m 2^LOGR.
template <int LOGM>
struct FsColCfg {
  static constexpr int m = 1 << LOGM;
  static constexpr int T = conv_row_threads(LOGM);  // one radix-16 butterfly per thread at m = 8192
  static constexpr int ROWS = T >= 128 ? 1 : 128 / T;
  static constexpr int THREADS = T * ROWS;
  static constexpr int NP = plan_npass(LOGM);
  static constexpr int RA = plan_radix(LOGM, 0, false);
  static constexpr int RB = plan_radix(LOGM, NP - 1, false);
  static constexpr int PADM = padded_len(m);
};

// K^ at natural bin k from the blocked layout of a cluster of 2^logC CTAs.
__device__ __forceinline__ float2 fs_spec(const float2* __restrict__ K2h, int k, int n, int logC) {
  const int C = 1 << logC;
  const long long i = (long long)(k & (C - 1)) * (n >> logC) + (k >> logC);
  return S4_IN(i, n) ? __ldcg(K2h + i) : make_float2(0.f, 0.f);
}

// 512 threads per SM at 128 registers (one CTA for m = 8192, more for shorter columns)
// K2o != nullptr: the spectrum in two halves, even bins from K2 and odd bins from
// K2o (each H x n/2, in the blocked order of 2^logC over n/2 bins), stored as the
// spectrum times n kscale and n kscale_o respectively.
template <int LOGM, int LOGR>
__global__ void __launch_bounds__(FsColCfg<LOGM>::THREADS, 512 / FsColCfg<LOGM>::THREADS) fs_column_kernel(
    float2* __restrict__ X, float2* __restrict__ Ci, const float2* __restrict__ K2,
    const float2* __restrict__ K2o, const float* __restrict__ D, int H, int pb, int logC, float kscale,
    float kscale_o, St status) {
  using C = FsColCfg<LOGM>;
  constexpr int m = C::m, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int R = 1 << LOGR, n = m * R;
  constexpr int NB0 = m / RA, PER0 = NB0 / T, NBL = m / RB, PERL = NBL / T;
  using IXF0 = PassIdx<m, RA, 1>;
  using IXFL = PassIdx<m, RB, m / RB>;
  using IXI0 = PassIdx<m, RB, 1>;
  using IXIL = PassIdx<m, RA, m / RA>;
  using TWFL = PassTw<LOGM, NP - 1, false>;
  using TWIL = PassTw<LOGM, NP - 1, true>;
  extern __shared__ float2 smem[];
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* bufA = smem + slot * 2 * C::PADM;
  float2* bufB = bufA + C::PADM;
  float2* const buf1[1] = {bufA};
  float2* const buf2[2] = {bufA, bufB};
  const bool zero = st_bad(status);
  const int cols = pb * H * R;
  const float sc = 1.f / n;
  for (int c0 = blockIdx.x * C::ROWS; c0 < cols; c0 += gridDim.x * C::ROWS) {
    // columns in reverse order: the first ones read are the across-column step's
    // last writes, still in L2, and the last ones written are the inverse step's first reads
    const bool act = c0 + slot < cols;
    const int col = act ? cols - 1 - (c0 + slot) : 0;
    const int p = act ? col / R : 0, k1 = col % R;
    const int h = p / pb;
    float2* xc = X + (size_t)p * n + (size_t)k1 * m;        // this column: X in, a out
    float2* cc = Ci + (size_t)p * n + (size_t)k1 * m;       // c out
    const bool split = K2o != nullptr, odd = split && (k1 & 1);
    const float2* K2h = split ? (odd ? K2o : K2) + (size_t)h * (n / 2) : K2 + (size_t)h * n;
    const float ksc = odd ? kscale_o : kscale;
    const float dv = act ? D[h] : 0.f;
    // forward pass 0: global -> shared
#pragma unroll
    for (int s = 0; s < PER0; ++s) {
      const int i = lt + s * T;
      float2 a[RA];
#pragma unroll
      for (int qq = 0; qq < RA; ++qq)
        a[qq] = (act && S4_IN((long long)p * n + (long long)k1 * m + i + qq * NB0, (long long)pb * H * n))
                    ? (S4_FS_XCG ? __ldcg(xc + i + qq * NB0) : __ldcs(xc + i + qq * NB0)) : make_float2(0.f, 0.f);
      dft<RA, false>(a);
#pragma unroll
      for (int qq = 0; qq < RA; ++qq) st_chk(bufA, IXF0::wr(i, qq), C::PADM, a[qq]);
    }
    __syncthreads();
    passes_rows<LOGM, false, 1, NP - 2, T, 1>(buf1, lt);
    // last forward pass in registers (bins k2 = i + q NBL), the two products,
    // the first inverse pass (P = 1) in registers
    float2 pa[PERL][RB], pc[PERL][RB];
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
      float2 z[RB], w[RB];
#pragma unroll
      for (int qq = 0; qq < RB; ++qq) z[qq] = ld_chk(bufA, IXFL::rd(i, qq), C::PADM);
      TWFL::load(w, i);
      TWFL::apply(z, w);
      dft<RB, false>(z);
#pragma unroll
      for (int qq = 0; qq < RB; ++qq) {
        const int k2 = i + qq * NBL;
        const int k = k1 + R * k2;
        // K^[k] and K^[-k] (the same parity: the same half when split)
        const int kmir = (n - k) & (n - 1);
        const float2 kv = split ? fs_spec(K2h, k >> 1, n / 2, logC) : fs_spec(K2h, k, n, logC);
        const float2 km = split ? fs_spec(K2h, kmir >> 1, n / 2, logC) : fs_spec(K2h, kmir, n, logC);
        // (K^r + D)/n and K^i/n, the stored spectrum being K^ n ksc
        const float2 kr = make_float2(fmaf(0.5f * ksc, kv.x + km.x, dv * sc), 0.5f * ksc * (kv.y - km.y));
        const float2 ki = make_float2(0.5f * ksc * (kv.y + km.y), 0.5f * ksc * (km.x - kv.x));
        pa[s][qq] = cmul(z[qq], kr);
        pc[s][qq] = cmul(z[qq], ki);
      }
      dft<RB, true>(pa[s]);
      dft<RB, true>(pc[s]);
#pragma unroll
      for (int qq = 0; qq < RB; ++qq) st_chk(bufB, IXI0::wr(i, qq), C::PADM, pc[s][qq]);
    }
    __syncthreads();  // every thread has read its last forward pass from bufA
#pragma unroll
    for (int s = 0; s < PERL; ++s) {
      const int i = lt + s * T;
#pragma unroll
      for (int qq = 0; qq < RB; ++qq) st_chk(bufA, IXI0::wr(i, qq), C::PADM, pa[s][qq]);
    }
    __syncthreads();
    passes_rows<LOGM, true, 1, NP - 2, T, 2>(buf2, lt);
    // last inverse pass: every t2 of both products, back over X's column and into Ci
#pragma unroll
    for (int s = 0; s < PER0; ++s) {
      const int i = lt + s * T;
      float2 a[RA], c[RA], w[RA];
#pragma unroll
      for (int qq = 0; qq < RA; ++qq) {
        a[qq] = ld_chk(bufA, IXIL::rd(i, qq), C::PADM);
        c[qq] = ld_chk(bufB, IXIL::rd(i, qq), C::PADM);
      }
      TWIL::load(w, i);
      TWIL::apply(a, w);
      TWIL::apply(c, w);
      dft<RA, true>(a);
      dft<RA, true>(c);
      if (act) {
#pragma unroll
        for (int qq = 0; qq < RA; ++qq) {
          if (!S4_IN((long long)p * n + (long long)k1 * m + i + qq * NB0, (long long)pb * H * n)) continue;
          xc[i + qq * NB0] = zero ? make_float2(0.f, 0.f) : a[qq];
          cc[i + qq * NB0] = zero ? make_float2(0.f, 0.f) : c[qq];
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace s4dev

namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_fourstep)
#endif

size_t fs_scratch_bytes(int logn, int batch, int H) {
  if (logn < kMinLogFourStep || logn > kMaxLogFourStep) return 0;
  const size_t pairs = (size_t)((batch + 1) / 2) * (size_t)H;
  return 2 * pairs * ((size_t)1 << logn) * sizeof(float2);
}

template <int LOGN>
static cudaError_t fs_launch(const float* u, const float2* K2, int k2_logC, float k2_scale, const float* D,
                             float2* y, int batch, int H, int L, float2* scratch, St st, cudaStream_t s,
                             const float2* K2o, float k2o_scale) {
  constexpr int LOGR = fs_log_radix(LOGN), R = 1 << LOGR, n = 1 << LOGN, m = n / R, LOGM = LOGN - LOGR;
  using C = FsColCfg<LOGM>;
  const int pb = (batch + 1) / 2;
  const long long pairs = (long long)pb * H;
  float2* X = scratch;
  float2* Ci = scratch + (size_t)pairs * n;
  const unsigned blocks = (unsigned)((pairs * m + kFsThreads - 1) / kFsThreads);
  {
    TimedLaunch tl("conv_fwd", s);
    fs_forward_kernel<LOGN><<<blocks, kFsThreads, 0, s>>>(u, X, batch, H, L, pb);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(float2) * 2 * (size_t)C::ROWS * C::PADM;
  auto k = fs_column_kernel<LOGM, LOGR>;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, C::THREADS, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const long long cols = pairs * R;
  const long long need = (cols + C::ROWS - 1) / C::ROWS;
  const int grid = (int)(need < (long long)per_sm * num_sms() ? need : (long long)per_sm * num_sms());
  {
    TimedLaunch tl("conv_col", s);
    k<<<grid, C::THREADS, smem, s>>>(X, Ci, K2, K2o, D, H, pb, k2_logC, k2_scale, k2o_scale, st);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    // R = 32: two lanes per (pair, t2)
    const unsigned iblocks = (unsigned)((pairs * m * (R == 32 ? 2 : 1) + kFsThreads - 1) / kFsThreads);
    TimedLaunch tl("conv_inv", s);
    fs_inverse_kernel<LOGN><<<iblocks, kFsThreads, 0, s>>>(X, Ci, y, batch, H, L, pb, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_conv_fourstep(int logn, const float* u, const float2* K2, int k2_logC, float k2_scale,
                                 const float* D, float2* y, int batch, int H, int L, float2* scratch, St st,
                                 cudaStream_t s, const float2* K2o, float k2o_scale) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return fs_launch<X>(u, K2, k2_logC, k2_scale, D, y, batch, H, L, scratch, st, s, K2o, k2o_scale);
    S4_CASE(14) S4_CASE(15) S4_CASE(16) S4_CASE(17)
#undef S4_CASE
    default: return cudaErrorInvalidValue;
  }
}

size_t fs_spec_scratch_bytes(int logn, int H) {
  if (logn < kMinLogFourStep || logn > kMaxLogFourStep) return 0;
  return (size_t)H * ((size_t)1 << logn) * sizeof(float2);
}

// The 2M = 2^logn spectrum of K [H][L] in column order, scaled 8/(2M) (see above).
template <int LOGN>
static cudaError_t fs_spec_launch(const float2* K, float2* K2, int H, int L, float2* scratch, St st,
                                  cudaStream_t s, bool realk) {
  constexpr int LOGR = fs_log_radix(LOGN), R = 1 << LOGR, n = 1 << LOGN, m = n / R;
  const unsigned blocks = (unsigned)(((long long)H * m + kFsThreads - 1) / kFsThreads);
  {
    TimedLaunch tl("spec_fwd", s);
    fs_kfwd_kernel<LOGN><<<blocks, kFsThreads, 0, s>>>(K, scratch, H, L, realk ? 1 : 0);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // columns of m points, no padding; records the call's generation
  return launch_spectrum_rows_full(LOGN - LOGR, scratch, K2, H * R, 8.f / n, st, s);
}

cudaError_t launch_spectrum_fourstep(int logn, const float2* K, float2* K2, int H, int L, float2* scratch, St st,
                                     cudaStream_t s, bool realk) {
  switch (logn) {
    case 14: return fs_spec_launch<14>(K, K2, H, L, scratch, st, s, realk);
    case 15: return fs_spec_launch<15>(K, K2, H, L, scratch, st, s, realk);
    case 16: return fs_spec_launch<16>(K, K2, H, L, scratch, st, s, realk);
    case 17: return fs_spec_launch<17>(K, K2, H, L, scratch, st, s, realk);
    default: return cudaErrorInvalidValue;
  }
}

// Layer path: root values Khat in column order -> K (out) and the 2M spectrum in
// column order.  G and X: scratch of H M and H 2M complex values.
template <int LOGM>
static cudaError_t ks_fs_launch(const float2* Khat, float2* K, float2* K2, int H, int L, float2* G, float2* X,
                                St st, cudaStream_t s) {
  constexpr int LOGRO = fs_log_radix(LOGM + 1), RO = 1 << LOGRO;
  constexpr int M = 1 << LOGM, mi = M / kKsRadix, n = 2 * M;
  cudaError_t e = launch_ifft_rows(LOGM - 4, Khat, G, H * kKsRadix, mi, st, s);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)(((long long)H * mi + kFsThreads - 1) / kFsThreads);
  {
    TimedLaunch tl("kspec_cross", s);
    ks_cross_kernel<LOGM><<<blocks, kFsThreads, 0, s>>>(G, K, X, H, L, st);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_spectrum_rows_full(LOGM + 1 - LOGRO, X, K2, H * RO, 8.f / n, st, s);
}

cudaError_t launch_kspec_fourstep(int logM, const float2* Khat, float2* K, float2* K2, int H, int L, float2* G,
                                  float2* X, St st, cudaStream_t s) {
  switch (logM) {
    case 13: return ks_fs_launch<13>(Khat, K, K2, H, L, G, X, st, s);
    case 14: return ks_fs_launch<14>(Khat, K, K2, H, L, G, X, st, s);
    case 15: return ks_fs_launch<15>(Khat, K, K2, H, L, G, X, st, s);
    case 16: return ks_fs_launch<16>(Khat, K, K2, H, L, G, X, st, s);
    default: return cudaErrorInvalidValue;
  }
}

// Layer path, L = M: root values in column order of C = R/2 -> K (out) and the
// odd bins of its 2M spectrum, T, in column order of C, scaled 8/(2M).  G and X:
// scratch of H M complex values each.
template <int LOGM>
static cudaError_t ks_half_launch(const float2* Khat, float2* K, float2* T, int H, int L, float2* G, float2* X,
                                  St st, cudaStream_t s) {
  constexpr int LC = fs_log_radix(LOGM + 1) - 1, C = 1 << LC;
  constexpr int M = 1 << LOGM, mi = M / C, n = 2 * M;
  cudaError_t e = launch_ifft_rows(LOGM - LC, Khat, G, H * C, mi, st, s);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)(((long long)H * mi + kFsThreads - 1) / kFsThreads);
  {
    TimedLaunch tl("kspec_cross", s);
    ks_cross_half_kernel<LOGM><<<blocks, kFsThreads, 0, s>>>(G, K, X, H, L, st);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_spectrum_rows_full(LOGM - LC, X, T, H * C, 8.f / n, st, s);
}

cudaError_t launch_kspec_fourstep_half(int logM, const float2* Khat, float2* K, float2* T, int H, int L,
                                       float2* G, float2* X, St st, cudaStream_t s) {
  switch (logM) {
    case 13: return ks_half_launch<13>(Khat, K, T, H, L, G, X, st, s);
    case 14: return ks_half_launch<14>(Khat, K, T, H, L, G, X, st, s);
    case 15: return ks_half_launch<15>(Khat, K, T, H, L, G, X, st, s);
    case 16: return ks_half_launch<16>(Khat, K, T, H, L, G, X, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
