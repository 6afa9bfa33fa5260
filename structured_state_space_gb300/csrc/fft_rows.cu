// Row FFT kernels whose rows fit one CTA's shared memory (length <= 16384):
//   ifft_kernel      K = first L of (1/M) iFFT_M(Khat)                (kernel generation)
//   spectrum_kernel  K2 = s FFT_{2M}(K zero-padded to 2M), s = 1/(4M)  (kernel spectrum)
//   conv_pair_kernel y = first L of iFFT_{2M}(FFT_{2M}(u) K2) + D u    (fused convolution)
//
// "Recurrent, LSTM, and structured state-space models": filter mode returns
// the first L coefficients of the inverse radix-two transform of the root
// values; "Roots-of-unity orthogonality and radix-two FFT cost": a product of
// two length-n polynomials by zero-padding to a radix-two length >= 2n - 1.
// Here both factors have length L <= M and the transforms have length n = 2M.
//
// The convolution takes two batch rows b, b+1 of one channel at a time and
// transforms them together as the real and imaginary parts of one complex
// row z = u_b + i u_{b+1}; the two spectra follow from Z and its mirror:
//   U_b[k] = (Z[k] + conj Z[n-k]) / 2,   U_{b+1}[k] = (Z[k] - conj Z[n-k]) / (2i).
// The factor 1/2 and the inverse transform's 1/n are folded into K2.
#include "s4_fft.cuh"
#include "s4_internal.h"
#include "s4_kspec.cuh"

namespace s4dev {

// ----------------------------------------------------------------------------
// Rows of length <= 16: one thread per row, the whole transform in registers.
// ----------------------------------------------------------------------------
template <int LOGN>
__global__ void __launch_bounds__(128) ifft_small_kernel(const float2* __restrict__ Khat,
                                                         float2* __restrict__ K, int H, int L,
                                                         St status) {
  constexpr int n = 1 << LOGN;
  const int h = blockIdx.x * 128 + threadIdx.x;
  if (h >= H) return;
  const bool zero = st_bad(status);
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
                                                             float scale, int realk,
                                                             St status) {
  constexpr int n = 1 << LOGN;  // n = 2M >= 2
  pdl_wait();  // (a programmatic launch) the previous kernel on the stream is done
  st_record_gen(status);  // the first kernel of a convolution call
  const int h = blockIdx.x * 128 + threadIdx.x;
  if (h >= H) return;
  float2 a[n];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    a[q] = q < L ? K[(size_t)h * L + q] : make_float2(0.f, 0.f);
    if (realk) a[q].y = 0.f;
  }
  dft<n, false, true>(a);
  bool fin = true;
#pragma unroll
  for (int q = 0; q < n; ++q) {
    fin = fin && cfinite(a[q]);
    K2[(size_t)h * n + q] = cscale(a[q], scale);
  }
  if (!fin) st_flag(status, ST_NONFINITE);
}

// rows of length n <= 16 with K2 scaled by 1/(2n): two rows per thread
template <int LOGN>
__global__ void __launch_bounds__(128) conv_small_kernel(const float* __restrict__ u,
                                                         const float2* __restrict__ K2,
                                                         const float* __restrict__ D,
                                                         float2* __restrict__ y, int batch, int H,
                                                         int L, St status) {
  constexpr int n = 1 << LOGN;  // n = 2M >= 2
  const int pairs = ((batch + 1) / 2) * H;
  const int p = blockIdx.x * 128 + threadIdx.x;
  if (p >= pairs) return;
  const int h = p % H, b0 = 2 * (p / H);
  const bool has1 = b0 + 1 < batch;
  const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
  const bool zero = st_bad(status);
  float u0[n / 2], u1[n / 2];
  float2 z[n];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    u0[q] = q < L ? u[row0 * L + q] : 0.f;
    u1[q] = (has1 && q < L) ? u[row1 * L + q] : 0.f;
    z[q] = make_float2(u0[q], u1[q]);
  }
  dft<n, false, true>(z);
  float2 a0[n], a1[n];
#pragma unroll
  for (int k = 0; k < n; ++k) {
    const float2 zp = z[(n - k) & (n - 1)];
    const float2 kv = K2[(size_t)h * n + k];
    a0[k] = cmul(make_float2(z[k].x + zp.x, z[k].y - zp.y), kv);
    a1[k] = cmul(make_float2(z[k].y + zp.y, zp.x - z[k].x), kv);
  }
  dft<n, true, false, true>(a0);
  dft<n, true, false, true>(a1);
  const float d = D[h];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    if (q < L) {
      y[row0 * L + q] = zero ? make_float2(0.f, 0.f) : make_float2(fmaf(d, u0[q], a0[q].x), a0[q].y);
      if (has1) y[row1 * L + q] = zero ? make_float2(0.f, 0.f) : make_float2(fmaf(d, u1[q], a1[q].x), a1[q].y);
    }
  }
}

// ----------------------------------------------------------------------------
// Rows of length 32 .. 16384: Stockham passes over padded shared memory.
// ----------------------------------------------------------------------------
template <int LOGN, bool CONV = false>
struct RowCfg {
  static constexpr int n = 1 << LOGN;
  static constexpr int T = CONV ? conv_row_threads(LOGN) : row_threads(LOGN);
  static constexpr int ROWS = T >= 128 ? 1 : 128 / T;
  static constexpr int THREADS = T * ROWS;
  static constexpr int NP = plan_npass(LOGN);
  static constexpr int RA = plan_radix(LOGN, 0, false);       // first forward radix
  static constexpr int RB = plan_radix(LOGN, NP - 1, false);  // last forward radix
  static constexpr int PADN = padded_len(n);
};

// Inverse transform of each channel's root values, first L outputs scaled 1/M.
template <int LOGN>
__global__ void __launch_bounds__(RowCfg<LOGN>::THREADS) ifft_kernel(
    const float2* __restrict__ Khat, float2* __restrict__ K, int H, int L,
    St status) {
  using C = RowCfg<LOGN>;
  constexpr int n = C::n, T = C::T, NP = C::NP;
  constexpr int R0 = plan_radix(LOGN, 0, true), RL = plan_radix(LOGN, NP - 1, true);
  constexpr int NB0 = n / R0, PER0 = NB0 / T, NBL = n / RL, PERL = NBL / T;
  using IX0 = PassIdx<n, R0, 1>;
  using IXL = PassIdx<n, RL, n / RL>;
  using TWL = PassTw<LOGN, NP - 1, true>;
  extern __shared__ float2 smem[];
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = smem + slot * C::PADN;
  float2* const bufs[1] = {buf};
  pdl_wait();  // (a programmatic launch) root values and status come from the previous kernel
  const bool zero = st_bad(status);
  const float sc = 1.f / n;
  for (int h0 = blockIdx.x * C::ROWS; h0 < H; h0 += gridDim.x * C::ROWS) {
    const int h = h0 + slot;
    const bool act = h < H;
#pragma unroll
    for (int s = 0; s < PER0; ++s) {  // inverse pass 0 (P = 1): global -> shared
      const int i = lt + s * T;
      float2 a[R0];
#pragma unroll
      for (int q = 0; q < R0; ++q)
        a[q] = (act && S4_IN((long long)h * n + i + q * NB0, (long long)H * n))
                   ? __ldcg(Khat + (size_t)h * n + i + q * NB0) : make_float2(0.f, 0.f);
      dft<R0, true>(a);
#pragma unroll
      for (int q = 0; q < R0; ++q) st_chk(buf, IX0::wr(i, q), C::PADN, a[q]);
    }
    __syncthreads();
    passes_rows<LOGN, true, 1, NP - 2, T, 1>(bufs, lt);
#pragma unroll
    for (int s = 0; s < PERL; ++s) {  // last inverse pass: shared -> global
      const int i = lt + s * T;
      float2 a[RL], w[RL];
#pragma unroll
      for (int q = 0; q < RL; ++q) a[q] = ld_chk(buf, IXL::rd(i, q), C::PADN);
      TWL::load(w, i);
      TWL::apply(a, w);
      dft<RL, true>(a);
#pragma unroll
      for (int q = 0; q < RL; ++q) {
        const int t = i + q * NBL;
        if (act && t < L) st_chk(K, (long long)h * L + t, (long long)H * L, zero ? make_float2(0.f, 0.f) : cscale(a[q], sc));
      }
    }
    __syncthreads();
  }
}

// Spectrum of each channel's kernel zero-padded to n = 2M, natural order, times `scale`.
// FULL: rows of n values with no padding (the column spectra of the four-step
// long-row path), every input read; one radix-16 butterfly per thread at 8192
// points (the convolution's thread count: at two per thread this form spilled).
template <int LOGN, bool FULL = false>
__global__ void __launch_bounds__(RowCfg<LOGN, FULL>::THREADS) spectrum_kernel(
    const float2* __restrict__ K, float2* __restrict__ K2, int H, int L, float scale, int realk,
    St status) {
  using C = RowCfg<LOGN, FULL>;
  constexpr int n = C::n, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  using IX0 = PassIdx<n, RA, 1>;
  using IXL = PassIdx<n, RB, n / RB>;
  using TWL = PassTw<LOGN, NP - 1, false>;
  extern __shared__ float2 smem[];
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = smem + slot * C::PADN;
  float2* const bufs[1] = {buf};
  bool fin = true;
  pdl_wait();  // (a programmatic launch) the previous kernel on the stream is done
  st_record_gen(status);  // the first kernel of a convolution call
  pdl_launch_dependents();  // the convolution may be scheduled; it waits for this grid before reading K2
  for (int h0 = blockIdx.x * C::ROWS; h0 < H; h0 += gridDim.x * C::ROWS) {
    const int h = h0 + slot;
    const bool act = h < H;
#pragma unroll
    for (int s = 0; s < PER0; ++s) {  // forward pass 0; the upper half is the zero padding
      const int i = lt + s * T;
      float2 a[RA];
#pragma unroll
      for (int q = 0; q < (FULL ? RA : RA / 2); ++q) {
        const int t = i + q * NB0;
        a[q] = (act && t < L && S4_IN((long long)h * L + t, (long long)H * L)) ? K[(size_t)h * L + t]
                                                                             : make_float2(0.f, 0.f);
        if (realk) a[q].y = 0.f;
      }
      dft<RA, false, !FULL>(a);
#pragma unroll
      for (int q = 0; q < RA; ++q) st_chk(buf, IX0::wr(i, q), C::PADN, a[q]);
    }
    __syncthreads();
    passes_rows<LOGN, false, 1, NP - 2, T, 1>(bufs, lt);
#pragma unroll
    for (int s = 0; s < PERL; ++s) {  // last forward pass: shared -> global
      const int i = lt + s * T;
      float2 a[RB], w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) a[q] = ld_chk(buf, IXL::rd(i, q), C::PADN);
      TWL::load(w, i);
      TWL::apply(a, w);
      dft<RB, false>(a);
      if (act) {
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          fin = fin && cfinite(a[q]);
          st_chk(K2, (long long)h * n + i + q * NBL, (long long)H * n, cscale(a[q], scale));
        }
      }
    }
    __syncthreads();
  }
  if (!fin) st_flag(status, ST_NONFINITE);
}

// Threads per SM the kspec kernel is compiled for (registers capped at
// 65536 / this): 512 measured ~10 % faster at M = 4096 than no cap and equal at
// M = 1024, with room left for the convolution's early CTAs.
#ifndef S4_KSPEC_THREADS_PER_SM
#define S4_KSPEC_THREADS_PER_SM 512
#endif
__host__ __device__ constexpr int kspec_min_blocks(int threads) {
  return threads >= S4_KSPEC_THREADS_PER_SM ? 1 : S4_KSPEC_THREADS_PER_SM / threads;
}

// Layer path: for each channel, K = first L of (1/M) iFFT_M(Khat) (written
// out) and, from the same shared-memory row, K2 = scale FFT_2M(K zero-padded).
// One launch instead of two, and K is not read back.  Rows of 2M <= 2^13
// points (LOGM = 5..12).
template <int LOGM>
__global__ void __launch_bounds__(RowCfg<LOGM + 1>::THREADS, kspec_min_blocks(RowCfg<LOGM + 1>::THREADS)) kspec_kernel(
    const float2* __restrict__ Khat, float2* __restrict__ K, float2* __restrict__ K2, int H, int L,
    float scale, St status, int wait_limit) {
  using C = RowCfg<LOGM + 1>;
  constexpr int M = 1 << LOGM, n = C::n, T = C::T;
  constexpr bool STW = kspec_stage_tw(LOGM);
  constexpr int TWI = kspec_tw_inv_len(LOGM), TWF = kspec_tw_fwd_len(LOGM);
  static_assert(!STW || (TWI % 2 == 0 && TWF % 2 == 0 && tw_offset(LOGM, true, 1) % 2 == 0 &&
                         tw_offset(LOGM + 1, false, 1) % 2 == 0),
                "staged tables: 16-byte aligned offsets and sizes");
  extern __shared__ __align__(16) float2 smem[];
  __shared__ unsigned long long twbar;
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = smem + slot * C::PADN;
  float2* twi = smem + kspec_tw_base(C::ROWS * C::PADN);  // STW: inverse-plan tables, then forward-plan
  float2* twf = twi + TWI;
  bool stall = false;
  if constexpr (STW) {  // the tables do not depend on the previous kernel: copy them now
    if (threadIdx.x == 0) {
      mbar_init(&twbar, 1u);
      fence_mbar_init();
      mbar_expect_tx(&twbar, (unsigned)((TWI + TWF) * sizeof(float2)));
      bulk_g2s(twi, TwTab<LOGM>::ptr() + tw_offset(LOGM, true, 1), (unsigned)(TWI * sizeof(float2)), &twbar);
      bulk_g2s(twf, TwTab<LOGM + 1>::ptr() + tw_offset(LOGM + 1, false, 1), (unsigned)(TWF * sizeof(float2)),
               &twbar);
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it
  }
  pdl_launch_dependents();
  pdl_wait();  // root values and status come from the previous kernel
  bool zero = st_bad(status);
  bool fin = true;
  for (int h0 = blockIdx.x * C::ROWS; h0 < H; h0 += gridDim.x * C::ROWS) {
    const int h = h0 + slot;
    const bool act = h < H;
    kspec_row<LOGM, STW>(Khat + (size_t)(act ? h : 0) * M, K + (size_t)(act ? h : 0) * L,
                         K2 + (size_t)(act ? h : 0) * n, L, scale, zero || stall, act, buf, lt, fin, twi,
                         twf, &twbar, &stall, wait_limit);
  }
  if (!fin) st_flag(status, ST_NONFINITE);
  if constexpr (STW) {
    if (stall) mbar_wait(&twbar, 0u);  // drain: one more wait, default limit, for the copy in flight
  }
  if (stall && threadIdx.x == 0) st_flag(status, ST_STALL);
}

// Resident CTAs per SM the convolution is compiled for: 512 threads per SM
// (4 CTAs of 128 threads, 128 registers each) measured fastest at 2M = 2048 --
// the kernel is latency-bound and occupancy beats the extra registers.  Rows
// of 8192 points take one 512-thread CTA per SM (their shared memory allows
// no second one).
#ifndef S4_CONV_THREADS_PER_SM
#define S4_CONV_THREADS_PER_SM 512
#endif
__host__ __device__ constexpr int conv_min_blocks(int logn, int threads) {
  return (logn >= 13 || threads >= S4_CONV_THREADS_PER_SM) ? 1 : S4_CONV_THREADS_PER_SM / threads;
}
// The real-output convolution holds one row buffer and one row in registers:
// 6 CTAs of 128 threads per SM (80 registers, no spills) measured 7 % faster
// than 4 at 2M = 2048, and 8 (64 registers) no faster.
#ifndef S4_CONV_REAL_THREADS_PER_SM
#define S4_CONV_REAL_THREADS_PER_SM 768
#endif
__host__ __device__ constexpr int conv_real_min_blocks(int logn, int threads) {
  return (logn >= 13 || threads >= S4_CONV_REAL_THREADS_PER_SM) ? 1 : S4_CONV_REAL_THREADS_PER_SM / threads;
}

// Butterfly index of slot `sl` of the last forward pass (and the first inverse
// pass) of a row.  With an even number of slots per thread, slot 2s takes
// butterfly s T + lt and slot 2s+1 its mirror NBL - s T - lt (thread 0 pairs
// the two self-mirrored butterflies 0 and NBL/2), so that every thread holds
// both bins k and n - k of the spectrum; otherwise slot sl is lt + sl T.
template <int T, int NBL, int PERL>
__device__ __forceinline__ int last_bfly(int sl, int lt) {
  if constexpr (PERL % 2 != 0) {
    return lt + sl * T;
  } else {
    const int s = sl >> 1;
    if ((sl & 1) == 0) return s * T + lt;
    return (s == 0 && lt == 0) ? NBL / 2 : NBL - s * T - lt;
  }
}

// Fused causal convolution, two batch rows (b, b+1) of one channel per row
// group; K2 is the channel spectrum scaled by 1/(2n).  The skip term D u is
// the convolution with D times the unit impulse, whose spectrum is D in every
// bin, so it enters as D/(2n) added to each K2 bin.
//
// STAGE (one pair per CTA, used for 2M = 8192): a third shared buffer receives, by bulk
// asynchronous copies, the channel's K2 row (requested after the first
// forward pass, used by the spectrum product) and the next pair's two input
// rows (requested once the product has read K2, used by the next forward
// pass 0), so neither global latency sits on the critical path.  Input rows
// are staged only when L is a multiple of 4 (stage_u; 16-byte copies).  A
// wait that gives up (after `wait_limit` polls) puts the CTA under the drain
// rule of mbar_wait: the vote at the next barrier makes `stall` the same in
// every thread, no copy is issued after it, staged data is read from global
// memory instead, and the round in flight is waited for once more at the end.
// The outputs are then zeros and the status is S4_ERR_TIMEOUT.
template <int LOGN, bool STAGE>
__global__ void __launch_bounds__(RowCfg<LOGN, true>::THREADS, conv_min_blocks(LOGN, RowCfg<LOGN, true>::THREADS))
conv_pair_kernel(
    const float* __restrict__ u, const float2* __restrict__ K2, const float* __restrict__ D,
    float2* __restrict__ y, int batch, int H, int L, St status, int stage_u, int wait_limit) {
  using C = RowCfg<LOGN, true>;
  constexpr int n = C::n, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  constexpr bool MIRROR = PERL % 2 == 0;
  using IXF0 = PassIdx<n, RA, 1>;        // forward pass 0 writes
  using IXFL = PassIdx<n, RB, n / RB>;   // forward last pass reads
  using IXI0 = PassIdx<n, RB, 1>;        // inverse pass 0 writes
  using IXIL = PassIdx<n, RA, n / RA>;   // inverse last pass reads
  using TWFL = PassTw<LOGN, NP - 1, false>;
  using TWIL = PassTw<LOGN, NP - 1, true>;
  extern __shared__ float2 smem[];
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* bufA = smem + slot * 2 * C::PADN;
  float2* bufB = bufA + C::PADN;
  float2* const buf1[1] = {bufA};
  float2* const buf2[2] = {bufA, bufB};
  bool zero = false, waited = false;
  const int pairs = ((batch + 1) / 2) * H;
  static_assert(!STAGE || C::ROWS == 1, "staging serves one pair per CTA");
  float2* stage = bufB + C::PADN;  // STAGE: n entries (K2 row, or input rows as floats)
  const float* stage_f = reinterpret_cast<const float*>(stage);
  __shared__ unsigned long long bar;
  unsigned ph = 0u;
  unsigned last_ph = 0u;  // parity of the latest wait: the round in flight after a stall
  bool stall = false;     // (STAGE) a wait gave up in this CTA; the same in every thread after a vote
  // one thread: announce and copy the two input rows of pair q into the stage
  auto issue_u = [&](int q) {
    const int hq = q % H, bq = 2 * (q / H);
    const unsigned bytes = (unsigned)L * 4u;
    const bool two = bq + 1 < batch;
    // (checked build: the rows fit their halves of the stage and of u)
    (void)S4_IN(L - 1, n);
    (void)S4_IN(((long long)bq * H + hq + (two ? H : 0)) * L + L - 1, (long long)batch * H * L);
    fence_proxy_async();
    mbar_expect_tx(&bar, two ? 2u * bytes : bytes);
    const size_t r0 = (size_t)bq * H + hq;
    bulk_g2s(stage, u + r0 * L, bytes, &bar);
    if (two) bulk_g2s(stage + n / 2, u + (r0 + H) * L, bytes, &bar);
  };
  auto issue_k2 = [&](const float2* src) {
    fence_proxy_async();
    mbar_expect_tx(&bar, (unsigned)(n * sizeof(float2)));
    bulk_g2s(stage, src, (unsigned)(n * sizeof(float2)), &bar);
  };
  if constexpr (STAGE) {
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1u);
      fence_mbar_init();
    }
    __syncthreads();
    if (stage_u && threadIdx.x == 0 && (int)blockIdx.x < pairs) issue_u(blockIdx.x);
  }
  for (int p0 = blockIdx.x * C::ROWS; p0 < pairs; p0 += gridDim.x * C::ROWS) {
    const int p = p0 + slot;
    const bool act = p < pairs;
    const int h = act ? p % H : 0;
    const int b0 = act ? 2 * (p / H) : 0;
    const bool has1 = act && b0 + 1 < batch;
    const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
    const float dk = act ? D[h] * (0.5f / n) : 0.f;
    const float2* K2h = K2 + (size_t)h * n;
    const bool from_stage = STAGE && stage_u && !stall;
    bool got_u = true;
    if (from_stage) {  // this pair's input rows
      got_u = mbar_wait(&bar, ph, wait_limit);
      last_ph = ph;
      ph ^= 1u;
    }
    const bool u_staged = from_stage && got_u;
    // forward pass 0: z = u_b + i u_{b+1}, zero-padded, global (or stage) -> shared
#pragma unroll
    for (int s = 0; s < PER0; ++s) {
      const int i = lt + s * T;
      float2 a[RA];
#pragma unroll
      for (int q = 0; q < RA / 2; ++q) {
        const int t = i + q * NB0;
        const long long nu = (long long)batch * H * L;
        if (u_staged)
          a[q] = make_float2((t < L && S4_IN(t, 2 * n)) ? stage_f[t] : 0.f,
                             (has1 && t < L && S4_IN(n + t, 2 * n)) ? stage_f[n + t] : 0.f);
        else
          a[q] = make_float2((act && t < L && S4_IN(row0 * L + t, nu)) ? u[row0 * L + t] : 0.f,
                             (has1 && t < L && S4_IN(row1 * L + t, nu)) ? u[row1 * L + t] : 0.f);
      }
      dft<RA, false, true>(a);
#pragma unroll
      for (int q = 0; q < RA; ++q) st_chk(bufA, IXF0::wr(i, q), C::PADN, a[q]);
    }
    if constexpr (STAGE) {
      stall = __syncthreads_or(stall || !got_u);
    } else {
      __syncthreads();
    }
    if (STAGE && waited && !stall && threadIdx.x == 0) issue_k2(K2h);  // the stage's inputs are consumed
    passes_rows<LOGN, false, 1, NP - 2, T, 1>(buf1, lt);
    if (!waited) {  // the forward transform of u needed nothing from the previous kernel
      pdl_wait();
      zero = st_bad(status);
      waited = true;
      if (STAGE && !stall && threadIdx.x == 0) issue_k2(K2h);  // K2 comes from the previous kernel
    }
    // forward last pass: Z in natural order, bin i + q NBL of butterfly i
    float2 z[PERL][RB];
#pragma unroll
    for (int sl = 0; sl < PERL; ++sl) {
      const int i = last_bfly<T, NBL, PERL>(sl, lt);
      float2 w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) z[sl][q] = ld_chk(bufA, IXFL::rd(i, q), C::PADN);
      TWFL::load(w, i);
      TWFL::apply(z[sl], w);
      dft<RB, false>(z[sl]);
    }
    // split the two spectra, multiply by K2 + D/(2n), first inverse pass (P = 1)
    // in registers; row b+1 goes to bufB at once (unused since the last
    // iteration), row b to bufA after every thread has read its last pass.
    float2 (&a0)[PERL][RB] = z;  // row b's products replace Z in place
    bool got_k = true;
    const bool k_wait = STAGE && !stall;
    if (k_wait) {  // the channel's K2 row
      got_k = mbar_wait(&bar, ph, wait_limit);
      last_ph = ph;
      ph ^= 1u;
    }
    const bool k_staged = k_wait && got_k;
    const float2* Kr = stage;
    if constexpr (MIRROR) {
#pragma unroll
      for (int s = 0; s < PERL / 2; ++s) {
        const int iA = last_bfly<T, NBL, PERL>(2 * s, lt), iB = last_bfly<T, NBL, PERL>(2 * s + 1, lt);
        float2 kA[RB], kB[RB], a1A[RB], a1B[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const long long nk = (long long)H * n, ha = (long long)h * n;
          kA[q] = !S4_IN(ha + iA + q * NBL, nk) ? make_float2(0.f, 0.f)
                  : k_staged ? ld_chk(Kr, iA + q * NBL, n) : __ldcg(K2h + iA + q * NBL);
          kB[q] = !S4_IN(ha + iB + q * NBL, nk) ? make_float2(0.f, 0.f)
                  : k_staged ? ld_chk(Kr, iB + q * NBL, n) : __ldcg(K2h + iB + q * NBL);
          kA[q].x += dk;
          kB[q].x += dk;
        }
        float2* zA = z[2 * s];
        float2* zB = z[2 * s + 1];
        if (s == 0 && lt == 0) {
          // butterflies 0 and NBL/2 are their own mirrors: bin q of 0 pairs
          // with bin -q mod RB, bin q of NBL/2 with bin RB-1-q
#pragma unroll
          for (int q = 0; q <= RB / 2; ++q) {
            const int qm = (RB - q) & (RB - 1);
            const float2 zk = zA[q], zm = zA[qm];
            split_mul(zk, zm, kA[q], zA[q], a1A[q]);
            if (qm != q) split_mul(zm, zk, kA[qm], zA[qm], a1A[qm]);
          }
#pragma unroll
          for (int q = 0; q < RB / 2; ++q) {
            const int qm = RB - 1 - q;
            const float2 zk = zB[q], zm = zB[qm];
            split_mul(zk, zm, kB[q], zB[q], a1B[q]);
            split_mul(zm, zk, kB[qm], zB[qm], a1B[qm]);
          }
        } else {  // bin q of iA pairs with bin RB-1-q of iB
#pragma unroll
          for (int q = 0; q < RB; ++q) {
            const int qm = RB - 1 - q;
            const float2 zk = zA[q], zm = zB[qm];
            split_mul(zk, zm, kA[q], zA[q], a1A[q]);
            split_mul(zm, zk, kB[qm], zB[qm], a1B[qm]);
          }
        }
        dft<RB, true>(a1A);
        dft<RB, true>(a1B);
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          st_chk(bufB, IXI0::wr(iA, q), C::PADN, a1A[q]);
          st_chk(bufB, IXI0::wr(iB, q), C::PADN, a1B[q]);
        }
        dft<RB, true>(zA);
        dft<RB, true>(zB);
      }
      if constexpr (STAGE) {
        stall = __syncthreads_or(stall || !got_k);
      } else {
        __syncthreads();
      }
      if (STAGE && stage_u && !stall && threadIdx.x == 0 && p0 + (int)gridDim.x < pairs) issue_u(p0 + gridDim.x);
    } else {
      // one butterfly per thread: the mirror bins sit in another thread
#pragma unroll
      for (int sl = 0; sl < PERL; ++sl) {
        const int i = last_bfly<T, NBL, PERL>(sl, lt);
#pragma unroll
        for (int q = 0; q < RB; ++q) st_chk(bufB, IXFL::rd(i, q), C::PADN, z[sl][q]);
      }
      __syncthreads();
      float2 a1[PERL][RB];
#pragma unroll
      for (int sl = 0; sl < PERL; ++sl) {
        const int i = last_bfly<T, NBL, PERL>(sl, lt);
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int k = i + q * NBL;
          float2 kv = !S4_IN((long long)h * n + k, (long long)H * n) ? make_float2(0.f, 0.f)
                      : k_staged ? ld_chk(Kr, k, n) : __ldcg(K2h + k);
          kv.x += dk;
          split_mul(z[sl][q], ld_chk(bufB, pad((n - k) & (n - 1)), C::PADN), kv, a0[sl][q], a1[sl][q]);
        }
        dft<RB, true>(a0[sl]);
        dft<RB, true>(a1[sl]);
      }
      if constexpr (STAGE) {
        stall = __syncthreads_or(stall || !got_k);
      } else {
        __syncthreads();
      }
      if (STAGE && stage_u && !stall && threadIdx.x == 0 && p0 + (int)gridDim.x < pairs) issue_u(p0 + gridDim.x);
#pragma unroll
      for (int sl = 0; sl < PERL; ++sl) {
        const int i = last_bfly<T, NBL, PERL>(sl, lt);
#pragma unroll
        for (int q = 0; q < RB; ++q) st_chk(bufB, IXI0::wr(i, q), C::PADN, a1[sl][q]);
      }
    }
    if (stall) zero = true;
#pragma unroll
    for (int sl = 0; sl < PERL; ++sl) {
      const int i = last_bfly<T, NBL, PERL>(sl, lt);
#pragma unroll
      for (int q = 0; q < RB; ++q) st_chk(bufA, IXI0::wr(i, q), C::PADN, a0[sl][q]);
    }
    __syncthreads();
    passes_rows<LOGN, true, 1, NP - 2, T, 2>(buf2, lt);
    // last inverse pass: first L outputs of both rows
#pragma unroll
    for (int s = 0; s < PER0; ++s) {
      const int i = lt + s * T;
      float2 c0[RA], c1[RA], w[RA];
#pragma unroll
      for (int q = 0; q < RA; ++q) {
        c0[q] = ld_chk(bufA, IXIL::rd(i, q), C::PADN);
        c1[q] = ld_chk(bufB, IXIL::rd(i, q), C::PADN);
      }
      TWIL::load(w, i);
      TWIL::apply(c0, w);
      TWIL::apply(c1, w);
      dft<RA, true, false, true>(c0);
      dft<RA, true, false, true>(c1);
#pragma unroll
      for (int q = 0; q < RA / 2; ++q) {
        const int t = i + q * NB0;
        const long long ny = (long long)batch * H * L;
        if (t < L) {
          if (act && S4_IN(row0 * L + t, ny)) __stcs(y + row0 * L + t, zero ? make_float2(0.f, 0.f) : c0[q]);
          if (has1 && S4_IN(row1 * L + t, ny)) __stcs(y + row1 * L + t, zero ? make_float2(0.f, 0.f) : c1[q]);
        }
      }
    }
    __syncthreads();
  }
  if constexpr (STAGE) {
    if (stall) mbar_wait(&bar, last_ph);  // drain: the round in flight, default limit
  }
  if (stall && threadIdx.x == 0) st_flag(status, ST_STALL);
}

// Real-output convolution y = Re(K) * u + D u.  K2 = FFT_n(Re K zero-padded)/n
// is Hermitian, so with z = u_b + i u_{b+1} the product Z K2 transforms back
// to y_b + i y_{b+1}: one forward and one inverse transform per pair of rows.
// The row kernel adds the skip term as D/n to every K2 bin (the spectrum of
// D times the unit impulse).
template <int LOGN>
__global__ void __launch_bounds__(128) conv_real_small_kernel(const float* __restrict__ u,
                                                              const float2* __restrict__ K2,
                                                              const float* __restrict__ D,
                                                              float* __restrict__ y, int batch, int H,
                                                              int L, St status) {
  constexpr int n = 1 << LOGN;
  const int pairs = ((batch + 1) / 2) * H;
  const int p = blockIdx.x * 128 + threadIdx.x;
  if (p >= pairs) return;
  const int h = p % H, b0 = 2 * (p / H);
  const bool has1 = b0 + 1 < batch;
  const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
  const bool zero = st_bad(status);
  float u0[n / 2], u1[n / 2];
  float2 z[n];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    u0[q] = q < L ? u[row0 * L + q] : 0.f;
    u1[q] = (has1 && q < L) ? u[row1 * L + q] : 0.f;
    z[q] = make_float2(u0[q], u1[q]);
  }
  dft<n, false, true>(z);
#pragma unroll
  for (int k = 0; k < n; ++k) z[k] = cmul(z[k], K2[(size_t)h * n + k]);
  dft<n, true, false, true>(z);
  const float d = D[h];
#pragma unroll
  for (int q = 0; q < n / 2; ++q) {
    if (q < L) {
      y[row0 * L + q] = zero ? 0.f : fmaf(d, u0[q], z[q].x);
      if (has1) y[row1 * L + q] = zero ? 0.f : fmaf(d, u1[q], z[q].y);
    }
  }
}

template <int LOGN>
__global__ void __launch_bounds__(RowCfg<LOGN, true>::THREADS, conv_real_min_blocks(LOGN, RowCfg<LOGN, true>::THREADS))
conv_real_pair_kernel(const float* __restrict__ u, const float2* __restrict__ K2,
                      const float* __restrict__ D, float* __restrict__ y, int batch, int H, int L,
                      St status) {
  using C = RowCfg<LOGN, true>;
  constexpr int n = C::n, T = C::T, NP = C::NP, RA = C::RA, RB = C::RB;
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  using IXF0 = PassIdx<n, RA, 1>;
  using IXFL = PassIdx<n, RB, n / RB>;
  using IXI0 = PassIdx<n, RB, 1>;
  using IXIL = PassIdx<n, RA, n / RA>;
  using TWFL = PassTw<LOGN, NP - 1, false>;
  using TWIL = PassTw<LOGN, NP - 1, true>;
  extern __shared__ float2 smem[];
  const int slot = threadIdx.x / T, lt = threadIdx.x % T;
  float2* buf = smem + slot * C::PADN;
  float2* const bufs[1] = {buf};
  bool zero = false, waited = false;
  const int pairs = ((batch + 1) / 2) * H;
  for (int p0 = blockIdx.x * C::ROWS; p0 < pairs; p0 += gridDim.x * C::ROWS) {
    const int p = p0 + slot;
    const bool act = p < pairs;
    const int h = act ? p % H : 0;
    const int b0 = act ? 2 * (p / H) : 0;
    const bool has1 = act && b0 + 1 < batch;
    const size_t row0 = (size_t)b0 * H + h, row1 = row0 + H;
    const float dk = act ? D[h] * (1.f / n) : 0.f;  // skip term: D/n in every bin
#pragma unroll
    for (int s = 0; s < PER0; ++s) {  // forward pass 0: z = u_b + i u_{b+1}, zero-padded
      const int i = lt + s * T;
      float2 a[RA];
#pragma unroll
      for (int q = 0; q < RA / 2; ++q) {
        const int t = i + q * NB0;
        a[q] = make_float2((act && t < L) ? u[row0 * L + t] : 0.f, (has1 && t < L) ? u[row1 * L + t] : 0.f);
      }
      dft<RA, false, true>(a);
#pragma unroll
      for (int q = 0; q < RA; ++q) buf[IXF0::wr(i, q)] = a[q];
    }
    __syncthreads();
    passes_rows<LOGN, false, 1, NP - 2, T, 1>(bufs, lt);
    if (!waited) {  // (a programmatic launch) K2 and the status come from the previous kernel
      pdl_wait();
      zero = st_bad(status);
      waited = true;
    }
    float2 a[PERL][RB];
#pragma unroll
    for (int s = 0; s < PERL; ++s) {  // last forward pass, product, first inverse pass
      const int i = lt + s * T;
      float2 w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) a[s][q] = buf[IXFL::rd(i, q)];
      TWFL::load(w, i);
      TWFL::apply(a[s], w);
      dft<RB, false>(a[s]);
#pragma unroll
      for (int q = 0; q < RB; ++q) {
        float2 kv = __ldcg(K2 + (size_t)h * n + i + q * NBL);
        kv.x += dk;
        a[s][q] = cmul(a[s][q], kv);
      }
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
    passes_rows<LOGN, true, 1, NP - 2, T, 1>(bufs, lt);
#pragma unroll
    for (int s = 0; s < PER0; ++s) {  // last inverse pass: y_b = Re, y_{b+1} = Im
      const int i = lt + s * T;
      float2 c[RA], w[RA];
#pragma unroll
      for (int q = 0; q < RA; ++q) c[q] = buf[IXIL::rd(i, q)];
      TWIL::load(w, i);
      TWIL::apply(c, w);
      dft<RA, true, false, true>(c);
#pragma unroll
      for (int q = 0; q < RA / 2; ++q) {
        const int t = i + q * NB0;
        if (t < L) {
          if (act) __stcs(y + row0 * L + t, zero ? 0.f : c[q].x);
          if (has1) __stcs(y + row1 * L + t, zero ? 0.f : c[q].y);
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace s4dev

// ----------------------------------------------------------------------------
// Host launchers
// ----------------------------------------------------------------------------
namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_rows)
#endif

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

// Launch with the programmatic-serialization attribute when `pdl` is set:
// the kernel may start before the previous kernel on the stream finishes and
// synchronises with it through pdl_wait().  Such a kernel is running while
// its predecessor writes, so it reads the predecessor's output through L2
// (__ldcg, or bulk copies), never through the non-coherent read-only path
// (__ldg): an SM's L1 may still hold that region from an earlier kernel.
template <typename... KArgs, typename... Args>
static cudaError_t launch_maybe_pdl(void (*kern)(KArgs...), int grid, int threads, size_t smem,
                                    cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int LOGN>
static cudaError_t ifft_launch(const float2* Khat, float2* K, int H, int L, St st,
                               cudaStream_t s) {
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("ifft", s);
    ifft_small_kernel<LOGN><<<(H + 127) / 128, 128, 0, s>>>(Khat, K, H, L, st);
  } else {
    using C = RowCfg<LOGN>;
    const size_t smem = sizeof(float2) * (size_t)C::ROWS * C::PADN;
    auto k = ifft_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (H + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("ifft", s);
    return launch_maybe_pdl(k, grid, C::THREADS, smem, s, true, Khat, K, H, L, st);
  }
  return cudaGetLastError();
}

template <int LOGN>
static cudaError_t spectrum_launch(const float2* K, float2* K2, int H, int L, St st,
                                   cudaStream_t s, bool realk, bool pdl) {
  // 1/(2n): pair split and inverse scaling; 1/n for the real-kernel variant (no split)
  const float scale = realk ? 1.f / (float)(1 << LOGN) : 1.f / (float)(2 << LOGN);
  const int rk = realk ? 1 : 0;
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("spectrum", s);
    spectrum_small_kernel<LOGN><<<(H + 127) / 128, 128, 0, s>>>(K, K2, H, L, scale, rk, st);
  } else {
    using C = RowCfg<LOGN>;
    const size_t smem = sizeof(float2) * (size_t)C::ROWS * C::PADN;
    auto k = spectrum_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (H + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("spectrum", s);
    return launch_maybe_pdl(k, grid, C::THREADS, smem, s, pdl, K, K2, H, L, scale, rk, st);
  }
  return cudaGetLastError();
}

template <int LOGN>
static cudaError_t conv_launch(const float* u, const float2* K2, const float* D, float2* y, int batch,
                               int H, int L, St st, cudaStream_t s, bool pdl) {
  const int pairs = ((batch + 1) / 2) * H;
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("conv", s);
    conv_small_kernel<LOGN><<<(pairs + 127) / 128, 128, 0, s>>>(u, K2, D, y, batch, H, L, st);
  } else {
    using C = RowCfg<LOGN, true>;
    // bulk-copy staging where one CTA (one pair) runs per SM, 2M = 8192: the
    // kernel is latency bound there and staging measured 5 % faster; at 2M =
    // 2048 (4 CTAs per SM) the third buffer cost more than it saved (the L1
    // share of each SM shrinks with the shared-memory carve-out)
    constexpr bool STAGE = C::ROWS == 1 && LOGN == 13;
    const size_t smem = sizeof(float2) * (2 * (size_t)C::ROWS * C::PADN + (STAGE ? (size_t)C::n : 0));
    auto k = conv_pair_kernel<LOGN, STAGE>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (pairs + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("conv", s);
    return launch_maybe_pdl(k, grid, C::THREADS, smem, s, pdl, u, K2, D, y, batch, H, L,
                            st, (L % 4 == 0) ? 1 : 0, wait_limit());
  }
  return cudaGetLastError();
}

template <int LOGM>
static cudaError_t kspec_launch(const float2* Khat, float2* K, float2* K2, int H, int L, St st,
                                cudaStream_t s) {
  using C = RowCfg<LOGM + 1>;
  const float scale = 1.f / (float)(4 << LOGM);  // 1/(2n), n = 2M
  const size_t smem = sizeof(float2) * (kspec_stage_tw(LOGM) ? (size_t)kspec_tw_base(C::ROWS * C::PADN) +
                                                                  kspec_tw_inv_len(LOGM) + kspec_tw_fwd_len(LOGM)
                                                            : (size_t)C::ROWS * C::PADN);
  auto k = kspec_kernel<LOGM>;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(k, C::THREADS, smem, (H + C::ROWS - 1) / C::ROWS);
  TimedLaunch tl("kspec", s);
  return launch_maybe_pdl(k, grid, C::THREADS, smem, s, true, Khat, K, K2, H, L, scale, st, wait_limit());
}

bool kspec_supported(int logM) { return logM >= 5 && logM <= 12; }

cudaError_t launch_kspec_rows(int logM, const float2* Khat, float2* K, float2* K2, int H, int L,
                              St st, cudaStream_t s) {
  switch (logM) {
    case 5: return kspec_launch<5>(Khat, K, K2, H, L, st, s);
    case 6: return kspec_launch<6>(Khat, K, K2, H, L, st, s);
    case 7: return kspec_launch<7>(Khat, K, K2, H, L, st, s);
    case 8: return kspec_launch<8>(Khat, K, K2, H, L, st, s);
    case 9: return kspec_launch<9>(Khat, K, K2, H, L, st, s);
    case 10: return kspec_launch<10>(Khat, K, K2, H, L, st, s);
    case 11: return kspec_launch<11>(Khat, K, K2, H, L, st, s);
    case 12: return kspec_launch<12>(Khat, K, K2, H, L, st, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int LOGN>
static cudaError_t conv_real_launch(const float* u, const float2* K2, const float* D, float* y,
                                    int batch, int H, int L, St st, cudaStream_t s, bool pdl) {
  const int pairs = ((batch + 1) / 2) * H;
  if constexpr (LOGN <= 4) {
    TimedLaunch tl("conv_real", s);
    conv_real_small_kernel<LOGN><<<(pairs + 127) / 128, 128, 0, s>>>(u, K2, D, y, batch, H, L, st);
  } else {
    using C = RowCfg<LOGN, true>;
    const size_t smem = sizeof(float2) * (size_t)C::ROWS * C::PADN;
    auto k = conv_real_pair_kernel<LOGN>;
    cudaError_t e = prepare(k, smem);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(k, C::THREADS, smem, (pairs + C::ROWS - 1) / C::ROWS);
    TimedLaunch tl("conv_real", s);
    return launch_maybe_pdl(k, grid, C::THREADS, smem, s, pdl, u, K2, D, y, batch, H, L, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_conv_real_rows(int logn, const float* u, const float2* K2, const float* D, float* y,
                                  int batch, int H, int L, St st, cudaStream_t s, bool pdl) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return conv_real_launch<X>(u, K2, D, y, batch, H, L, st, s, pdl);
    S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_ifft_rows(int logM, const float2* Khat, float2* K, int H, int L,
                             St st, cudaStream_t s) {
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

cudaError_t launch_spectrum_rows(int logn, const float2* K, float2* K2, int H, int L, St st,
                                 cudaStream_t s, bool realk, bool pdl) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return spectrum_launch<X>(K, K2, H, L, st, s, realk, pdl);
    S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

template <int LOGN>
static cudaError_t spectrum_full_launch(const float2* X, float2* K2, int rows, float scale, St st,
                                        cudaStream_t s) {
  using C = RowCfg<LOGN, true>;
  const size_t smem = sizeof(float2) * (size_t)C::ROWS * C::PADN;
  auto k = spectrum_kernel<LOGN, true>;
  cudaError_t e = prepare(k, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_for(k, C::THREADS, smem, (rows + C::ROWS - 1) / C::ROWS);
  TimedLaunch tl("spectrum", s);
  return launch_maybe_pdl(k, grid, C::THREADS, smem, s, false, X, K2, rows, 1 << LOGN, scale, 0, st);
}

cudaError_t launch_spectrum_rows_full(int logn, const float2* X, float2* K2, int rows, float scale, St st,
                                      cudaStream_t s) {
  switch (logn) {
    case 10: return spectrum_full_launch<10>(X, K2, rows, scale, st, s);
    case 11: return spectrum_full_launch<11>(X, K2, rows, scale, st, s);
    case 12: return spectrum_full_launch<12>(X, K2, rows, scale, st, s);
    case 13: return spectrum_full_launch<13>(X, K2, rows, scale, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_conv_rows(int logn, const float* u, const float2* K2, const float* D, float2* y,
                             int batch, int H, int L, St st, cudaStream_t s, bool pdl) {
  switch (logn) {
#define S4_CASE(X) \
  case X:          \
    return conv_launch<X>(u, K2, D, y, batch, H, L, st, s, pdl);
    S4_CASE(1) S4_CASE(2) S4_CASE(3) S4_CASE(4) S4_CASE(5) S4_CASE(6) S4_CASE(7)
    S4_CASE(8) S4_CASE(9) S4_CASE(10) S4_CASE(11) S4_CASE(12) S4_CASE(13)
#undef S4_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
