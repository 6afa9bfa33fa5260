// One channel of the layer path's inverse transform + kernel spectrum:
//   K = first L of (1/M) iFFT_M(Khat)      (written out)
//   K2 = scale FFT_2M(K zero-padded to 2M)  (written out, natural order)
// from one shared-memory row of padded_len(2M) entries (the body of the
// layer path's kspec kernel).  "Recurrent, LSTM, and structured state-space
// models", filter mode (first L coefficients of the inverse radix-two
// transform) and "Roots-of-unity orthogonality and radix-two FFT cost" (zero
// padding).
#pragma once
#include "s4_fft.cuh"

namespace s4dev {

template <int LOGM>
struct KspecCfg {
  static constexpr int LOGN = LOGM + 1;
  static constexpr int M = 1 << LOGM, n = 2 * M;
  static constexpr int T = row_threads(LOGN);   // threads of the forward passes
  static constexpr int TI = row_threads(LOGM);  // threads of the inverse passes
  static constexpr int PADN = padded_len(n);
};

// Twiddle tables a kspec CTA copies into shared memory at its start (the
// inverse plan of M and the forward plan of 2M, each from pass 1 on), so that
// one copy, in flight beside the root-value loads, replaces a first-touch L2
// read in each pass.  Only where the copy is small (M <= 1024: 27 KiB) and
// does not cost resident CTAs.
__host__ __device__ constexpr bool kspec_stage_tw(int logm) { return logm <= 10; }
__host__ __device__ constexpr int kspec_tw_inv_len(int logm) {
  return tw_offset(logm, true, plan_npass(logm)) - tw_offset(logm, true, 1);
}
__host__ __device__ constexpr int kspec_tw_fwd_len(int logm) {
  return tw_offset(logm + 1, false, plan_npass(logm + 1)) - tw_offset(logm + 1, false, 1);
}
// float2 offset of the staged tables after `rows_len` entries of row buffers
// (rounded up to 16 bytes for the bulk copies)
__host__ __device__ constexpr int kspec_tw_base(int rows_len) { return (rows_len + 1) & ~1; }

// All threads with lt < nthreads_row take part in the barriers; lt >= T idle.
// `zero`: write zeros (a device-detected condition).  Khat is read through
// L2 (it may have been written by other SMs of the same grid).  With STW the
// twiddles come from the shared-memory copies twi (inverse plan of M) and twf
// (forward plan of 2M), which arrive on the mbarrier `twbar` (phase 0); a
// wait that gives up sets `stall`.
template <int LOGM, bool STW = false>
__device__ __forceinline__ void kspec_row(const float2* __restrict__ khat, float2* __restrict__ Krow,
                                          float2* __restrict__ K2row, int L, float scale, bool zero,
                                          bool act, float2* buf, int lt, bool& fin,
                                          const float2* twi = nullptr, const float2* twf = nullptr,
                                          unsigned long long* twbar = nullptr, bool* stall = nullptr,
                                          int wait_limit = kMbarWaitLimit) {
  using KC = KspecCfg<LOGM>;
  constexpr int LOGN = KC::LOGN, M = KC::M, n = KC::n, T = KC::T, TI = KC::TI;
  static_assert(TI <= T, "thread split");
  constexpr int NPI = plan_npass(LOGM);
  constexpr int RI0 = plan_radix(LOGM, 0, true), RIL = plan_radix(LOGM, NPI - 1, true);
  constexpr int NBI0 = M / RI0, PERI0 = NBI0 / TI, NBIL = M / RIL, PERIL = NBIL / TI;
  using IXI0 = PassIdx<M, RI0, 1>;
  using IXIL = PassIdx<M, RIL, M / RIL>;
  using TWIL = PassTw<LOGM, NPI - 1, true>;
  constexpr int NPF = plan_npass(LOGN), RA = plan_radix(LOGN, 0, false),
                RB = plan_radix(LOGN, NPF - 1, false);
  constexpr int NB0 = n / RA, PER0 = NB0 / T, NBL = n / RB, PERL = NBL / T;
  using IXF0 = PassIdx<n, RA, 1>;
  using IXFL = PassIdx<n, RB, n / RB>;
  using TWFL = PassTw<LOGN, NPF - 1, false>;
  static_assert(NPI >= 2 && NPF >= 2, "sizes");
  float2* const bufs[1] = {buf};
  const float sc = 1.f / M;
  if (lt < TI) {  // inverse pass 0 (P = 1): root values -> shared
#pragma unroll
    for (int s = 0; s < PERI0; ++s) {
      const int i = lt + s * TI;
      float2 a[RI0];
#pragma unroll
      for (int q = 0; q < RI0; ++q)
        a[q] = (act && S4_IN(i + q * NBI0, M)) ? __ldcg(khat + i + q * NBI0) : make_float2(0.f, 0.f);
      dft<RI0, true>(a);
#pragma unroll
      for (int q = 0; q < RI0; ++q) st_chk(buf, IXI0::wr(i, q), padded_len(n), a[q]);
    }
  }
  __syncthreads();
  if constexpr (STW) {
    if (!mbar_wait(twbar, 0u, wait_limit)) {  // tables missing: the row is written as zeros
      *stall = true;
      zero = true;
    }
  }
  passes_rows<LOGM, true, 1, NPI - 2, TI, 1, STW>(bufs, lt, twi);
  float2 kv[PERIL][RIL];
  if (lt < TI) {  // last inverse pass: K in registers
#pragma unroll
    for (int s = 0; s < PERIL; ++s) {
      const int i = lt + s * TI;
      float2 w[RIL];
#pragma unroll
      for (int q = 0; q < RIL; ++q) kv[s][q] = ld_chk(buf, IXIL::rd(i, q), padded_len(n));
      TWIL::template load<STW>(w, i, STW ? twi + TWIL::REL : nullptr);
      TWIL::apply(kv[s], w);
      dft<RIL, true>(kv[s]);
    }
  }
  __syncthreads();
  if (lt < TI) {  // K out (first L, scaled) and into shared memory, natural order
#pragma unroll
    for (int s = 0; s < PERIL; ++s) {
      const int i = lt + s * TI;
#pragma unroll
      for (int q = 0; q < RIL; ++q) {
        const int t = i + q * NBIL;
        const float2 v = (zero || t >= L) ? make_float2(0.f, 0.f) : cscale(kv[s][q], sc);
        if (act && t < L) st_chk(Krow, t, L, v);
        st_chk(buf, pad(t), padded_len(n), v);
      }
    }
  }
  __syncthreads();
  {  // forward pass 0 of the spectrum (upper half is the zero padding)
    float2 a[PER0][RA];
    if (lt < T) {
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
#pragma unroll
        for (int q = 0; q < RA / 2; ++q) a[s][q] = ld_chk(buf, pad(i + q * NB0), padded_len(n));
        dft<RA, false, true>(a[s]);
      }
    }
    __syncthreads();
    if (lt < T) {
#pragma unroll
      for (int s = 0; s < PER0; ++s) {
        const int i = lt + s * T;
#pragma unroll
        for (int q = 0; q < RA; ++q) st_chk(buf, IXF0::wr(i, q), padded_len(n), a[s][q]);
      }
    }
    __syncthreads();
  }
  passes_rows<LOGN, false, 1, NPF - 2, T, 1, STW>(bufs, lt, twf);
  if (lt < T) {
#pragma unroll
    for (int s = 0; s < PERL; ++s) {  // last forward pass -> K2
      const int i = lt + s * T;
      float2 a[RB], w[RB];
#pragma unroll
      for (int q = 0; q < RB; ++q) a[q] = ld_chk(buf, IXFL::rd(i, q), padded_len(n));
      TWFL::template load<STW>(w, i, STW ? twf + TWFL::REL : nullptr);
      TWFL::apply(a, w);
      dft<RB, false>(a);
      if (act) {
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          fin = fin && cfinite(a[q]);
          st_chk(K2row, i + q * NBL, n, cscale(a[q], scale));
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace s4dev
