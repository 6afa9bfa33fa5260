// Stockham FFT passes over rows in padded shared memory, with twiddle
// factors read from the static tables generated at build time.
#pragma once
#include "s4_plan.cuh"
#include "s4_twiddles.cuh"

namespace s4dev {

__device__ __forceinline__ float2 cmul_conj(float2 a, float2 w) {  // a * conj(w)
  return make_float2(fmaf(a.x, w.x, a.y * w.y), fmaf(a.y, w.x, -a.x * w.y));
}

// Padded shared-memory offsets of one Stockham pass (N points, radix R,
// P = product of earlier radices).  Reads x[i + q N/R]; writes
// x[(i - k) R + k + q P], k = i mod P.  When the stride is a multiple of 16
// the padding splits into a per-thread base plus a constant per q.
template <int N, int R, int P>
struct PassIdx {
  static constexpr int NB = N / R;
  __device__ __forceinline__ static int rd(int i, int q) {
    if constexpr (NB % 16 == 0) return pad(i) + q * (NB + NB / 16);
    else return pad(i + q * NB);
  }
  __device__ __forceinline__ static int wr(int i, int q) {
    const int k = i & (P - 1);
    const int j0 = (i - k) * R + k;
    if constexpr (P % 16 == 0) return pad(j0) + q * (P + P / 16);
    else return pad(j0 + q * P);
  }
};

// Build-time tuning: read only the first two powers of a butterfly's factors
// from the "rows" tables and form the others by products (1), or read all (0),
// for passes with at least S4_TW_LIGHT_MINP butterfly indices P.  A quarter of
// the table's bytes stays hot in L1 at the price of R - 3 complex products; on
// GB300 the row kernels gained 3-8 % from it (inverse transforms of 4096
// points 185.8 -> 175.0 us on N=256 H=1024 L=65536), the 4096-point column
// kernel only for its P = 256 passes (1140 -> 1115 us; with every pass light the
// 2048-point columns lost 4 %).
#ifndef S4_TW_LIGHT
#define S4_TW_LIGHT 1
#endif
#ifndef S4_TW_LIGHT_MINP
#define S4_TW_LIGHT_MINP 1
#endif

// Twiddle factors of pass IDX for butterfly k, applied to a[1..R-1]
// (conjugated for an inverse pass).  `w` is filled from the table first so
// several rows that share the butterfly index can reuse it.  With SMEM the
// table is read from a shared-memory copy `sm` of this pass's table.
template <int LOGN, int IDX, bool INV>
struct PassTw {
  static constexpr int R = plan_radix(LOGN, IDX, INV);
  static constexpr int P = plan_p(LOGN, IDX, INV);
  static constexpr bool ROWS = tw_is_rows(P, R);
  __device__ __forceinline__ static const float2* table() {
    return TwTab<LOGN>::ptr() + tw_offset(LOGN, INV, IDX);
  }
  // offset of this pass's table from the plan's pass-1 table
  static constexpr int REL = tw_offset(LOGN, INV, IDX) - tw_offset(LOGN, INV, 1);
  // w[q] = w^(k q) for q = 1..R-1
  template <bool SMEM = false>
  __device__ __forceinline__ static void load(float2 (&w)[R], int k, const float2* sm = nullptr) {
    if constexpr (ROWS && S4_TW_LIGHT && !SMEM && R > 4 && P >= S4_TW_LIGHT_MINP) {
      // the first word of butterfly k's entry (w^k, w^2k), the other powers by products
      const float4 t = __ldg(reinterpret_cast<const float4*>(table()) + k);
      w[1] = make_float2(t.x, t.y);
      w[2] = make_float2(t.z, t.w);
#pragma unroll
      for (int q = 3; q < R; ++q) {
        const int hb = highbit(q);
        w[q] = (hb == q) ? cmul(w[q / 2], w[q / 2]) : cmul(w[hb], w[q - hb]);
      }
    } else if constexpr (ROWS) {
      const float4* col = reinterpret_cast<const float4*>(SMEM ? sm : table()) + k;
#pragma unroll
      for (int v = 0; v < R / 2; ++v) {
        const float4 t = SMEM ? col[v * P] : __ldg(col + v * P);
        w[1 + 2 * v] = make_float2(t.x, t.y);
        if (2 + 2 * v < R) w[2 + 2 * v] = make_float2(t.z, t.w);
      }
    } else {
      w[1] = SMEM ? sm[k] : __ldg(table() + k);
#pragma unroll
      for (int q = 2; q < R; ++q) {
        const int hb = highbit(q);
        w[q] = (hb == q) ? cmul(w[q / 2], w[q / 2]) : cmul(w[hb], w[q - hb]);
      }
    }
  }
  __device__ __forceinline__ static void apply(float2* a, const float2 (&w)[R]) {
#pragma unroll
    for (int q = 1; q < R; ++q) a[q] = INV ? cmul_conj(a[q], w[q]) : cmul(a[q], w[q]);
  }
};

// One shared-memory Stockham pass of the plan, over NR rows that share the
// thread layout (buffers bufs[0..NR-1]); T threads per row group do the work
// (threads with lt >= T only take part in the barriers).  With STW the
// twiddles come from `twsm`, a shared-memory copy of the plan's tables from
// pass 1 on.
template <int LOGN, int IDX, bool INV, int T, int NR, bool STW = false>
__device__ __forceinline__ void pass_rows(float2* const* bufs, int lt, const float2* twsm = nullptr) {
  constexpr int N = 1 << LOGN;
  constexpr int R = plan_radix(LOGN, IDX, INV), P = plan_p(LOGN, IDX, INV);
  constexpr int NB = N / R, PER = NB / T;
  static_assert(NB % T == 0, "pass layout");
  using IX = PassIdx<N, R, P>;
  using TW = PassTw<LOGN, IDX, INV>;
  const bool work = lt < T;
  float2 a[NR][PER][R];
  if (work) {
#pragma unroll
  for (int s = 0; s < PER; ++s) {
    const int i = lt + s * T;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int q = 0; q < R; ++q) a[r][s][q] = ld_chk(bufs[r], IX::rd(i, q), padded_len(N));
    if constexpr (P > 1) {
      float2 w[R];
      TW::template load<STW>(w, i & (P - 1), STW ? twsm + TW::REL : nullptr);
#pragma unroll
      for (int r = 0; r < NR; ++r) TW::apply(a[r][s], w);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) dft<R, INV>(a[r][s]);
  }
  }
  __syncthreads();
  if (work) {
#pragma unroll
  for (int s = 0; s < PER; ++s) {
    const int i = lt + s * T;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int q = 0; q < R; ++q) st_chk(bufs[r], IX::wr(i, q), padded_len(N), a[r][s][q]);
  }
  }
  __syncthreads();
}

template <int LOGN, bool INV, int IDX, int LAST, int T, int NR, bool STW = false>
__device__ __forceinline__ void passes_rows(float2* const* bufs, int lt, const float2* twsm = nullptr) {
  if constexpr (IDX <= LAST) {
    pass_rows<LOGN, IDX, INV, T, NR, STW>(bufs, lt, twsm);
    passes_rows<LOGN, INV, IDX + 1, LAST, T, NR, STW>(bufs, lt, twsm);
  }
}

}  // namespace s4dev
