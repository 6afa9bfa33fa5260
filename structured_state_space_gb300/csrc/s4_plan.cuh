// Radix plans of the row FFTs and their launch shapes.
//
// A length-2^LOGN transform is a sequence of Stockham passes: radix 16 as
// often as it divides, then one pass of the remaining power of two.  The
// inverse runs the same radices in reverse order, so that the last forward
// pass and the first inverse pass (and the first forward / last inverse
// pass) touch the same elements in the same threads; the convolution uses
// that to keep data in registers across the spectrum product and to keep
// the input for the skip term.
#pragma once
#include "s4_dev.cuh"

namespace s4dev {

__host__ __device__ constexpr int plan_npass(int logn) { return logn == 0 ? 1 : (logn + 3) / 4; }

__host__ __device__ constexpr int plan_radix_fwd(int logn, int idx) {
  return logn == 0 ? 1 : (idx < logn / 4 ? 16 : (1 << (logn % 4)));
}

__host__ __device__ constexpr int plan_radix(int logn, int idx, bool inv) {
  return inv ? plan_radix_fwd(logn, plan_npass(logn) - 1 - idx) : plan_radix_fwd(logn, idx);
}

// Product of the radices of the passes before `idx`.
__host__ __device__ constexpr int plan_p(int logn, int idx, bool inv) {
  int p = 1;
  for (int j = 0; j < idx; ++j) p *= plan_radix(logn, j, inv);
  return p;
}

// Offset of pass idx's twiddle base table (passes 1.. have tables of P entries).
__host__ __device__ constexpr int plan_tw_off(int logn, int idx, bool inv) {
  int off = 0;
  for (int j = 1; j < idx; ++j) off += plan_p(logn, j, inv);
  return off;
}

__host__ __device__ constexpr int plan_tw_size(int logn, bool inv) {
  return plan_tw_off(logn, plan_npass(logn), inv);
}

// Threads that share one row, rows per CTA.
__host__ __device__ constexpr int row_threads(int logn) {
  return logn <= 4 ? 1 : (logn <= 12 ? (1 << (logn - 4)) : (1 << (logn - 5)));
}
__host__ __device__ constexpr int rows_per_cta(int logn) {
  return row_threads(logn) >= 128 ? 1 : 128 / row_threads(logn);
}

template <int LOGN, bool INV>
__device__ __forceinline__ void fill_plan_twiddles(float2* tw, int tid, int nth) {
#pragma unroll 1
  for (int idx = 1; idx < plan_npass(LOGN); ++idx) {
    const int P = plan_p(LOGN, idx, INV);
    fill_twiddles(tw + plan_tw_off(LOGN, idx, INV), P, P * plan_radix(LOGN, idx, INV), tid, nth);
  }
}

// Stockham passes FIRST..LAST of the plan, all in shared memory.
template <int LOGN, bool INV, int IDX, int LAST, int T>
__device__ __forceinline__ void run_passes(float2* buf, const float2* tw, int lt) {
  if constexpr (IDX <= LAST) {
    constexpr int R = plan_radix(LOGN, IDX, INV);
    constexpr int P = plan_p(LOGN, IDX, INV);
    pass_smem<(1 << LOGN), R, P, INV, T>(buf, tw + plan_tw_off(LOGN, IDX, INV), lt);
    run_passes<LOGN, INV, IDX + 1, LAST, T>(buf, tw, lt);
  }
}

}  // namespace s4dev
