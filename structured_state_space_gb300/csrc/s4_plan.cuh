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

// ---- static twiddle tables (generated at build time, see gen_twiddles.py) ----
// Pass idx >= 1 of a plan either reads its R-1 factors w^(k q) from a
// column-major block ("rows": P <= 256, R > 2; float4 v of butterfly k,
// holding w^(k(2v+1)) and w^(k(2v+2)), at float4 index v P + k, so that a
// warp's consecutive k read consecutive 16-byte words) or the single base
// factor w^k from which it builds the powers.
__host__ __device__ constexpr bool tw_is_rows(int P, int R) { return P <= 256 && R > 2; }
__host__ __device__ constexpr int tw_pass_size(int logn, int idx, bool inv) {
  return idx < 1 ? 0
                 : (tw_is_rows(plan_p(logn, idx, inv), plan_radix(logn, idx, inv))
                        ? plan_p(logn, idx, inv) * plan_radix(logn, idx, inv)
                        : plan_p(logn, idx, inv));
}
// Offset of pass idx's table in the per-length array: forward passes first.
__host__ __device__ constexpr int tw_offset(int logn, bool inv, int idx) {
  int off = 0;
  if (inv)
    for (int j = 1; j < plan_npass(logn); ++j) off += tw_pass_size(logn, j, false);
  for (int j = 1; j < idx; ++j) off += tw_pass_size(logn, j, inv);
  return off;
}
__host__ __device__ constexpr int tw_total(int logn) { return tw_offset(logn, true, plan_npass(logn)); }

// Threads that share one row (RowCfg packs 128 / that many rows into a CTA when below 128).
__host__ __device__ constexpr int row_threads(int logn) {
  return logn <= 4 ? 1 : (logn <= 12 ? (1 << (logn - 4)) : (1 << (logn - 5)));
}
// The paired convolution kernels give 8192-point rows one thread per radix-16
// butterfly (512 threads): they run one CTA per SM there, and the extra warps
// hide latency (measured faster; the other kernels of that length are not).
__host__ __device__ constexpr int conv_row_threads(int logn) {
  return logn == 13 ? 512 : row_threads(logn);
}

}  // namespace s4dev
