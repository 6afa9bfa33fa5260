// Small dense solves shared by the recurrent-mode kernels: complex helpers,
// group sums by shuffles, in-register Gauss-Jordan inversion, and the
// diagonal d_j = 1 - (Delta/2) lambda_j of the bilinear matrix G = I -
// (Delta/2) A ("Recurrent, LSTM, and structured state-space models", section
// "DPLR structured state-space parameterization", recurrent mode).
#pragma once
#include "s4_dev.cuh"

namespace s4dev {

__device__ __forceinline__ float2 cconj(float2 a) { return make_float2(a.x, -a.y); }

__device__ __forceinline__ float2 cdiv_safe(float2 a, float2 b) {  // a / b, b != 0
  const float s = __fdiv_rn(1.f, fmaf(b.x, b.x, b.y * b.y));
  return make_float2((a.x * b.x + a.y * b.y) * s, (a.y * b.x - a.x * b.y) * s);
}

// Sum over the G lanes of a group (G = 16 or 32; every lane of the warp
// takes part, offsets below G stay inside the group).
template <int G = 32>
__device__ __forceinline__ float2 warp_sum(float2 v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  return v;
}

// Invert an r x r complex matrix in place (Gauss-Jordan, partial pivoting).
// Returns false on an exactly zero pivot.
template <int R>
__device__ bool invert_small(float2 (&A)[R][R]) {
  float2 I[R][R];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j) I[i][j] = make_float2(i == j ? 1.f : 0.f, 0.f);
#pragma unroll
  for (int c = 0; c < R; ++c) {
    int piv = c;
    float best = fmaxf(fabsf(A[c][c].x), fabsf(A[c][c].y));
#pragma unroll
    for (int i = c + 1; i < R; ++i) {
      const float m = fmaxf(fabsf(A[i][c].x), fabsf(A[i][c].y));
      if (m > best) { best = m; piv = i; }
    }
    if (!(best > 0.f)) return false;
#pragma unroll
    for (int i = c + 1; i < R; ++i)
      if (i == piv)
#pragma unroll
        for (int j = 0; j < R; ++j) {
          float2 t = A[c][j]; A[c][j] = A[i][j]; A[i][j] = t;
          t = I[c][j]; I[c][j] = I[i][j]; I[i][j] = t;
        }
    const float2 inv = cdiv_safe(make_float2(1.f, 0.f), A[c][c]);
#pragma unroll
    for (int j = 0; j < R; ++j) { A[c][j] = cmul(A[c][j], inv); I[c][j] = cmul(I[c][j], inv); }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (i == c) continue;
      const float2 f = A[i][c];
#pragma unroll
      for (int j = 0; j < R; ++j) { A[i][j] = csub(A[i][j], cmul(f, A[c][j])); I[i][j] = csub(I[i][j], cmul(f, I[c][j])); }
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j) A[i][j] = I[i][j];
  return true;
}

// d_j = 1 - alpha lambda_j in fp32, the same arithmetic wherever the branch
// between the Woodbury and the bordered solve is decided.
__device__ __forceinline__ float2 dpl_diag(float2 lam, float alpha) {
  return make_float2(fmaf(-alpha, lam.x, 1.f), -alpha * lam.y);
}

}  // namespace s4dev
