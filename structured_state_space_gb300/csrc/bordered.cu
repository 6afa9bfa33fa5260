// The bordered branch of the recurrent mode's solver, for channels whose
// bilinear diagonal d_j = 1 - (Delta/2) lambda_j is exactly zero somewhere.
//
// "Recurrent, LSTM, and structured state-space models", section "DPLR
// structured state-space parameterization", recurrent mode: with J the states
// where d_j != 0 and Z the others (s = |Z|), the step's solve G x = b becomes,
// when s <= r, the (r + s)-square bordered system for (Q^* x, x_Z) with
// x_J = D_J^{-1}(b_J - (Delta/2) P_J Q^* x); s > r, or a singular bordered
// matrix, is the status singular-bilinear-matrix.  The same system with
// conjugated diagonal and P, Q exchanged solves G^* for the truncated output
// vector C~ = (I - Abar^M)^* C.
//
// These kernels run after the recurrent / C~ kernels of recurrent.cu, which
// leave such channels alone (both sides decide with the same fp32 test of d_j);
// every other warp returns after reading its channel's diagonal.
#include <float.h>

#include "s4_dev.cuh"
#include "s4_internal.h"
#include "s4_solve.cuh"

namespace s4dev {

// Gauss-Jordan inversion with partial pivoting of an n x n complex matrix in
// local memory: a once-per-warp step of a rare branch, kept as plain loops.
// Returns false on an exactly zero pivot.
template <int NN>
__device__ __noinline__ bool invert_local(float2 (&A)[NN][NN]) {
  float2 I[NN][NN];
#pragma unroll 1
  for (int i = 0; i < NN; ++i)
#pragma unroll 1
    for (int j = 0; j < NN; ++j) I[i][j] = make_float2(i == j ? 1.f : 0.f, 0.f);
#pragma unroll 1
  for (int c = 0; c < NN; ++c) {
    int piv = c;
    float best = fmaxf(fabsf(A[c][c].x), fabsf(A[c][c].y));
#pragma unroll 1
    for (int i = c + 1; i < NN; ++i) {
      const float m = fmaxf(fabsf(A[i][c].x), fabsf(A[i][c].y));
      if (m > best) {
        best = m;
        piv = i;
      }
    }
    if (!(best > 0.f)) return false;
    if (piv != c) {
#pragma unroll 1
      for (int j = 0; j < NN; ++j) {
        float2 t = A[c][j];
        A[c][j] = A[piv][j];
        A[piv][j] = t;
        t = I[c][j];
        I[c][j] = I[piv][j];
        I[piv][j] = t;
      }
    }
    const float2 inv = cdiv_safe(make_float2(1.f, 0.f), A[c][c]);
#pragma unroll 1
    for (int j = 0; j < NN; ++j) {
      A[c][j] = cmul(A[c][j], inv);
      I[c][j] = cmul(I[c][j], inv);
    }
#pragma unroll 1
    for (int i = 0; i < NN; ++i) {
      if (i == c) continue;
      const float2 f = A[i][c];
#pragma unroll 1
      for (int j = 0; j < NN; ++j) {
        A[i][j] = csub(A[i][j], cmul(f, A[c][j]));
        I[i][j] = csub(I[i][j], cmul(f, I[c][j]));
      }
    }
  }
#pragma unroll 1
  for (int i = 0; i < NN; ++i)
#pragma unroll 1
    for (int j = 0; j < NN; ++j) A[i][j] = I[i][j];
  return true;
}

// ---- the bordered branch of the solver ------------------------------------------------
// One warp per sequence (lane l holds states l, l + 32, ...) whose channel has an
// exactly zero d_j.  The system S w = b with S = diag(dd) + alpha X Y^* -- the
// recurrent step's G (dd = d, X = P, Y = Q) or C~'s G^* (dd = conj d, X = Q,
// Y = P) -- is solved over J = {dd_j != 0} and Z = {dd_j = 0}, s = |Z| <= r, by
// the bordered system of the pages' recurrent mode:
//   [ I_r + alpha Y_J^* DD_J^{-1} X_J   -Y_Z^* ] [ z   ]   [ Y_J^* DD_J^{-1} b_J ]
//   [ alpha X_Z                          0     ] [ w_Z ] = [ b_Z                 ]
//   w_J = DD_J^{-1} (b_J - alpha X_J z).
// The (r + s)-square matrix is padded to 2r x 2r with an identity block (the
// unused unknowns come out zero) and inverted once per warp.
template <int RANK, int E>
struct Bordered {
  float2 yd[E][RANK];  // conj(Y_jl) / dd_j on J; 0 on Z and past N
  float2 xd[E][RANK];  // alpha X_jl / dd_j on J; 0 on Z and past N
  float2 di[E];        // 1 / dd_j on J; 0 on Z and past N
  float2 Mi[2 * RANK][2 * RANK];
  int z[RANK];         // state indices of Z, ascending (the first min(s, r))
  int s;               // |Z|
  bool ok;             // s <= r and the bordered matrix is invertible
};

// Phase one (cheap, for every warp): mark the zero diagonal entries, count them
// and record where they are.  Returns s, the same on every lane.
template <int RANK, int E>
__device__ int bordered_find(const float2* __restrict__ lam, float alpha, int N, int lane,
                             bool (&zero)[E], Bordered<RANK, E>& bd) {
  int s = 0;
#pragma unroll
  for (int i = 0; i < RANK; ++i) bd.z[i] = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    zero[e] = false;
    if (j < N) {
      const float2 d = dpl_diag(lam[j], alpha);
      zero[e] = d.x == 0.f && d.y == 0.f;
    }
    unsigned m = __ballot_sync(0xffffffffu, zero[e]);
    while (m) {  // the same bits on every lane
      const int l = __ffs(m) - 1;
      m &= m - 1;
      if (s < RANK) bd.z[s] = l + 32 * e;
      ++s;
    }
  }
  bd.s = s;
  return s;
}

// Phase two: the per-state constants and the inverse of the padded bordered
// matrix.  conjd: the C~ system (dd = conj d, X = Q, Y = P).
template <int RANK, int E>
__device__ void bordered_build(const float2* __restrict__ lam, const float2* __restrict__ Pm,
                               const float2* __restrict__ Qm, float alpha, int N, int lane, bool conjd,
                               const bool (&zero)[E], Bordered<RANK, E>& bd) {
  const float2* Xm = conjd ? Qm : Pm;
  const float2* Ym = conjd ? Pm : Qm;
  float2 Wp[RANK][RANK];
#pragma unroll
  for (int i = 0; i < RANK; ++i)
#pragma unroll
    for (int l = 0; l < RANK; ++l) Wp[i][l] = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    const bool in = j < N && !zero[e];
    float2 di = make_float2(0.f, 0.f);
    if (in) {
      const float2 d = dpl_diag(lam[j], alpha);
      di = cdiv_safe(make_float2(1.f, 0.f), conjd ? cconj(d) : d);
    }
    bd.di[e] = di;
    float2 xv[RANK];
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      xv[l] = in ? Xm[(size_t)j * RANK + l] : make_float2(0.f, 0.f);
      const float2 yv = in ? Ym[(size_t)j * RANK + l] : make_float2(0.f, 0.f);
      bd.xd[e][l] = cscale(cmul(xv[l], di), alpha);
      bd.yd[e][l] = cmul(cconj(yv), di);
    }
    // (Y_J^* DD_J^{-1} X_J)_{il}: one factor 1/dd_j, carried by yd
#pragma unroll
    for (int i = 0; i < RANK; ++i)
#pragma unroll
      for (int l = 0; l < RANK; ++l) Wp[i][l] = cadd(Wp[i][l], cmul(bd.yd[e][i], xv[l]));
  }
  float2 Mb[2 * RANK][2 * RANK];
#pragma unroll
  for (int i = 0; i < 2 * RANK; ++i)
#pragma unroll
    for (int l = 0; l < 2 * RANK; ++l) Mb[i][l] = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RANK; ++i)
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      const float2 sm = cscale(warp_sum<32>(Wp[i][l]), alpha);
      Mb[i][l] = make_float2(sm.x + (i == l ? 1.f : 0.f), sm.y);
    }
#pragma unroll
  for (int i = 0; i < RANK; ++i) {
    if (i < bd.s) {
      const size_t zi = (size_t)bd.z[i];
#pragma unroll
      for (int l = 0; l < RANK; ++l) {
        Mb[l][RANK + i] = make_float2(-Ym[zi * RANK + l].x, Ym[zi * RANK + l].y);  // -conj(Y_{z_i l})
        Mb[RANK + i][l] = cscale(Xm[zi * RANK + l], alpha);
      }
    } else {
      Mb[RANK + i][RANK + i] = make_float2(1.f, 0.f);
    }
  }
  bd.ok = bd.s <= RANK && invert_local<2 * RANK>(Mb);
#pragma unroll
  for (int i = 0; i < 2 * RANK; ++i)
#pragma unroll
    for (int l = 0; l < 2 * RANK; ++l) bd.Mi[i][l] = Mb[i][l];
}

// w = S^{-1} b for the warp's system (b, w: this lane's states).
template <int RANK, int E>
__device__ __forceinline__ void bordered_solve(const Bordered<RANK, E>& bd, const float2 (&b)[E], float2 (&w)[E],
                                               int lane) {
  float2 rhs[2 * RANK];
#pragma unroll
  for (int l = 0; l < RANK; ++l) {
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) t = cadd(t, cmul(bd.yd[e][l], b[e]));
    rhs[l] = warp_sum<32>(t);
  }
#pragma unroll
  for (int i = 0; i < RANK; ++i) {
    rhs[RANK + i] = make_float2(0.f, 0.f);
    if (i < bd.s) {  // b_{z_i}, broadcast from the lane that holds it
      const int ei = bd.z[i] >> 5, src = bd.z[i] & 31;
      float2 v = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e == ei) v = b[e];
      rhs[RANK + i] = make_float2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
    }
  }
  float2 sol[2 * RANK];
#pragma unroll
  for (int a = 0; a < 2 * RANK; ++a) {
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 2 * RANK; ++c) t = cadd(t, cmul(bd.Mi[a][c], rhs[c]));
    sol[a] = t;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float2 v = cmul(bd.di[e], b[e]);
#pragma unroll
    for (int l = 0; l < RANK; ++l) v = csub(v, cmul(bd.xd[e][l], sol[l]));
    w[e] = v;
  }
#pragma unroll
  for (int i = 0; i < RANK; ++i) {
    if (i < bd.s && lane == (bd.z[i] & 31)) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e == (bd.z[i] >> 5)) w[e] = sol[RANK + i];
    }
  }
}

// Recurrent mode for the sequences whose channel has an exactly zero d_j:
// x_t = G^{-1}(2 x_{t-1} + Delta B u_t) - x_{t-1} with G solved by the bordered
// system, y_t = C^* x_t + D u_t.  Other sequences return at once (the
// recurrent kernel has them); so do channels with an invalid step.
template <int RANK, int E>
__global__ void __launch_bounds__(128) recurrent_bordered_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Cv, const float* __restrict__ dt,
    const float* __restrict__ Dskip, const float* __restrict__ u, int batch, int H, int N, int L,
    float2* __restrict__ x, float2* __restrict__ y, St status) {
  const int warp = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (warp >= batch * H) return;  // (whole warps)
  const int lane = threadIdx.x & 31;
  const int h = warp % H;
  const size_t pb = (size_t)h * N;
  const float delta = dt[h];
  if (!(delta > 0.f) || !(delta <= FLT_MAX)) return;  // reported by the recurrent kernel
  const float alpha = 0.5f * delta;
  Bordered<RANK, E> bd;
  bool zero[E];
  if (bordered_find<RANK, E>(Lambda + pb, alpha, N, lane, zero, bd) == 0) return;
  bordered_build<RANK, E>(Lambda + pb, Pm + pb * RANK, Qm + pb * RANK, alpha, N, lane, false, zero, bd);
  float2* xr = x + (size_t)warp * N;
  if (!bd.ok) {  // s > r, or the bordered matrix is singular
    for (int t = lane; t < L; t += 32) st_chk(y, (long long)warp * L + t, (long long)batch * H * L, make_float2(0.f, 0.f));
    for (int j = lane; j < N; j += 32) xr[j] = make_float2(0.f, 0.f);
    if (lane == 0) st_flag(status, ST_SINGULAR);
    return;
  }
  float2 xs[E], eb[E], cc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    const bool in = j < N;
    xs[e] = in ? xr[j] : make_float2(0.f, 0.f);
    eb[e] = in ? cscale(Bv[pb + j], delta) : make_float2(0.f, 0.f);
    cc[e] = in ? cconj(Cv[pb + j]) : make_float2(0.f, 0.f);
  }
  const float dsk = Dskip[h];
  for (int t = 0; t < L; ++t) {
    const float ut = ld_chk(u, (long long)warp * L + t, (long long)batch * H * L);
    float2 b[E], wv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) b[e] = make_float2(fmaf(2.f, xs[e].x, eb[e].x * ut), fmaf(2.f, xs[e].y, eb[e].y * ut));
    bordered_solve<RANK, E>(bd, b, wv, lane);
    float2 yp = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      xs[e] = csub(wv[e], xs[e]);
      yp = cadd(yp, cmul(cc[e], xs[e]));
    }
    yp = warp_sum<32>(yp);
    if (lane == 0) st_chk(y, (long long)warp * L + t, (long long)batch * H * L, make_float2(fmaf(dsk, ut, yp.x), yp.y));
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    if (j < N) xr[j] = xs[e];
  }
}

// C~ = C - (Abar^*)^M C for the channels with an exactly zero d_j: M steps of
// w <- 2 G^{-*} w - w, G^* = diag(conj d) + alpha Q P^* solved by the bordered
// system.  Other channels (and channels with an invalid step) return at once.
template <int RANK, int E>
__global__ void __launch_bounds__(128) ctilde_bordered_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float* __restrict__ dt, const float2* __restrict__ Cv, int H, int N, int M,
    float2* __restrict__ Ct, St status) {
  const int h = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (h >= H) return;  // (whole warps)
  const int lane = threadIdx.x & 31;
  const size_t pb = (size_t)h * N;
  const float delta = dt[h];
  if (!(delta > 0.f) || !(delta <= FLT_MAX)) return;  // reported by the C~ kernel
  const float alpha = 0.5f * delta;
  Bordered<RANK, E> bd;
  bool zero[E];
  if (bordered_find<RANK, E>(Lambda + pb, alpha, N, lane, zero, bd) == 0) return;
  bordered_build<RANK, E>(Lambda + pb, Pm + pb * RANK, Qm + pb * RANK, alpha, N, lane, true, zero, bd);
  if (!bd.ok) {
    for (int j = lane; j < N; j += 32) st_chk(Ct, (long long)pb + j, (long long)H * N, make_float2(0.f, 0.f));
    if (lane == 0) st_flag(status, ST_SINGULAR);
    return;
  }
  float2 c0[E], w[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    c0[e] = j < N ? Cv[pb + j] : make_float2(0.f, 0.f);
    w[e] = c0[e];
  }
  for (int it = 0; it < M; ++it) {
    float2 g[E];
    bordered_solve<RANK, E>(bd, w, g, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) w[e] = make_float2(fmaf(2.f, g[e].x, -w[e].x), fmaf(2.f, g[e].y, -w[e].y));
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + 32 * e;
    if (j < N) st_chk(Ct, (long long)pb + j, (long long)H * N, csub(c0[e], w[e]));
  }
}

}  // namespace s4dev

namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_bordered)
#endif

// The bordered branch: one warp per sequence; E = 2 covers N <= 64, E = 8 the rest.
template <int RANK>
static cudaError_t rec_bordered(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                                const float2* C, const float* dt, const float* D, const float* u,
                                int batch, int H, int N, int L, float2* x, float2* y, St st,
                                cudaStream_t s) {
  const long long threads = (long long)batch * H * 32;
  const unsigned blocks = (unsigned)((threads + 127) / 128);
  TimedLaunch tl("bordered", s);
  if (N <= 64)
    recurrent_bordered_kernel<RANK, 2><<<blocks, 128, 0, s>>>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st);
  else
    recurrent_bordered_kernel<RANK, 8><<<blocks, 128, 0, s>>>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st);
  return cudaGetLastError();
}

template <int RANK>
static cudaError_t ct_bordered(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                               const float2* C, int H, int N, int M, float2* Ct, St st, cudaStream_t s) {
  const unsigned blocks = (unsigned)(((long long)H * 32 + 127) / 128);
  TimedLaunch tl("bordered", s);
  if (N <= 64)
    ctilde_bordered_kernel<RANK, 2><<<blocks, 128, 0, s>>>(Lam, P, Q, dt, C, H, N, M, Ct, st);
  else
    ctilde_bordered_kernel<RANK, 8><<<blocks, 128, 0, s>>>(Lam, P, Q, dt, C, H, N, M, Ct, st);
  return cudaGetLastError();
}

cudaError_t launch_recurrent_bordered(int r, const float2* Lam, const float2* P, const float2* Q,
                                      const float2* B, const float2* C, const float* dt, const float* D,
                                      const float* u, int batch, int H, int N, int L, float2* x, float2* y,
                                      St st, cudaStream_t s) {
  switch (r) {
    case 1: return rec_bordered<1>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 2: return rec_bordered<2>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 3: return rec_bordered<3>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 4: return rec_bordered<4>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_ctilde_bordered(int r, const float2* Lam, const float2* P, const float2* Q,
                                   const float* dt, const float2* C, int H, int N, int M, float2* Ct,
                                   St st, cudaStream_t s) {
  switch (r) {
    case 1: return ct_bordered<1>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 2: return ct_bordered<2>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 3: return ct_bordered<3>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 4: return ct_bordered<4>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
