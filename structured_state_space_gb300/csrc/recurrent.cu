// Recurrent mode of the bilinear-discretised DPLR model, and the formation of
// the truncated output vector C~ from C.
//
// "Recurrent, LSTM, and structured state-space models", section "DPLR
// structured state-space parameterization": with alpha = Delta/2,
// G = I - alpha A, the recurrent mode computes b_t = (I + alpha A) x_{t-1} +
// Delta B u_t, G x_t = b_t, y_t = C^* x_t (+ D u_t, the separate direct term);
// the solve uses the Woodbury inverse with D = diag(d_j), d_j = 1 - alpha
// lambda_j and the correction I_r + alpha Q^* D^{-1} P.  The truncated output
// vector is C~ = (I - Abar^M)^* C.
//
// Since I + alpha A = 2I - G, one step is x_t = G^{-1}(2 x_{t-1} + Delta B u_t)
// - x_{t-1}: one Woodbury solve, i.e. one reduction of r values over the N
// states, plus one reduction for y_t (the recurrent kernel folds D^{-1} into
// its per-state constants, so a step touches each state with three complex
// multiply-adds and one complex product).  Likewise Abar^* = 2 G^{-*} - I, and
// G^* = diag(conj d_j) + alpha Q P^* has the correction W^* (W = I_r + alpha
// Q^* D^{-1} P), so C~ = C - (Abar^*)^M C takes M solves with W^{-*}; the C~
// kernel groups them p at a time (Abar^{*p} as diagonal plus rank p r, see
// ctilde_kernel).
//
// A group of G lanes owns one sequence (one channel of one batch row, or one
// channel for C~): G = 16 for N <= 64 in the recurrent mode (two sequences per
// warp, so each reduction takes four shuffle rounds for both), otherwise 32;
// lane l of a group holds states j = l, l + G, ...  W^{-1} is formed once per
// group.  An exactly singular W is reported as S4_ERR_SINGULAR_BILINEAR and the
// outputs are zeros.
//
// The pages' solver has a second branch: when some d_j is exactly zero (the set
// Z, s = |Z| <= r) the correction is replaced by the bordered system of size
// r + s over (Q^* x, x_Z).  A channel with such a d_j (and a valid step) is
// left alone by the two kernels above and taken by recurrent_bordered_kernel /
// ctilde_bordered_kernel, one warp per sequence, a plain step at a time (the
// branch is rare: it needs 1 - (Delta/2) lambda_j to round to exactly zero).
// Both partitions use the same fp32 test of d_j, so every sequence is written
// by exactly one kernel.
#include <float.h>

#include "s4_dev.cuh"
#include "s4_internal.h"
#include "s4_solve.cuh"

namespace s4dev {

// Sums over a 16-lane group of two complex values at once by recursive
// halving: a (returned to every lane) and b (returned to lane 8 of the group,
// the others get a partial value).  Offset 8 exchanges two floats, offset 4
// one, offsets 2 and 1 one each; then three shuffles broadcast a and finish b:
// 9 shuffles, 5 adds and 6 selects instead of 16 shuffles and 16 adds.
__device__ __forceinline__ void group16_sum2(float2& a, float2& b) {
  const unsigned lane = threadIdx.x & 15u;
  const bool hi8 = lane & 8u, hi4 = lane & 4u;
  float k0 = hi8 ? b.x : a.x, k1 = hi8 ? b.y : a.y;
  const float s0 = hi8 ? a.x : b.x, s1 = hi8 ? a.y : b.y;
  k0 += __shfl_xor_sync(0xffffffffu, s0, 8);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 8);
  float k = hi4 ? k1 : k0;  // lane holds (hi8 ? b : a).(hi4 ? y : x)
  k += __shfl_xor_sync(0xffffffffu, hi4 ? k0 : k1, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  a.x = __shfl_sync(0xffffffffu, k, 0, 16);
  a.y = __shfl_sync(0xffffffffu, k, 4, 16);
  const float by = __shfl_sync(0xffffffffu, k, 12, 16);
  b = make_float2(k, by);  // complete in lane 8
}

// Sums of NF floats over the G lanes of a group, returned to every lane, by
// recursive halving (NF a power of two <= G): at offset G/2 each lane keeps one
// half of its values and sends the other, at G/4 a half of that, ... until one
// value is left, which the remaining offsets finish; component j then sits in
// lane j G/NF, from which it is broadcast.  NF - 1 + log2(G/NF) exchange
// shuffles and NF broadcasts instead of NF log2(G).
template <int NF, int G>
__device__ __forceinline__ void group_sum_all(float (&v)[NF]) {
  static_assert((NF & (NF - 1)) == 0 && NF <= G, "NF: a power of two <= G");
  const unsigned lane = threadIdx.x % G;
  float w[NF];
#pragma unroll
  for (int i = 0; i < NF; ++i) w[i] = v[i];
  int off = G / 2;
#pragma unroll
  for (int cnt = NF; cnt > 1; cnt >>= 1, off >>= 1) {
    const bool hi = lane & off;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float keep = hi ? w[cnt / 2 + i] : w[i];
      const float send = hi ? w[i] : w[cnt / 2 + i];
      w[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int o = G / (2 * NF); o > 0; o >>= 1) w[0] += __shfl_xor_sync(0xffffffffu, w[0], o);
#pragma unroll
  for (int j = 0; j < NF; ++j) v[j] = __shfl_sync(0xffffffffu, w[0], j * (G / NF), G);
}

// Per-warp channel constants: dinv_j = 1/d_j, and W^{-1} (conjugate-transposed for C~).
template <int RANK, int E>
struct ChanConst {
  float2 dinv[E];
  float2 Winv[RANK][RANK];
  bool ok;
  bool zero_d;  // some d_j of the channel is exactly zero (the bordered branch)
};

template <int RANK, int E, int G = 32>
__device__ void channel_constants(const float2* __restrict__ lam, const float2* __restrict__ Pm,
                                  const float2* __restrict__ Qm, float alpha, int N, int lane,
                                  ChanConst<RANK, E>& cc) {
  bool zero_d = false;
  float2 Wp[RANK][RANK];
#pragma unroll
  for (int i = 0; i < RANK; ++i)
#pragma unroll
    for (int l = 0; l < RANK; ++l) Wp[i][l] = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + G * e;
    cc.dinv[e] = make_float2(0.f, 0.f);
    if (j < N) {
      const float2 d = dpl_diag(lam[j], alpha);
      if (d.x == 0.f && d.y == 0.f) {
        zero_d = true;
        continue;
      }
      cc.dinv[e] = cdiv_safe(make_float2(1.f, 0.f), d);
      // W = I + alpha Q^* D^{-1} P
#pragma unroll
      for (int i = 0; i < RANK; ++i) {
        const float2 qd = cmul(cconj(Qm[(size_t)j * RANK + i]), cc.dinv[e]);
#pragma unroll
        for (int l = 0; l < RANK; ++l) Wp[i][l] = cadd(Wp[i][l], cmul(qd, Pm[(size_t)j * RANK + l]));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RANK; ++i)
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      const float2 s = warp_sum<G>(Wp[i][l]);
      cc.Winv[i][l] = make_float2(alpha * s.x + (i == l ? 1.f : 0.f), alpha * s.y);
    }
  int zd = zero_d ? 1 : 0;  // OR over the group
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) zd |= __shfl_xor_sync(0xffffffffu, zd, o);
  zero_d = zd != 0;
  cc.zero_d = zero_d;
  cc.ok = !zero_d && invert_small<RANK>(cc.Winv);
}

// Steps per unrolled iteration of the recurrence: the output reduction of one
// step overlaps the next step's work (4 measured 6 % faster than 1; 8 no better).
#ifndef S4_RECURRENT_UNROLL
#define S4_RECURRENT_UNROLL 4
#endif
constexpr int kRecurrentUnroll = S4_RECURRENT_UNROLL;

// x_t = G^{-1}(2 x_{t-1} + Delta B u_t) - x_{t-1},  y_t = C^* x_t + D u_t.
template <int RANK, int E, int G>
__global__ void __launch_bounds__(128) recurrent_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Cv, const float* __restrict__ dt,
    const float* __restrict__ Dskip, const float* __restrict__ u, int batch, int H, int N, int L,
    float2* __restrict__ x, float2* __restrict__ y, St status) {
  const int gt = blockIdx.x * blockDim.x + threadIdx.x;
  if ((gt & ~31) / G >= batch * H) return;  // the whole warp is past the last sequence
  // a group past the last sequence (odd count, G = 16) runs on sequence 0 and
  // stores nothing, so that every lane of the warp takes part in the shuffles
  const bool valid = gt / G < batch * H;
  const int warp = valid ? gt / G : 0;
  const int lane = threadIdx.x % G;
  const int h = warp % H;
  const size_t pb = (size_t)h * N;
  const float delta = dt[h];
  const bool bad = !(delta > 0.f) || !(delta <= FLT_MAX);
  const float alpha = 0.5f * delta;
  ChanConst<RANK, E> cc;
  channel_constants<RANK, E, G>(Lambda + pb, Pm + pb * RANK, Qm + pb * RANK, alpha, N, lane, cc);
  const bool ok = cc.ok && !bad;
  // a channel with an exactly zero d_j (and a valid step) belongs to
  // recurrent_bordered_kernel: run along for the shuffles, store nothing
  const bool mine = valid && !(cc.zero_d && !bad);
  // With w = D^{-1}(2 x + Delta B u) substituted, one step is
  //   s = sum_j h_j x_j + c0 u,  h_j = 2 conj(Q_j) / d_j,  c0 = sum_j conj(Q_j) Delta B_j / d_j,
  //   z = W^{-1} s,  x'_j = a_j x_j + e_j u - pd_j z,  a_j = 2/d_j - 1, e_j = Delta B_j / d_j,
  // and the next step's partial s is accumulated while x' is formed.
  float2 xs[E], av[E], eb[E], pd[E][RANK], hq[E][RANK], cc_[E], c0[RANK];
#pragma unroll
  for (int l = 0; l < RANK; ++l) c0[l] = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + G * e;
    const bool in = j < N;
    const float2 di = cc.dinv[e];  // zero outside the states
    xs[e] = in ? ld_chk(x, (long long)warp * N + j, (long long)batch * H * N) : make_float2(0.f, 0.f);
    eb[e] = in ? cscale(cmul(di, Bv[pb + j]), delta) : make_float2(0.f, 0.f);
    av[e] = in ? make_float2(fmaf(2.f, di.x, -1.f), 2.f * di.y) : make_float2(0.f, 0.f);
    cc_[e] = in ? cconj(Cv[pb + j]) : make_float2(0.f, 0.f);
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      const float2 qcl = in ? cconj(Qm[(pb + j) * RANK + l]) : make_float2(0.f, 0.f);
      pd[e][l] = in ? cscale(cmul(di, Pm[(pb + j) * RANK + l]), alpha) : make_float2(0.f, 0.f);
      hq[e][l] = cscale(cmul(qcl, di), 2.f);
      c0[l] = cadd(c0[l], cmul(qcl, eb[e]));
    }
  }
#pragma unroll
  for (int l = 0; l < RANK; ++l) c0[l] = warp_sum<G>(c0[l]);
  const float dsk = Dskip[h];
  float2 s[RANK];  // this lane's part of sum_j h_j x_j for the coming step
#pragma unroll
  for (int l = 0; l < RANK; ++l) {
    s[l] = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) s[l] = cadd(s[l], cmul(hq[e][l], xs[e]));
  }
  // rank 1 in 16-lane groups: a step ends with one joint reduction of the next
  // step's s and this step's output, so s enters each step already summed
  constexpr bool JOINT = RANK == 1 && G == 16;
  if constexpr (JOINT) s[0] = warp_sum<G>(s[0]);
  const int ylane = JOINT ? 8 : 0;  // the lane that holds the summed output
#pragma unroll kRecurrentUnroll
  for (int t = 0; t < L; ++t) {
    const float ut = ld_chk(u, (long long)warp * L + t, (long long)batch * H * L);
    float2 z[RANK];
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      if constexpr (!JOINT) s[l] = warp_sum<G>(s[l]);
      s[l] = make_float2(fmaf(c0[l].x, ut, s[l].x), fmaf(c0[l].y, ut, s[l].y));
    }
#pragma unroll
    for (int i = 0; i < RANK; ++i) {
      z[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int l = 0; l < RANK; ++l) z[i] = cadd(z[i], cmul(cc.Winv[i][l], s[l]));
    }
    float2 yp = make_float2(0.f, 0.f);
#pragma unroll
    for (int l = 0; l < RANK; ++l) s[l] = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) {  // x = a x + e u - pd z
      float2 v = cmul(av[e], xs[e]);
      v = make_float2(fmaf(eb[e].x, ut, v.x), fmaf(eb[e].y, ut, v.y));
#pragma unroll
      for (int l = 0; l < RANK; ++l) v = csub(v, cmul(pd[e][l], z[l]));
      xs[e] = v;
      yp = cadd(yp, cmul(cc_[e], v));
#pragma unroll
      for (int l = 0; l < RANK; ++l) s[l] = cadd(s[l], cmul(hq[e][l], v));
    }
    if constexpr (JOINT) {
      group16_sum2(s[0], yp);
    } else {
      yp = warp_sum<G>(yp);
    }
    if (mine && lane == ylane)
      st_chk(y, (long long)warp * L + t, (long long)batch * H * L,
             ok ? make_float2(fmaf(dsk, ut, yp.x), yp.y) : make_float2(0.f, 0.f));
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + G * e;
    if (mine && j < N) st_chk(x, (long long)warp * N + j, (long long)batch * H * N, ok ? xs[e] : make_float2(0.f, 0.f));
  }
  if (mine && lane == 0 && !ok) st_flag(status, bad ? ST_BAD_STEP : ST_SINGULAR);
}

// C~ = C - (Abar^*)^M C with Abar^* w = 2 G^{-*} w - w.
//
// G^{-*} w = conj(D)^{-1} w - alpha conj(D)^{-1} Q W^{-*} P^* conj(D)^{-1} w, so
// Abar^* = diag(a) - U V^T with a_j = 2/conj(d_j) - 1, U = 2 alpha conj(D)^{-1} Q W^{-*}
// and V = conj(D)^{-1} conj(P) (V^T w = P^* conj(D)^{-1} w): diagonal plus rank r.
// Its square is again diagonal plus low rank,
//   (diag(a) - U V^T)^2 = diag(a^2) - [aU - U K, U] [V, aV]^T,  K = V^T U,
// so LOGP squarings give Abar^{*P} (P = 2^LOGP) at rank P r, and M/P steps of
// w <- a w - U (V^T w) finish the power: each step's P r reductions over the N
// states share one pass of shuffle rounds, so the chain of dependent
// reductions is M/P long instead of M, for the same arithmetic per original
// step (about 8 r complex flop pairs per state).
template <int RANK, int E, int G, int LOGP>
__global__ void __launch_bounds__(128) ctilde_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float* __restrict__ dt, const float2* __restrict__ Cv, int H, int N, int M,
    float2* __restrict__ Ct, St status) {
  constexpr int P = 1 << LOGP, KP = RANK * P;
  constexpr int KH = KP / 2 > 0 ? KP / 2 : 1;  // columns before the last squaring
  const int gt = blockIdx.x * blockDim.x + threadIdx.x;
  if ((gt & ~31) / G >= H) return;  // the whole warp is past the last channel
  const bool valid = gt / G < H;    // (a surplus group runs on channel 0 and stores nothing)
  const int h = valid ? gt / G : 0;
  const int lane = threadIdx.x % G;
  const size_t pb = (size_t)h * N;
  const float delta = dt[h];
  const bool bad = !(delta > 0.f) || !(delta <= FLT_MAX);
  const float alpha = 0.5f * delta;
  ChanConst<RANK, E> cc;
  channel_constants<RANK, E, G>(Lambda + pb, Pm + pb * RANK, Qm + pb * RANK, alpha, N, lane, cc);
  const bool ok = cc.ok && !bad;
  // an exactly zero d_j (with a valid step): ctilde_bordered_kernel's channel
  const bool mine = valid && !(cc.zero_d && !bad);
  // factors of Abar^*: columns 0..RANK-1 of U, V
  float2 av[E], w[E], c0[E], Uf[E][KP], Vf[E][KP];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + G * e;
    const bool in = j < N;
    const float2 dc = cconj(cc.dinv[e]);  // zero outside the states
    av[e] = in ? make_float2(fmaf(2.f, dc.x, -1.f), 2.f * dc.y) : make_float2(0.f, 0.f);
    c0[e] = in ? Cv[pb + j] : make_float2(0.f, 0.f);
    w[e] = c0[e];
    float2 q2[RANK];
#pragma unroll
    for (int i = 0; i < RANK; ++i)
      q2[i] = in ? cscale(cmul(dc, Qm[(pb + j) * RANK + i]), 2.f * alpha) : make_float2(0.f, 0.f);
#pragma unroll
    for (int l = 0; l < RANK; ++l) {
      float2 u = make_float2(0.f, 0.f);  // (2 alpha conj(D)^{-1} Q W^{-*})_{j l}
#pragma unroll
      for (int i = 0; i < RANK; ++i) u = cadd(u, cmul(q2[i], cconj(cc.Winv[l][i])));
      Uf[e][l] = u;
      Vf[e][l] = in ? cmul(cconj(Pm[(pb + j) * RANK + l]), dc) : make_float2(0.f, 0.f);
    }
  }
  // LOGP squarings: rank k -> 2k
#pragma unroll
  for (int lev = 0; lev < LOGP; ++lev) {
    const int k = RANK << lev;
    float2 Km[KH][KH];  // K = V^T U over the first k columns
#pragma unroll
    for (int m = 0; m < KH; ++m)
#pragma unroll
      for (int c = 0; c < KH; ++c) {
        if (m < k && c < k) {
          float2 t = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < E; ++e) t = cadd(t, cmul(Vf[e][m], Uf[e][c]));
          Km[m][c] = warp_sum<G>(t);
        }
      }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float2 un[KH];
#pragma unroll
      for (int c = 0; c < KH; ++c) {
        if (c < k) {
          float2 t = cmul(av[e], Uf[e][c]);
#pragma unroll
          for (int m = 0; m < KH; ++m)
            if (m < k) t = csub(t, cmul(Uf[e][m], Km[m][c]));
          un[c] = t;
        }
      }
#pragma unroll
      for (int c = 0; c < KH; ++c) {
        if (c < k) {
          Uf[e][k + c] = Uf[e][c];
          Uf[e][c] = un[c];
          Vf[e][k + c] = cmul(av[e], Vf[e][c]);
        }
      }
      av[e] = cmul(av[e], av[e]);
    }
  }
  float2 sv[KP];  // this lane's part of V^T w for the coming step
#pragma unroll
  for (int m = 0; m < KP; ++m) {
    sv[m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) sv[m] = cadd(sv[m], cmul(Vf[e][m], w[e]));
  }
  const int steps = M >> LOGP;
  // the step's KP complex sums together by recursive halving when 2 KP is a
  // power of two no larger than the group
  constexpr bool HALVE = ((2 * KP) & (2 * KP - 1)) == 0 && 2 * KP <= G;
  for (int it = 0; it < steps; ++it) {
    if constexpr (HALVE) {
      float f[2 * KP];
#pragma unroll
      for (int m = 0; m < KP; ++m) {
        f[2 * m] = sv[m].x;
        f[2 * m + 1] = sv[m].y;
      }
      group_sum_all<2 * KP, G>(f);
#pragma unroll
      for (int m = 0; m < KP; ++m) sv[m] = make_float2(f[2 * m], f[2 * m + 1]);
    } else {
#pragma unroll
      for (int m = 0; m < KP; ++m) sv[m] = warp_sum<G>(sv[m]);
    }
    float2 sn[KP];
#pragma unroll
    for (int m = 0; m < KP; ++m) sn[m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E; ++e) {  // w <- Abar^{*P} w
      float2 g = cmul(av[e], w[e]);
#pragma unroll
      for (int m = 0; m < KP; ++m) g = csub(g, cmul(Uf[e][m], sv[m]));
      w[e] = g;
#pragma unroll
      for (int m = 0; m < KP; ++m) sn[m] = cadd(sn[m], cmul(Vf[e][m], g));
    }
#pragma unroll
    for (int m = 0; m < KP; ++m) sv[m] = sn[m];
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = lane + G * e;
    if (mine && j < N) st_chk(Ct, (long long)pb + j, (long long)H * N, ok ? csub(c0[e], w[e]) : make_float2(0.f, 0.f));
  }
  if (mine && lane == 0 && !ok) st_flag(status, bad ? ST_BAD_STEP : ST_SINGULAR);
}

}  // namespace s4dev

namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_recurrent)
#endif

template <int RANK, int E, int G>
static cudaError_t rec_launch(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                              const float2* C, const float* dt, const float* D, const float* u,
                              int batch, int H, int N, int L, float2* x, float2* y, St st,
                              cudaStream_t s) {
  const long long threads = (long long)batch * H * G;
  TimedLaunch tl("recurrent", s);
  recurrent_kernel<RANK, E, G><<<(unsigned)((threads + 127) / 128), 128, 0, s>>>(Lam, P, Q, B, C, dt, D, u,
                                                                                 batch, H, N, L, x, y, st);
  return cudaGetLastError();
}

// 16 lanes per sequence (two per warp) up to N = 64, a whole warp above
template <int RANK>
static cudaError_t rec_dispatch(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                                const float2* C, const float* dt, const float* D, const float* u,
                                int batch, int H, int N, int L, float2* x, float2* y, St st,
                                cudaStream_t s) {
  if (N <= 16) return rec_launch<RANK, 1, 16>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
  if (N <= 32) return rec_launch<RANK, 2, 16>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
  if (N <= 64) return rec_launch<RANK, 4, 16>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
  if (N <= 128) return rec_launch<RANK, 4, 32>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
  return rec_launch<RANK, 8, 32>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
}

template <int RANK, int E, int G, int LOGP>
static cudaError_t ct_launch(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                             const float2* C, int H, int N, int M, float2* Ct, St st,
                             cudaStream_t s) {
  const long long threads = (long long)H * G;
  TimedLaunch tl("ctilde", s);
  ctilde_kernel<RANK, E, G, LOGP><<<(unsigned)((threads + 127) / 128), 128, 0, s>>>(Lam, P, Q, dt, C, H, N, M, Ct, st);
  return cudaGetLastError();
}

// Look-ahead of 2^LOGP steps per reduction pass, as far as the registers hold
// the factors (E x 2^LOGP x r <= 16 complex columns per lane) and M allows.
constexpr int ct_logp(int rank, int e) {
  int lp = 0;
  while (lp < 4 && e * (rank << (lp + 1)) <= 16) ++lp;
  return lp;
}

template <int RANK, int E>
static cudaError_t ct_launch_p(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                               const float2* C, int H, int N, int M, float2* Ct, St st,
                               cudaStream_t s) {
  constexpr int LP = ct_logp(RANK, E);
  if (M % (1 << LP) == 0) return ct_launch<RANK, E, 32, LP>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
  return ct_launch<RANK, E, 32, 0>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
}

// One warp per channel: C~ runs one chain of M / 2^LOGP dependent steps per
// channel with only H chains in flight, so it is latency-bound and wants the
// most lanes (the fewest elements per lane) on each chain.
template <int RANK>
static cudaError_t ct_dispatch(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                               const float2* C, int H, int N, int M, float2* Ct, St st,
                               cudaStream_t s) {
  if (N <= 32) return ct_launch_p<RANK, 1>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
  if (N <= 64) return ct_launch_p<RANK, 2>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
  if (N <= 128) return ct_launch_p<RANK, 4>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
  return ct_launch_p<RANK, 8>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
}

template <int RANK>
static cudaError_t rec_both(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                            const float2* C, const float* dt, const float* D, const float* u,
                            int batch, int H, int N, int L, float2* x, float2* y, St st, cudaStream_t s) {
  const cudaError_t e = rec_dispatch<RANK>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
  if (e != cudaSuccess) return e;
  return launch_recurrent_bordered(RANK, Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
}

cudaError_t launch_recurrent(const float2* Lam, const float2* P, const float2* Q, const float2* B,
                             const float2* C, const float* dt, const float* D, const float* u,
                             int batch, int H, int N, int r, int L, float2* x, float2* y,
                             St st, cudaStream_t s) {
  switch (r) {
    case 1: return rec_both<1>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 2: return rec_both<2>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 3: return rec_both<3>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    case 4: return rec_both<4>(Lam, P, Q, B, C, dt, D, u, batch, H, N, L, x, y, st, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int RANK>
static cudaError_t ct_both(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                           const float2* C, int H, int N, int M, float2* Ct, St st, cudaStream_t s) {
  const cudaError_t e = ct_dispatch<RANK>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
  if (e != cudaSuccess) return e;
  return launch_ctilde_bordered(RANK, Lam, P, Q, dt, C, H, N, M, Ct, st, s);
}

cudaError_t launch_ctilde(const float2* Lam, const float2* P, const float2* Q, const float* dt,
                          const float2* C, int H, int N, int r, int M, float2* Ct, St st,
                          cudaStream_t s) {
  switch (r) {
    case 1: return ct_both<1>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 2: return ct_both<2>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 3: return ct_both<3>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    case 4: return ct_both<4>(Lam, P, Q, dt, C, H, N, M, Ct, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
