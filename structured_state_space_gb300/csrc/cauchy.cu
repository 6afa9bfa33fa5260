// Root values of the S4 filter on the radix-two root grid.
//
// "Recurrent, LSTM, and structured state-space models", section "DPLR
// structured state-space parameterization", filter mode.  At the roots
// z_k = exp(-2 pi i k/M), k != M/2,
//     s(z_k) = (2/Delta)(1 - z_k)/(1 + z_k) = i a tan(pi k/M),   a = 2/Delta,
//     R = diag(1/(s - lambda_j)),  W = I_r + Q^* R P,
//     H(z_k) = 2/(1+z_k) (C~^* R B - C~^* R P W^{-1} Q^* R B),
// and 2/(1 + z_k) = 1 + i tan(pi k/M).  The four resolvent families
// C~^*RB, C~^*RP, Q^*RB, Q^*RP are the (r+1)^2 Cauchy sums of that section,
// evaluated here directly over the N poles; the root z = -1 takes its finite
// value (Delta/2) C~^* B.  Statuses: an fp32 denominator |s - lambda_j|^2 equal
// to zero is 'resonant-diagonal'; an exactly singular W is 'resonant-correction'.
//
// Far roots.  Most roots lie far from every pole: with c the centre of the
// channel's poles and R = max_j |lambda_j - c|, a root with |s - c| >= 1.5 R has
//     sum_j w_j / (s - lambda_j) = (1/(s - c)) sum_m mu_m x^m,   x = R/(s - c),
//     mu_m = sum_j w_j ((lambda_j - c)/R)^m,
// each term's geometric series converging with ratio |y_j| <= |x| <= 2/3,
// y_j = (lambda_j - c)/(s - c).  Truncated after P terms, term j of the Cauchy
// sum is off by the factor 1 - y_j^P: a relative error of at most |x|^P, held to
// 2^-23 (1.2e-7, the level of the fp32 rounding of the direct sum).  P is at most
// kFarTerms = 42 (at |x| = 2/3) and falls quickly with |x| (8 terms at |x| = 0.1);
// a warp takes the largest P its roots need.  The
// moments come from cauchy_moments_kernel, once per channel; a root is far when
// |s - c|^2 >= 2.25 R^2 (in fp32), and a CTA whose roots are all far skips the
// pole loop and evaluates the series by Horner's rule: (r+1)^2 (P - 1) complex
// multiply-adds per root instead of (r+1)^2 N.  Near roots keep the direct sum
// (and the resonance statuses, which only they can meet).  This is an
// epsilon-accurate evaluation of the same Cauchy sums, the kind the pages' cost
// section allows for the filter; the oracle computes the exact definition.
//
// Arithmetic: s is carried as an fp32 (hi, lo) pair (tan(pi k/M) from a table
// computed in float64 at build time, a = 2/Delta split exactly), so that the
// difference s - lambda_j near a resonance keeps full fp32 relative accuracy.
// Each (root, pole) then costs two adds, one FMA, one reciprocal and
// 4 (r+1)^2 FMAs.
#include <float.h>

#include "s4_dev.cuh"
#include "s4_internal.h"
#include "s4_tan.cuh"

// Build-time tuning: poles per unrolled step of the pole loop (1..16 measured
// within noise of each other; 2 kept).
#ifndef S4_CAUCHY_UNROLL
#define S4_CAUCHY_UNROLL 2
#endif
// Packed loop: the per-root denominators in scalar instructions (1) or packed (0).
#ifndef S4_CAUCHY_SCALAR_DEN
#define S4_CAUCHY_SCALAR_DEN 0
#endif

// Poles per chunk of the grouped moments kernel's accumulation (its shared-memory
// power tables hold 2 x chunk x kFarTerms complex values; 16 and 8 measured
// slower: 57 -> 61 and 76 us on N=256 H=1024).
#ifndef S4_CAUCHY_MOM_CHUNK
#define S4_CAUCHY_MOM_CHUNK 32
#endif

namespace s4dev {

constexpr int kCauchyUnroll = S4_CAUCHY_UNROLL;  // poles per unrolled step of the pole loop

__device__ __forceinline__ float2 conj_mul(float2 a, float2 b) {  // conj(a) * b
  return make_float2(fmaf(a.x, b.x, a.y * b.y), fmaf(a.x, b.y, -a.y * b.x));
}

// Build-time tuning: the Woodbury solve's reciprocals by the approximate reciprocal,
// within an ulp or two (1: root values 1011 -> 970 us on N=256 H=1024 M=65536), or
// correctly rounded (0).  An exactly zero pivot is caught before either.
#ifndef S4_CAUCHY_FAST_SOLVE
#define S4_CAUCHY_FAST_SOLVE 1
#endif
__device__ __forceinline__ float2 crecip(float2 w) {
  const float n = fmaf(w.x, w.x, w.y * w.y);
  const float s = S4_CAUCHY_FAST_SOLVE ? rcp_approx(n) : __fdiv_rn(1.f, n);
  return make_float2(w.x * s, -w.y * s);
}

// Solve W z = v for an r x r complex system by Gaussian elimination with
// partial pivoting; v is overwritten by z.  Returns false on an exactly zero pivot.
template <int R>
__device__ __forceinline__ bool solve_small(float2 (&W)[R][R], float2 (&v)[R]) {
#pragma unroll
  for (int col = 0; col < R; ++col) {
    int piv = col;
    float best = fmaxf(fabsf(W[col][col].x), fabsf(W[col][col].y));
#pragma unroll
    for (int row = col + 1; row < R; ++row) {
      const float m = fmaxf(fabsf(W[row][col].x), fabsf(W[row][col].y));
      if (m > best) {
        best = m;
        piv = row;
      }
    }
    if (!(best > 0.f)) return false;
#pragma unroll
    for (int row = col + 1; row < R; ++row) {
      if (row == piv) {
#pragma unroll
        for (int c2 = 0; c2 < R; ++c2) {
          const float2 t = W[col][c2];
          W[col][c2] = W[row][c2];
          W[row][c2] = t;
        }
        const float2 t = v[col];
        v[col] = v[row];
        v[row] = t;
      }
    }
    const float2 inv = crecip(W[col][col]);
#pragma unroll
    for (int row = col + 1; row < R; ++row) {
      const float2 f = cmul(W[row][col], inv);
#pragma unroll
      for (int c2 = col + 1; c2 < R; ++c2) W[row][c2] = csub(W[row][c2], cmul(f, W[col][c2]));
      v[row] = csub(v[row], cmul(f, v[col]));
    }
  }
#pragma unroll
  for (int col = R - 1; col >= 0; --col) {
    float2 acc = v[col];
#pragma unroll
    for (int c2 = col + 1; c2 < R; ++c2) acc = csub(acc, cmul(W[col][c2], v[c2]));
    v[col] = cmul(acc, crecip(W[col][col]));
  }
  return true;
}

// ---- far-field constants of a channel ---------------------------------------------
using s4impl::kFarTerms;   // series terms kept at most
using s4impl::kFarStride;  // float2 entries of the whole set: [c, (R, 0), mu[w][m]]
using s4impl::kFarChannel;  // float2 entries per channel: whole set, groups, permutation
using s4impl::kFarGroups;
using s4impl::kFarGStride;
using s4impl::kFarPermMax;
constexpr float kFarRadius2 = 2.25f;  // far: |s - c|^2 >= (1.5 R)^2

__device__ __forceinline__ float2 far_weight(int widx, int RANKv, float2 c, float2 b, const float2* p,
                                             const float2* q) {
  // order: 0 (C~,B); 1+l (C~,P_l); 1+r+i (Q_i,B); 1+2r+i r+l (Q_i,P_l)
  if (widx == 0) return conj_mul(c, b);
  if (widx < 1 + RANKv) return conj_mul(c, p[widx - 1]);
  if (widx < 1 + 2 * RANKv) return conj_mul(q[widx - 1 - RANKv], b);
  const int t = widx - 1 - 2 * RANKv;
  return conj_mul(q[t / RANKv], p[t % RANKv]);
}

// One CTA per channel: c (centre of the poles' bounding box), R, and the
// moments mu[w][m] = sum_j w_j rho_j^m, rho_j = (lambda_j - c)/R (R = 1 when all
// poles coincide: then every rho_j is 0).  The first kernel of a call: records
// its generation.
template <int RANK>
__global__ void __launch_bounds__(256) cauchy_moments_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Ct, int N, float2* __restrict__ mom, St status) {
  constexpr int NW = (RANK + 1) * (RANK + 1), P = kFarTerms, JC = 32, T = 256;
  constexpr int OWN = (NW * P + T - 1) / T;  // (w, m) pairs per thread
  __shared__ float2 pw[JC][P];
  __shared__ float2 wt[JC][NW];
  __shared__ float red[T / 32][4];
  __shared__ float cr[3];
  pdl_wait();
  st_record_gen(status);
  pdl_launch_dependents();
  const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const float2* lam = Lambda + (size_t)h * N;
  // bounding box of the poles
  float b0 = INFINITY, b1 = -INFINITY, b2 = INFINITY, b3 = -INFINITY;
  for (int j = tid; j < N; j += T) {
    const float2 l = ld_chk(lam, j, N);
    b0 = fminf(b0, l.x); b1 = fmaxf(b1, l.x); b2 = fminf(b2, l.y); b3 = fmaxf(b3, l.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    b0 = fminf(b0, __shfl_xor_sync(0xffffffffu, b0, o));
    b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, o));
    b2 = fminf(b2, __shfl_xor_sync(0xffffffffu, b2, o));
    b3 = fmaxf(b3, __shfl_xor_sync(0xffffffffu, b3, o));
  }
  if (lane == 0) { red[wp][0] = b0; red[wp][1] = b1; red[wp][2] = b2; red[wp][3] = b3; }
  __syncthreads();
  if (tid == 0) {
    for (int i = 1; i < T / 32; ++i) {
      b0 = fminf(b0, red[i][0]); b1 = fmaxf(b1, red[i][1]); b2 = fminf(b2, red[i][2]); b3 = fmaxf(b3, red[i][3]);
    }
    cr[0] = 0.5f * (b0 + b1);
    cr[1] = 0.5f * (b2 + b3);
  }
  __syncthreads();
  const float2 c = make_float2(cr[0], cr[1]);
  float r2 = 0.f;
  for (int j = tid; j < N; j += T) {
    const float2 l = ld_chk(lam, j, N);
    const float dx = l.x - c.x, dy = l.y - c.y;
    r2 = fmaxf(r2, fmaf(dx, dx, dy * dy));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r2 = fmaxf(r2, __shfl_xor_sync(0xffffffffu, r2, o));
  __syncthreads();
  if (lane == 0) red[wp][0] = r2;
  __syncthreads();
  if (tid == 0) {
    for (int i = 1; i < T / 32; ++i) r2 = fmaxf(r2, red[i][0]);
    const float R = sqrtf(r2);
    cr[2] = (R > 0.f && R <= FLT_MAX) ? R : 1.f;
  }
  __syncthreads();
  const float R = cr[2], invR = 1.f / R;
  float2 acc[OWN];
#pragma unroll
  for (int o = 0; o < OWN; ++o) acc[o] = make_float2(0.f, 0.f);
  for (int j0 = 0; j0 < N; j0 += JC) {
    const int jn = min(JC, N - j0);
    __syncthreads();
    if (tid < jn) {  // weights and the powers rho^0 .. rho^(P-1) of pole j0 + tid
      const size_t j = (size_t)h * N + j0 + tid;
      const float2 l = ld_chk(Lambda, j, (long long)gridDim.x * N);
      float2 pp[RANK], qq[RANK];
#pragma unroll
      for (int i = 0; i < RANK; ++i) {
        pp[i] = ld_chk(Pm, (long long)j * RANK + i, (long long)gridDim.x * N * RANK);
        qq[i] = ld_chk(Qm, (long long)j * RANK + i, (long long)gridDim.x * N * RANK);
      }
      const float2 bj = ld_chk(Bv, j, (long long)gridDim.x * N), cj = ld_chk(Ct, j, (long long)gridDim.x * N);
#pragma unroll
      for (int w = 0; w < NW; ++w) wt[tid][w] = far_weight(w, RANK, cj, bj, pp, qq);
      const float2 rho = make_float2((l.x - c.x) * invR, (l.y - c.y) * invR);
      float2 pwr = make_float2(1.f, 0.f);
#pragma unroll
      for (int m = 0; m < P; ++m) {
        pw[tid][m] = pwr;
        pwr = cmul(pwr, rho);
      }
    }
    __syncthreads();
#pragma unroll
    for (int o = 0; o < OWN; ++o) {
      const int t = tid + o * T;
      if (t < NW * P) {
        const int w = t / P, m = t % P;
        float2 a = acc[o];
        for (int jj = 0; jj < jn; ++jj) {
          const float2 x = wt[jj][w], y = pw[jj][m];
          a = make_float2(fmaf(x.x, y.x, fmaf(-x.y, y.y, a.x)), fmaf(x.x, y.y, fmaf(x.y, y.x, a.y)));
        }
        acc[o] = a;
      }
    }
  }
  float2* out = mom + (size_t)h * kFarChannel;
  const long long nout = (long long)gridDim.x * kFarChannel;
  if (tid == 0) {
    st_chk(out, 0, nout - (long long)h * kFarChannel, c);
    st_chk(out, 1, nout - (long long)h * kFarChannel, make_float2(R, 0.f));
  }
#pragma unroll
  for (int o = 0; o < OWN; ++o) {
    const int t = tid + o * T;
    if (t < NW * P) st_chk(out, 2 + t, nout - (long long)h * kFarChannel, acc[o]);
  }
}

// The series' second level (N <= kFarPermMax poles; launched at rank 1): one CTA per
// channel.  The poles fall into kFarGroups groups of equal width in imaginary part
// (between the smallest and largest), numbered in that order and, within a group,
// by pole index; the rank is a pole's position in that order.  The CTA writes the
// whole set's constants, each group's centre, radius (its start rank in the
// imaginary slot) and moments, and the poles by rank.  The five sets' moments
// accumulate over the poles in rank order, one thread per (set, m) with the
// (r+1)^2 weights in registers.
template <int RANK>
__global__ void __launch_bounds__(256) cauchy_moments_grouped_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Ct, int N, float2* __restrict__ mom, St status) {
  constexpr int NW = (RANK + 1) * (RANK + 1), P = kFarTerms, T = 256, G = kFarGroups, NS = 1 + G;
  constexpr int JC = S4_CAUCHY_MOM_CHUNK, PPT = kFarPermMax / T;
  static_assert(2 + NW * P <= kFarGStride, "group stride");
  __shared__ float2 sl[kFarPermMax];                    // poles by rank
  __shared__ __align__(16) float2 sw[kFarPermMax][NW];  // their weights by rank
  __shared__ unsigned char sgid[kFarPermMax];
  __shared__ short sloc[kFarPermMax];      // place within the group (by pole index)
  __shared__ int sperm[kFarPermMax];
  __shared__ int sstart[G + 1];
  __shared__ float scr[NS][3];             // centre and radius of each set (0: all poles)
  __shared__ float sred[T / 32][4];
  __shared__ float2 pw0[JC][P], pwg[JC][P];  // powers of a chunk's poles about the whole set / their group
  pdl_wait();
  st_record_gen(status);
  pdl_launch_dependents();
  const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const long long nj = (long long)gridDim.x * N;
  // this thread's poles j = tid + q T in registers; the whole set's bounding box
  float2 lr[PPT], wr[PPT][NW];
  float b0 = INFINITY, b1 = -INFINITY, b2 = INFINITY, b3 = -INFINITY;
#pragma unroll
  for (int q = 0; q < PPT; ++q) {
    const int j = tid + q * T;
    if (j >= N) continue;
    const long long jg = (long long)h * N + j;
    lr[q] = ld_chk(Lambda, jg, nj);
    float2 pp[RANK], qq[RANK];
#pragma unroll
    for (int i = 0; i < RANK; ++i) {
      pp[i] = ld_chk(Pm, jg * RANK + i, nj * RANK);
      qq[i] = ld_chk(Qm, jg * RANK + i, nj * RANK);
    }
    const float2 bj = ld_chk(Bv, jg, nj), cj = ld_chk(Ct, jg, nj);
#pragma unroll
    for (int w = 0; w < NW; ++w) wr[q][w] = far_weight(w, RANK, cj, bj, pp, qq);
    b0 = fminf(b0, lr[q].x); b1 = fmaxf(b1, lr[q].x); b2 = fminf(b2, lr[q].y); b3 = fmaxf(b3, lr[q].y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    b0 = fminf(b0, __shfl_xor_sync(0xffffffffu, b0, o));
    b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, o));
    b2 = fminf(b2, __shfl_xor_sync(0xffffffffu, b2, o));
    b3 = fmaxf(b3, __shfl_xor_sync(0xffffffffu, b3, o));
  }
  if (lane == 0) { sred[wp][0] = b0; sred[wp][1] = b1; sred[wp][2] = b2; sred[wp][3] = b3; }
  __syncthreads();
  if (tid == 0) {
    for (int i = 1; i < T / 32; ++i) {
      b0 = fminf(b0, sred[i][0]); b1 = fmaxf(b1, sred[i][1]); b2 = fminf(b2, sred[i][2]); b3 = fmaxf(b3, sred[i][3]);
    }
    sred[0][0] = b0; sred[0][1] = b1; sred[0][2] = b2; sred[0][3] = b3;
  }
  __syncthreads();
  const float ylo = sred[0][2], yhi = sred[0][3];
  const float gscale = yhi > ylo ? (float)G / (yhi - ylo) : 0.f;
#pragma unroll
  for (int q = 0; q < PPT; ++q) {
    const int j = tid + q * T;
    if (j >= N) continue;
    const float gf = (lr[q].y - ylo) * gscale;  // (NaN: group 0)
    sgid[j] = (unsigned char)(gf >= 1.f ? min((int)gf, G - 1) : 0);
  }
  __syncthreads();
  if (wp == 0) {  // stable counting by group: place of each pole within its group, group starts
    int cnt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) cnt[g] = 0;
    for (int j0 = 0; j0 < N; j0 += 32) {
      const int j = j0 + lane;
      const int g = j < N ? sgid[j] : -1;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const unsigned b = __ballot_sync(0xffffffffu, g == gg);
        if (g == gg) sloc[j] = (short)(cnt[gg] + __popc(b & ((1u << lane) - 1u)));
        cnt[gg] += __popc(b);
      }
    }
    if (lane == 0) {
      int acc = 0;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sstart[g] = acc;
        acc += cnt[g];
      }
      sstart[G] = acc;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < PPT; ++q) {
    const int j = tid + q * T;
    if (j >= N) continue;
    const int rk = sstart[sgid[j]] + sloc[j];
    if (!S4_IN(rk, kFarPermMax)) continue;
    sperm[rk] = j;
    sl[rk] = lr[q];
#pragma unroll
    for (int w = 0; w < NW; ++w) sw[rk][w] = wr[q][w];
  }
  __syncthreads();
  // warp 0: the whole set's centre and radius; warps 1..G: group wp - 1
  if (wp <= G) {
    const int lo = wp == 0 ? 0 : sstart[wp - 1], hi = wp == 0 ? N : sstart[wp];
    float a0 = INFINITY, a1 = -INFINITY, a2 = INFINITY, a3 = -INFINITY;
    for (int rk = lo + lane; rk < hi; rk += 32) {
      const float2 l = sl[rk];
      a0 = fminf(a0, l.x); a1 = fmaxf(a1, l.x); a2 = fminf(a2, l.y); a3 = fmaxf(a3, l.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a0 = fminf(a0, __shfl_xor_sync(0xffffffffu, a0, o));
      a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, o));
      a2 = fminf(a2, __shfl_xor_sync(0xffffffffu, a2, o));
      a3 = fmaxf(a3, __shfl_xor_sync(0xffffffffu, a3, o));
    }
    const float c0 = hi > lo ? 0.5f * (a0 + a1) : 0.f, c1 = hi > lo ? 0.5f * (a2 + a3) : 0.f;
    float q2 = 0.f;
    for (int rk = lo + lane; rk < hi; rk += 32) {
      const float2 l = sl[rk];
      const float dx = l.x - c0, dy = l.y - c1;
      q2 = fmaxf(q2, fmaf(dx, dx, dy * dy));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q2 = fmaxf(q2, __shfl_xor_sync(0xffffffffu, q2, o));
    if (lane == 0) {
      const float Rq = sqrtf(q2);
      scr[wp][0] = c0;
      scr[wp][1] = c1;
      scr[wp][2] = (Rq > 0.f && Rq <= FLT_MAX) ? Rq : 1.f;
    }
  }
  __syncthreads();
  // moments: thread (set, m) for set < NS, m < P, the 4 weights at once
  const int set = tid / P, m = tid % P;
  const bool mine = set < NS;
  const int lo = set == 0 ? 0 : (mine ? sstart[set - 1] : 0), hi = set == 0 ? N : (mine ? sstart[set] : 0);
  float2 acc[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) acc[w] = make_float2(0.f, 0.f);
  for (int r0 = 0; r0 < N; r0 += JC) {
    const int jn = min(JC, N - r0);
    __syncthreads();
    if (tid < 2 * jn) {  // powers of chunk pole c about the whole set (first half) or its group
      const int c = tid < jn ? tid : tid - jn, rk = r0 + c;
      int g = 0;
      while (g + 1 < G && sstart[g + 1] <= rk) ++g;
      const int st = tid < jn ? 0 : 1 + g;
      const float2 l = sl[rk];
      const float ir = 1.f / scr[st][2];
      const float2 rho = make_float2((l.x - scr[st][0]) * ir, (l.y - scr[st][1]) * ir);
      float2* dst = tid < jn ? pw0[c] : pwg[c];
      float2 pwr = make_float2(1.f, 0.f);
#pragma unroll
      for (int mm = 0; mm < P; ++mm) {
        dst[mm] = pwr;
        pwr = cmul(pwr, rho);
      }
    }
    __syncthreads();
    if (!mine) continue;
    const int jlo = max(lo - r0, 0), jhi = min(hi - r0, jn);
    for (int jj = jlo; jj < jhi; ++jj) {
      const float2 y = set == 0 ? pw0[jj][m] : pwg[jj][m];
      float2 x[NW];
      if constexpr (NW % 2 == 0) {  // 16-byte loads of weight pairs
        const float4* x4 = reinterpret_cast<const float4*>(sw[r0 + jj]);
#pragma unroll
        for (int w = 0; w < NW / 2; ++w) {
          const float4 t = x4[w];
          x[2 * w] = make_float2(t.x, t.y);
          x[2 * w + 1] = make_float2(t.z, t.w);
        }
      } else {
#pragma unroll
        for (int w = 0; w < NW; ++w) x[w] = sw[r0 + jj][w];
      }
#pragma unroll
      for (int w = 0; w < NW; ++w)
        acc[w] = make_float2(fmaf(x[w].x, y.x, fmaf(-x[w].y, y.y, acc[w].x)),
                             fmaf(x[w].x, y.y, fmaf(x[w].y, y.x, acc[w].y)));
    }
  }
  // [whole set: c, (R, 0), mu[w][m] (room for rank 4)] [group g: c, (R, start), mu[w][m]] [poles by rank]
  float2* out = mom + (size_t)h * kFarChannel;
  const long long nout = (long long)kFarChannel;
  if (tid < NS) {
    const long long base = tid == 0 ? 0 : kFarStride + (long long)(tid - 1) * kFarGStride;
    st_chk(out, base, nout, make_float2(scr[tid][0], scr[tid][1]));
    st_chk(out, base + 1, nout, make_float2(scr[tid][2], tid == 0 ? 0.f : (float)sstart[tid - 1]));
  }
  if (mine) {
    const long long base = set == 0 ? 0 : kFarStride + (long long)(set - 1) * kFarGStride;
#pragma unroll
    for (int w = 0; w < NW; ++w) st_chk(out, base + 2 + w * P + m, nout, acc[w]);
  }
  int* outp = reinterpret_cast<int*>(out + kFarStride + G * kFarGStride);
  for (int rk = tid; rk < N; rk += T)
    if (S4_IN(kFarStride + G * kFarGStride + rk / 2, kFarChannel)) outp[rk] = sperm[rk];
}

// The far-field series of the weight sums at this thread's roots s = i (shi + slo):
// with u = s - cen and x = Rr/u, S_w = (1/u) sum_m mu[w FP + m] x^m by Horner's rule,
// with the terms the warp's roots need (P >= 23 / -log2|x|, one more for the
// approximate logarithm, at most FP; roots with live[rr] false do not count).
// Written into acc (ADD false) or added to it.  Called by whole warps.
template <int NW, int RPT, bool PACKED, int FP, bool ADD>
__device__ __forceinline__ void far_series(const float2* __restrict__ mu, float2 cen, float Rr,
                                           const float (&shi)[RPT], const float (&slo)[RPT],
                                           const bool (&live)[RPT], float2 (&acc)[RPT][NW]) {
  float2 iu[RPT], xx[RPT];
  int pneed = 1;
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    const float2 u = make_float2(-cen.x, (shi[rr] - cen.y) + slo[rr]);
    const float n2u = fmaf(u.x, u.x, u.y * u.y);
    // 1/|u|^2 to within an ulp or two (the approximate reciprocal), which the
    // series inherits as a relative error of the same size
    const float r = n2u > 0.f ? rcp_approx(n2u) : 0.f;
    iu[rr] = make_float2(u.x * r, -u.y * r);
    xx[rr] = cscale(iu[rr], Rr);
    const float ax2 = Rr * Rr * r;  // |x|^2 <= 1/2.25 on a far root
    if (live[rr] && ax2 > 0.f) {
      const float p = 23.f * rcp_approx(-0.5f * __log2f(ax2));
      pneed = max(pneed, min(FP, (int)p + 2));
    }
  }
  const int P = __reduce_max_sync(0xffffffffu, (unsigned)pneed);
  if constexpr (PACKED) {
    constexpr int NPR = RPT / 2;
    // root pairs in packed fp32x2: hx = {Re h of root 2pr, of root 2pr+1}, hy likewise;
    // each step is the scalar step below, operation for operation
    float2 x2x[NPR], x2y[NPR], n2y[NPR];
#pragma unroll
    for (int pr = 0; pr < NPR; ++pr) {
      x2x[pr] = make_float2(xx[2 * pr].x, xx[2 * pr + 1].x);
      x2y[pr] = make_float2(xx[2 * pr].y, xx[2 * pr + 1].y);
      n2y[pr] = make_float2(-x2y[pr].x, -x2y[pr].y);
    }
    // all weights' chains advance together: NW NPR independent chains per step
    // (one weight after another measured 2 % slower on N=256 H=1024 M=65536)
    float2 hx[NW][NPR], hy[NW][NPR];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float2 top = mu[w * FP + P - 1];
#pragma unroll
      for (int pr = 0; pr < NPR; ++pr) {
        hx[w][pr] = make_float2(top.x, top.x);
        hy[w][pr] = make_float2(top.y, top.y);
      }
    }
#pragma unroll 2
    for (int m = P - 2; m >= 0; --m) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float2 mv = mu[w * FP + m];
        const float2 mx = make_float2(mv.x, mv.x), my = make_float2(mv.y, mv.y);
#pragma unroll
        for (int pr = 0; pr < NPR; ++pr) {
          const float2 nx = __ffma2_rn(hx[w][pr], x2x[pr], __ffma2_rn(hy[w][pr], n2y[pr], mx));
          const float2 ny = __ffma2_rn(hx[w][pr], x2y[pr], __ffma2_rn(hy[w][pr], x2x[pr], my));
          hx[w][pr] = nx;
          hy[w][pr] = ny;
        }
      }
    }
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int pr = 0; pr < NPR; ++pr) {
        const float2 v0 = cmul(make_float2(hx[w][pr].x, hy[w][pr].x), iu[2 * pr]);
        const float2 v1 = cmul(make_float2(hx[w][pr].y, hy[w][pr].y), iu[2 * pr + 1]);
        acc[2 * pr][w] = ADD ? cadd(acc[2 * pr][w], v0) : v0;
        acc[2 * pr + 1][w] = ADD ? cadd(acc[2 * pr + 1][w], v1) : v1;
      }
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      float2 hw[RPT];
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) hw[rr] = mu[w * FP + P - 1];
#pragma unroll 4
      for (int m = P - 2; m >= 0; --m) {
        const float2 mv = mu[w * FP + m];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr)
          hw[rr] = make_float2(fmaf(hw[rr].x, xx[rr].x, fmaf(-hw[rr].y, xx[rr].y, mv.x)),
                               fmaf(hw[rr].x, xx[rr].y, fmaf(hw[rr].y, xx[rr].x, mv.y)));
      }
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) {
        const float2 v = cmul(hw[rr], iu[rr]);
        acc[rr][w] = ADD ? cadd(acc[rr][w], v) : v;
      }
    }
  }
}

// Per pole j in shared memory: Im lambda_j, (Re lambda_j)^2, then for each
// weight w (order 0: (C~,B); 1+l: (C~,P_l); 1+r+i: (Q_i,B); 1+2r+i r+l: (Q_i,P_l))
// the pair w and w (-Re lambda_j).  With d = s - lambda_j = -Re lambda_j + i dim,
//   w / d = (w (-Re lambda_j) - i dim w) / |d|^2
// costs two FMAs for the numerator and two for the accumulation.
//
// PACKED: two roots per packed fp32x2 instruction (__ffma2_rn / __fadd2_rn, the
// same per-lane rounding as the scalar form, so the sums are bit-identical).
// A packed instruction does two lanes' work for one issue slot, which matters
// because the scalar loop is issue-bound (about 24 issued instructions per
// term for 19 FMA-pipe ones).  The pole data is then staged as duplicated
// pairs -- {-Im lambda, -Im lambda}, {(Re lambda)^2, ...}, and per weight
// {w.y, w.y}, {w.x a, w.x a}, {-w.x, -w.x}, {w.y a, w.y a} with a = -Re lambda --
// so one 16-byte shared load gives two packed operands.
template <int RANK, bool PACKED = false>
struct CauchyLayout {
  static constexpr int NW = (RANK + 1) * (RANK + 1);      // weight vectors
  static constexpr int PS = PACKED ? 4 * (1 + 2 * NW)     // floats per pole (float4-padded)
                                   : (2 + 4 * NW + 3) / 4 * 4;
  static constexpr int JT = PS <= 48 ? 128 : 64;          // poles staged at a time
};

// (4 roots per thread: compiled for 4 CTAs per SM, the schedule measured fastest;
// left to itself the compiler picks a tighter, slower one)
#ifndef S4_CAUCHY_MINB
#define S4_CAUCHY_MINB 4
#endif
// (rank >= 2: resident CTAs per SM; 4 spills at 128 registers)
#ifndef S4_CAUCHY_MINB_FAR2
#define S4_CAUCHY_MINB_FAR2 3
#endif
// FAR: the far-root series is compiled in (it is used when `far_on` and the
// constants are given); without it the kernel is the direct sum alone.
// GRP: the second level of the series is compiled in (used when `grouped`: the
// moments kernel formed the groups and the permutation for this call).
template <int RANK, int RPT, int T, bool PACKED = false, bool FAR = false, bool GRP = false>
__global__ void __launch_bounds__(T, RPT >= 4 ? (RANK >= 2 ? S4_CAUCHY_MINB_FAR2 : S4_CAUCHY_MINB) : 0)
    cauchy_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Ct, const float* __restrict__ dt,
    float2* __restrict__ Khat, const float2* __restrict__ mom, int far_on, int grouped, int N, int logM,
    int logC, St status) {
  using Lay = CauchyLayout<RANK, PACKED>;
  constexpr int NW = Lay::NW, PS = Lay::PS, JT = Lay::JT;
  static_assert(!PACKED || RPT % 2 == 0, "packed roots come in pairs");
  constexpr int NPR = RPT / 2;  // (PACKED) root pairs per thread
  constexpr int FP = kFarTerms;
  __shared__ __align__(16) float par[JT * PS];
  __shared__ float2 mus[2 + NW * FP];  // c, (R, 0), mu[w][m] of this channel
  __shared__ float2 red[T / 32 + 1];
  // the groups' constants [c_g, (R_g, 0), mu_g[w][m]], loaded at the first near tile
  constexpr int GSL = 2 + NW * FP;  // a group's constants in shared memory
  __shared__ float2 musg[GRP ? kFarGroups * GSL : 1];
  static_assert(!GRP || (FAR && 2 + NW * FP <= kFarGStride), "groups: the series, the group stride");

  if constexpr (!FAR) far_on = 0;
  if constexpr (!GRP) grouped = 0;
  grouped = far_on ? grouped : 0;
  pdl_wait();  // the moments kernel (and whatever ran before it) is done
  if (!far_on) st_record_gen(status);  // (else the moments kernel, this call's first, did)
  pdl_launch_dependents();  // the next kernel may start; it waits for this grid before reading
  const int h = blockIdx.x;
  if (far_on) {
    for (int i = threadIdx.x; i < 2 + NW * FP; i += T)
      mus[i] = ld_chk(mom, (long long)h * kFarChannel + i, (long long)gridDim.x * kFarChannel);
    __syncthreads();  // every warp reads c and R below (far_on is uniform)
  }
  const int M = 1 << logM;
  const float delta = dt[h];
  const bool bad = !(delta > 0.f) || !(delta <= FLT_MAX);
  const int Mc = M >> logC;
  // a = 2/Delta as an exact fp32 pair a_hi + a_lo
  const float a_hi = bad ? 0.f : __fdiv_rn(2.f, delta);
  const float a_lo = bad ? 0.f : __fdiv_rn(fmaf(-a_hi, delta, 2.f), delta);

  // A tile is RPT T consecutive roots k (so that near and far roots fall in
  // separate tiles); root k is stored at position (k mod C) M/C + k div C.  With
  // the far-root series a warp owns 32 RPT consecutive roots of the tile (lane l
  // takes l, l + 32, ...), so that near and far roots also fall in separate warps.  The
  // CTA takes the tiles of its channel numbered v = blockIdx.y, blockIdx.y +
  // gridDim.y, ..., tile v/2 for even v and tiles - 1 - v/2 for odd v: the roots
  // near the poles lie at the two ends of the range (s = i a tan(pi k/M) small),
  // so their costly direct tiles start first instead of forming the grid's tail.
  // The next tile's tan values are loaded while the current one is computed.
  const int tiles = (M + RPT * T - 1) / (RPT * T);
  auto tile_of = [&](int v) { return (v & 1) ? tiles - 1 - (v >> 1) : (v >> 1); };
  auto root_of = [&](int tile, int rr) {
    return FAR ? tile * RPT * T + (int)(threadIdx.x >> 5) * 32 * RPT + rr * 32 + (int)(threadIdx.x & 31)
               : (tile * RPT + rr) * T + (int)threadIdx.x;
  };
  auto tan_of = [&](int tile, int rr) {
    const int kr = root_of(tile, rr);
    return (kr < M && S4_IN(kr << (16 - logM), 65536)) ? __ldg(g_tan + (kr << (16 - logM)))
                                                      : make_float2(0.f, 0.f);
  };
  float2 tnext[FAR ? RPT : 1];
  if constexpr (FAR) {
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) tnext[rr] = tan_of(tile_of(blockIdx.y), rr);
  }
  unsigned flags = bad ? ST_BAD_STEP : 0u;
  bool groups_loaded = false;
  const int* permh = reinterpret_cast<const int*>(mom + (size_t)h * kFarChannel + kFarStride +
                                                  kFarGroups * kFarGStride);
  for (int v = blockIdx.y; v < tiles; v += gridDim.y) {
    const int tile = tile_of(v);
    int pos[RPT];
    bool zm1[RPT];
    float shi[RPT], slo[RPT], th[RPT];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
      const int kr = root_of(tile, rr);
      const bool valid = kr < M;
      const int k = valid ? kr : 0;
      pos[rr] = valid ? (k & ((1 << logC) - 1)) * Mc + (k >> logC) : M;
      float2 tt;
      if constexpr (FAR) tt = tnext[rr];
      else tt = tan_of(tile, rr);
      zm1[rr] = valid && M >= 2 && 2 * k == M;
      const float p = a_hi * tt.x;
      const float perr = fmaf(a_hi, tt.x, -p);
      const float lo = perr + fmaf(a_hi, tt.y, a_lo * tt.x);
      shi[rr] = zm1[rr] ? 0.f : p;
      slo[rr] = zm1[rr] ? 0.f : lo;
      th[rr] = tt.x;
    }
    if (FAR && v + (int)gridDim.y < tiles) {
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) tnext[FAR ? rr : 0] = tan_of(tile_of(v + gridDim.y), rr);
    }
    // far roots: |s - c|^2 >= 2.25 R^2 with u = s - c (s = i (shi + slo)); the z = -1
    // root and positions past M need no sums.  A warp takes the series only when all
    // its roots are far; otherwise each of its roots takes the direct sum.  The CTA
    // stages the poles unless all its warps are far.
    const float2 fc = far_on ? mus[0] : make_float2(0.f, 0.f);
    const float fR = far_on ? mus[1].x : 0.f;
    float2 fu[RPT];
    bool warp_far = false, cta_far = false;
    if constexpr (FAR) {
      bool mine = far_on != 0;
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) {
        fu[rr] = make_float2(-fc.x, (shi[rr] - fc.y) + slo[rr]);
        const float n2u = fmaf(fu[rr].x, fu[rr].x, fu[rr].y * fu[rr].y);
        mine = mine && (pos[rr] >= M || zm1[rr] || (n2u >= kFarRadius2 * fR * fR && n2u > 0.f));
      }
      warp_far = __all_sync(0xffffffffu, mine);
      cta_far = __syncthreads_and(warp_far) != 0;
    }
    // a near warp of a grouped channel: bit g of gnear when some root of the warp is
    // near group g (|s - c_g| < 1.5 R_g); it sums directly over those groups' poles only
    unsigned gnear = 0u;
    if constexpr (GRP) {
      if (grouped && !cta_far) {
        if (!groups_loaded) {  // (uniform)
          for (int i = threadIdx.x; i < kFarGroups * GSL; i += T)
            musg[i] = ld_chk(mom, (long long)h * kFarChannel + kFarStride + (i / GSL) * kFarGStride + i % GSL,
                             (long long)gridDim.x * kFarChannel);
          groups_loaded = true;
          __syncthreads();
        }
        if (!warp_far) {
#pragma unroll
          for (int g = 0; g < kFarGroups; ++g) {
            const float2 cg = musg[g * GSL];
            const float Rg = musg[g * GSL + 1].x;
            bool gfar = true;
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr) {
              const float2 u = make_float2(-cg.x, (shi[rr] - cg.y) + slo[rr]);
              const float n2 = fmaf(u.x, u.x, u.y * u.y);
              gfar = gfar && (pos[rr] >= M || zm1[rr] || (n2 >= kFarRadius2 * Rg * Rg && n2 > 0.f));
            }
            if (!__all_sync(0xffffffffu, gfar)) gnear |= 1u << g;
          }
        }
      }
    }

    float2 acc[RPT][NW];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
      for (int w = 0; w < NW; ++w) acc[rr][w] = make_float2(0.f, 0.f);
    float2 cb = make_float2(0.f, 0.f);  // this thread's part of C~^* B (pole loop)
    // (PACKED) the accumulators of root pair pr: ax = {acc[2pr][w].x, acc[2pr+1][w].x}, ay likewise
    float2 ax[PACKED ? NPR : 1][NW], ay[PACKED ? NPR : 1][NW], sh2[PACKED ? NPR : 1], sl2[PACKED ? NPR : 1];
    if constexpr (PACKED) {
#pragma unroll
      for (int pr = 0; pr < NPR; ++pr) {
        sh2[pr] = make_float2(shi[2 * pr], shi[2 * pr + 1]);
        sl2[pr] = make_float2(slo[2 * pr], slo[2 * pr + 1]);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          ax[pr][w] = make_float2(0.f, 0.f);
          ay[pr][w] = make_float2(0.f, 0.f);
        }
      }
    }

    for (int j0 = 0; j0 < (cta_far ? 0 : N); j0 += JT) {
      const int jn = min(JT, N - j0);
      __syncthreads();
      for (int jj = threadIdx.x; jj < jn; jj += T) {
        // (grouped: the poles in rank order, so that each group is one range)
        const int jp = (GRP && grouped && S4_IN((long long)h * kFarChannel + kFarStride + kFarGroups * kFarGStride +
                                                    (j0 + jj) / 2,
                                                (long long)gridDim.x * kFarChannel))
                           ? __ldg(permh + j0 + jj)
                           : j0 + jj;
        const size_t j = (size_t)h * N + jp;
        const long long nj = (long long)gridDim.x * N;  // H N
        if (!S4_IN(j, nj) || !S4_IN((long long)j * RANK + RANK - 1, nj * RANK) || !S4_IN(jj * PS + PS - 1, JT * PS))
          continue;
        const float2 lam = Lambda[j], b = Bv[j], c = Ct[j];
        float* pp = par + jj * PS;
        const float nre = -lam.x;
        if constexpr (PACKED) {
          reinterpret_cast<float4*>(pp)[0] = make_float4(-lam.y, -lam.y, lam.x * lam.x, lam.x * lam.x);
        } else {
          pp[0] = lam.y;
          pp[1] = lam.x * lam.x;
        }
        auto put = [&](int widx, float2 w) {
          if constexpr (PACKED) {
            float4* p4 = reinterpret_cast<float4*>(pp) + 1 + 2 * widx;
            p4[0] = make_float4(w.y, w.y, w.x * nre, w.x * nre);
            p4[1] = make_float4(-w.x, -w.x, w.y * nre, w.y * nre);
          } else {
            pp[2 + 4 * widx] = w.x;
            pp[3 + 4 * widx] = w.y;
            pp[4 + 4 * widx] = w.x * nre;
            pp[5 + 4 * widx] = w.y * nre;
          }
        };
        const float2 w0 = conj_mul(c, b);
        cb = cadd(cb, w0);
        put(0, w0);
#pragma unroll
        for (int l = 0; l < RANK; ++l) put(1 + l, conj_mul(c, Pm[j * RANK + l]));
#pragma unroll
        for (int i = 0; i < RANK; ++i) {
          const float2 qi = Qm[j * RANK + i];
          put(1 + RANK + i, conj_mul(qi, b));
#pragma unroll
          for (int l = 0; l < RANK; ++l) put(1 + 2 * RANK + i * RANK + l, conj_mul(qi, Pm[j * RANK + l]));
        }
        if constexpr (!PACKED) {
#pragma unroll
          for (int f = 2 + 4 * NW; f < PS; ++f) pp[f] = 0.f;
        }
      }
      __syncthreads();
      if (warp_far) continue;  // (a far warp only helps stage the poles)
      if constexpr (PACKED) {
        // the staged poles this warp sums over: all, or the ranges of its near groups
        for (int g = 0; g < (GRP && grouped ? kFarGroups : 1); ++g) {
        int jlo = 0, jhi = jn;
        if (GRP && grouped) {
          if (!((gnear >> g) & 1u)) continue;
          jlo = max((int)musg[g * GSL + 1].y - j0, 0);
          jhi = min((g + 1 < kFarGroups ? (int)musg[(g + 1) * GSL + 1].y : N) - j0, jn);
        }
#pragma unroll kCauchyUnroll
        for (int jj = jlo; jj < jhi; ++jj) {
          const float4* p4 = reinterpret_cast<const float4*>(par + jj * PS);
          const float4 pl = p4[0];
          const float2 nim = make_float2(pl.x, pl.y), re2 = make_float2(pl.z, pl.w);
          float2 dim[NPR], rn[NPR];
#pragma unroll
          for (int pr = 0; pr < NPR; ++pr) {
#if S4_CAUCHY_SCALAR_DEN
            // the denominators in scalar instructions, which may issue to the FMA
            // pipe's other half while the packed products keep the first busy
            dim[pr] = make_float2((sh2[pr].x + nim.x) + sl2[pr].x, (sh2[pr].y + nim.y) + sl2[pr].y);
            rn[pr] = make_float2(rcp_approx(fmaf(dim[pr].x, dim[pr].x, re2.x)),
                                 rcp_approx(fmaf(dim[pr].y, dim[pr].y, re2.y)));
#else
            dim[pr] = __fadd2_rn(__fadd2_rn(sh2[pr], nim), sl2[pr]);
            const float2 n2 = __ffma2_rn(dim[pr], dim[pr], re2);
            rn[pr] = make_float2(rcp_approx(n2.x), rcp_approx(n2.y));
#endif
          }
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float4 b4 = p4[1 + 2 * w], c4 = p4[2 + 2 * w];
            const float2 wy = make_float2(b4.x, b4.y), wax = make_float2(b4.z, b4.w);
            const float2 nwx = make_float2(c4.x, c4.y), way = make_float2(c4.z, c4.w);
#pragma unroll
            for (int pr = 0; pr < NPR; ++pr) {
              const float2 tx = __ffma2_rn(dim[pr], wy, wax);
              const float2 ty = __ffma2_rn(dim[pr], nwx, way);
              ax[pr][w] = __ffma2_rn(rn[pr], tx, ax[pr][w]);
              ay[pr][w] = __ffma2_rn(rn[pr], ty, ay[pr][w]);
            }
          }
        }
        }  // groups
        continue;
      }
      for (int g = 0; g < (GRP && grouped ? kFarGroups : 1); ++g) {
      int jlo = 0, jhi = jn;
      if (GRP && grouped) {
        if (!((gnear >> g) & 1u)) continue;
        jlo = max((int)musg[g * GSL + 1].y - j0, 0);
        jhi = min((g + 1 < kFarGroups ? (int)musg[(g + 1) * GSL + 1].y : N) - j0, jn);
      }
#pragma unroll kCauchyUnroll
      for (int jj = jlo; jj < jhi; ++jj) {
        float pr[PS];
        const float4* p4 = reinterpret_cast<const float4*>(par + jj * PS);
#pragma unroll
        for (int v = 0; v < PS / 4; ++v) {
          const float4 t = p4[v];
          pr[4 * v] = t.x;
          pr[4 * v + 1] = t.y;
          pr[4 * v + 2] = t.z;
          pr[4 * v + 3] = t.w;
        }
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) {
          const float dim = (shi[rr] - pr[0]) + slo[rr];
          const float n2 = fmaf(dim, dim, pr[1]);
          const float rn = rcp_approx(n2);
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float wx = pr[2 + 4 * w], wy = pr[3 + 4 * w];
            const float tx = fmaf(dim, wy, pr[4 + 4 * w]);
            const float ty = fmaf(-dim, wx, pr[5 + 4 * w]);
            acc[rr][w].x = fmaf(rn, tx, acc[rr][w].x);
            acc[rr][w].y = fmaf(rn, ty, acc[rr][w].y);
          }
        }
      }
      }  // groups
    }

    if constexpr (PACKED) {
#pragma unroll
      for (int pr = 0; pr < NPR; ++pr)
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          acc[2 * pr][w] = make_float2(ax[pr][w].x, ay[pr][w].x);
          acc[2 * pr + 1][w] = make_float2(ax[pr][w].y, ay[pr][w].y);
        }
    }

    // far warps: the series of the whole set; near warps of a grouped channel: the
    // series of each group they are far from, added to the direct sums of the others
    if (FAR && (warp_far || (GRP && grouped))) {
      bool live[RPT];
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) live[rr] = pos[rr] < M && !zm1[rr];
      if (warp_far) {
        far_series<NW, RPT, PACKED, FP, false>(mus + 2, fc, fR, shi, slo, live, acc);
      } else if constexpr (GRP) {
#pragma unroll
        for (int g = 0; g < kFarGroups; ++g)
          if (!((gnear >> g) & 1u))
            far_series<NW, RPT, PACKED, FP, true>(musg + g * GSL + 2, musg[g * GSL], musg[g * GSL + 1].x, shi, slo,
                                                  live, acc);
      }
    }
    // C~^* B over all poles, for the root z = -1: the zeroth moment of that weight
    // when the pole loop was skipped, else the loop's sum
    float2 cb_all;
    if (FAR && cta_far) {
      cb_all = mus[2];
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cb.x += __shfl_xor_sync(0xffffffffu, cb.x, o);
        cb.y += __shfl_xor_sync(0xffffffffu, cb.y, o);
      }
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cb;
      __syncthreads();
      if (threadIdx.x == 0) {
        float2 t = make_float2(0.f, 0.f);
        for (int i = 0; i < T / 32; ++i) t = cadd(t, red[i]);
        red[T / 32] = t;
      }
      __syncthreads();
      cb_all = red[T / 32];
    }

#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
      if (pos[rr] >= M) continue;
      float2 Hk = make_float2(0.f, 0.f);
      if (!bad) {
        if (zm1[rr]) {
          Hk = cscale(cb_all, 0.5f * delta);
        } else {
          // (far tiles cannot meet a resonance: a non-finite value there shows in Hk)
          bool fin = true;
          if (!(FAR && warp_far)) {
#pragma unroll
            for (int w = 0; w < NW; ++w) fin = fin && cfinite(acc[rr][w]);
          }
          if (!fin) {
            // an exactly zero denominator gives inf/nan; tell it apart from overflow
            bool res = false;
            for (int j = 0; j < N; ++j) {
              const float2 lam = Lambda[(size_t)h * N + j];
              const float dim = (shi[rr] - lam.y) + slo[rr];
              res = res || (fmaf(dim, dim, lam.x * lam.x) == 0.f);
            }
            flags |= res ? ST_RES_DIAG : ST_NONFINITE;
            st_chk(Khat, (long long)h * M + pos[rr], (long long)gridDim.x * M, Hk);
            continue;
          }
          float2 Wm[RANK][RANK], z[RANK];
#pragma unroll
          for (int i = 0; i < RANK; ++i) {
            z[i] = acc[rr][1 + RANK + i];
#pragma unroll
            for (int l = 0; l < RANK; ++l) {
              Wm[i][l] = acc[rr][1 + 2 * RANK + i * RANK + l];
              if (i == l) Wm[i][l].x += 1.f;
            }
          }
          if (!solve_small<RANK>(Wm, z)) {
            flags |= ST_RES_CORR;
          } else {
            float2 g = acc[rr][0];
#pragma unroll
            for (int l = 0; l < RANK; ++l) g = csub(g, cmul(acc[rr][1 + l], z[l]));
            Hk = make_float2(fmaf(-th[rr], g.y, g.x), fmaf(th[rr], g.x, g.y));
            if (!cfinite(Hk)) {
              flags |= ST_NONFINITE;
              Hk = make_float2(0.f, 0.f);
            }
          }
        }
      }
      st_chk(Khat, (long long)h * M + pos[rr], (long long)gridDim.x * M, Hk);
    }
    if constexpr (!FAR) break;  // one tile per CTA
  }  // tiles
  if (flags) st_flag(status, flags);
}

}  // namespace s4dev

namespace s4impl {
using namespace s4dev;

#ifdef S4_BOUNDS_CHECK
S4_OOB_COUNTER(oob_cauchy)
#endif

// Build-time tuning: threads per CTA and roots per thread for rank 1 on small
// grids (block sizes 32..256 and 2..8 roots per thread measured within 3 %).
#ifndef S4_CAUCHY_T
#define S4_CAUCHY_T 128
#endif
#ifndef S4_CAUCHY_RPT1
#define S4_CAUCHY_RPT1 2
#endif
// ... and on grids of two waves or more (4 was faster there until the status
// generation entered the kernel: the compiler then schedules the 4-root kernel
// more tightly (85 registers, or 109 when told 4 CTAs per SM suffice), and 2
// roots measured 1-2 % faster on both large workloads)
#ifndef S4_CAUCHY_RPT1_BIG
#define S4_CAUCHY_RPT1_BIG 2
#endif
// Packed (fp32x2) root pairs at rank 1 on grids of two waves or more, 4 roots
// (two pairs) per thread: 3.4 % faster than the scalar loop on the
// N=256 H=1024 M=65536 grid and 3.5 % on N=64 H=512 M=4096; the scalar loop
// stays faster on smaller grids (20.5 against 22.5 us on N=64 H=256 M=1024),
// and 2 roots per thread packed was 35 % slower (two shared loads per term).
#ifndef S4_CAUCHY_PACKED
#define S4_CAUCHY_PACKED 1
#endif
#ifndef S4_CAUCHY_PRPT1_BIG
#define S4_CAUCHY_PRPT1_BIG 4
#endif
#ifndef S4_CAUCHY_FAR_TILES
#define S4_CAUCHY_FAR_TILES 8
#endif
// The far series' second level (pole groups) for near warps (1) or none (0).
#ifndef S4_CAUCHY_GROUPS
#define S4_CAUCHY_GROUPS 1
#endif


template <int RANK, int RPT, bool PACKED, bool FAR, bool GRP = false>
static cudaError_t cauchy_launch_far(const float2* Lambda, const float2* P, const float2* Q,
                                     const float2* B, const float2* Ct, const float* dt,
                                     float2* Khat, const float2* mom, int H, int N, int M, int logC, St status,
                                     cudaStream_t s, bool pdl) {
  constexpr int T = S4_CAUCHY_T;
  const int tiles = (M + T * RPT - 1) / (T * RPT);
  static int per_sm = -1;  // resident CTAs per SM (queried once per instantiation)
  if (per_sm < 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cauchy_kernel<RANK, RPT, T, PACKED, FAR, GRP>, T,
                                                    0) != cudaSuccess)
    per_sm = 0;
  // With the far-root series, a CTA loops over up to S4_CAUCHY_FAR_TILES tiles of
  // its channel (most of them cheap series tiles, which would otherwise each pay a
  // CTA's set-up), as long as the grid keeps 16 CTAs per resident slot for the
  // balance of the costly direct tiles (measured on N=256 H=1024 M=65536: 1511 ->
  // 1394 us at 4 tiles when the series was introduced; with the later far path 8
  // tiles 969 -> 957 us and 2 tiles 1001 us; on N=64 H=256 M=16384, whose grid is
  // 16 times smaller, 4 tiles were slower: 184 -> 198 us).  The direct sum alone
  // keeps one tile per CTA.
  long long per_cta = 1;
  if (FAR && per_sm > 0) {
    per_cta = (long long)H * tiles / (16LL * per_sm * num_sms());
    per_cta = per_cta < 1 ? 1 : (per_cta > S4_CAUCHY_FAR_TILES ? S4_CAUCHY_FAR_TILES : per_cta);
  }
  dim3 grid(H, (unsigned)((tiles + per_cta - 1) / per_cta));
  TimedLaunch tl("cauchy", s);
  int logM = 0;
  while ((1 << logM) < M) ++logM;
  // A programmatic launch lets this grid's CTAs become resident while the
  // previous kernel drains; that pays when the grid fits in one wave.  A larger
  // grid's first wave would only sit on the SMs beside the previous kernel's tail.
  pdl = pdl && (long long)grid.x * grid.y <= (long long)per_sm * num_sms();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(T);
  cfg.stream = s;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, cauchy_kernel<RANK, RPT, T, PACKED, FAR, GRP>, Lambda, P, Q, B, Ct, dt, Khat,
                            mom, mom ? 1 : 0, GRP ? 1 : 0, N, logM, logC, status);
}

// the far-root series compiled in only where its constants are given, and its
// second level where the groups were formed (`grouped`)
template <int RANK, int RPT, bool PACKED = false>
static cudaError_t cauchy_launch(const float2* Lambda, const float2* P, const float2* Q,
                                 const float2* B, const float2* Ct, const float* dt,
                                 float2* Khat, const float2* mom, int H, int N, int M, int logC, St status,
                                 cudaStream_t s, bool pdl, bool grouped = false) {
  if constexpr (RANK == 1 && PACKED) {
    if (mom != nullptr && grouped)
      return cauchy_launch_far<RANK, RPT, PACKED, true, true>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC,
                                                              status, s, pdl);
  }
  if (mom != nullptr)
    return cauchy_launch_far<RANK, RPT, PACKED, true>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s,
                                                      pdl);
  return cauchy_launch_far<RANK, RPT, PACKED, false>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s,
                                                     pdl);
}

template <int RANK, bool GROUPS = false>
static cudaError_t moments_launch(const float2* Lambda, const float2* P, const float2* Q, const float2* B,
                                  const float2* Ct, float2* mom, int H, int N, St status, cudaStream_t s,
                                  bool pdl) {
  static_assert(!GROUPS || RANK == 1, "groups at rank 1");
  TimedLaunch tl("moments", s);
  using Kern = void (*)(const float2*, const float2*, const float2*, const float2*, const float2*, int, float2*, St);
  Kern kern = cauchy_moments_kernel<RANK>;
  if constexpr (GROUPS) kern = cauchy_moments_grouped_kernel<RANK>;
  static int per_sm = -1;
  if (pdl && per_sm < 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess)
    per_sm = 0;
  pdl = pdl && (long long)H <= (long long)per_sm * num_sms();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(H);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, Lambda, P, Q, B, Ct, N, mom, status);
}

cudaError_t launch_cauchy(const float2* Lambda, const float2* P, const float2* Q, const float2* B,
                          const float2* Ct, const float* dt, float2* Khat, float2* mom, int H, int N, int r,
                          int M, int logC, St status, cudaStream_t s, bool pdl) {
  // the far-field constants first (this call's first kernel), then the root values,
  // a programmatic dependent that waits for them.  Only on rows of M >= 8192 roots
  // and N >= 48 poles: on shorter rows every CTA of roots holds near roots, and
  // with few poles the series is not shorter than the sum, so the extra launch
  // would not pay (measured slower on N=64 M=1024 and M=4096).
  if (M < 8192 || N < 48) mom = nullptr;
  // roots per thread: rank 1 takes 2 on every grid (S4_CAUCHY_RPT1_BIG); rank 2
  // takes 4 (512 per CTA) once the grid holds at least two waves of such CTAs
  // and 2 below that, to keep enough warps resident
  const bool small = (long long)H * M < 512LL * 5 * 2 * num_sms();
  // the series' second level (pole groups) for the packed rank-1 kernel of large
  // grids, 128 <= N <= kFarPermMax: groups of 32 poles or more, where a group's
  // series (<= 41 steps of 4 complex multiply-adds) costs less than its direct sum.
  // (At rank 2 with N = 64, groups of 16 poles, the root values measured slower:
  // 160 -> 245 us on N=64 r=2 H=256 M=16384.  The kernels are templated on the
  // rank; only rank 1 is launched, and the group stride holds its 4 weight vectors.)
  const bool grouped = S4_CAUCHY_GROUPS && S4_CAUCHY_PACKED && r == 1 && !small && N >= 128 && N <= kFarPermMax;
  if (mom != nullptr) {
    cudaError_t e;
    switch (r) {
      case 1:
        e = grouped ? moments_launch<1, true>(Lambda, P, Q, B, Ct, mom, H, N, status, s, pdl)
                    : moments_launch<1>(Lambda, P, Q, B, Ct, mom, H, N, status, s, pdl);
        break;
      case 2: e = moments_launch<2>(Lambda, P, Q, B, Ct, mom, H, N, status, s, pdl); break;
      case 3: e = moments_launch<3>(Lambda, P, Q, B, Ct, mom, H, N, status, s, pdl); break;
      case 4: e = moments_launch<4>(Lambda, P, Q, B, Ct, mom, H, N, status, s, pdl); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    pdl = true;
  }
  switch (r) {
    case 1:
#if S4_CAUCHY_PACKED
      return small ? cauchy_launch<1, S4_CAUCHY_RPT1>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<1, S4_CAUCHY_PRPT1_BIG, true>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s,
                                                               pdl, grouped);
#else
      return small ? cauchy_launch<1, S4_CAUCHY_RPT1>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<1, S4_CAUCHY_RPT1_BIG>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl);
#endif
    case 2:  // 4 roots per thread on large grids measured 2 % faster (8 at rank 1 was 11 % slower)
      return small ? cauchy_launch<2, 2>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<2, 4>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl);
    case 3:
      return cauchy_launch<3, 1>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl);
    case 4:
      return cauchy_launch<4, 1>(Lambda, P, Q, B, Ct, dt, Khat, mom, H, N, M, logC, status, s, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
