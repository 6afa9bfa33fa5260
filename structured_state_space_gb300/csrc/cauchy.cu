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

namespace s4dev {

constexpr int kCauchyUnroll = S4_CAUCHY_UNROLL;  // poles per unrolled step of the pole loop

__device__ __forceinline__ float2 conj_mul(float2 a, float2 b) {  // conj(a) * b
  return make_float2(fmaf(a.x, b.x, a.y * b.y), fmaf(a.x, b.y, -a.y * b.x));
}

__device__ __forceinline__ float2 crecip(float2 w) {
  const float n = fmaf(w.x, w.x, w.y * w.y);
  const float s = __fdiv_rn(1.f, n);
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
template <int RANK, int RPT, int T, bool PACKED = false>
__global__ void __launch_bounds__(T, RPT >= 4 ? S4_CAUCHY_MINB : 0) cauchy_kernel(
    const float2* __restrict__ Lambda, const float2* __restrict__ Pm, const float2* __restrict__ Qm,
    const float2* __restrict__ Bv, const float2* __restrict__ Ct, const float* __restrict__ dt,
    float2* __restrict__ Khat, int N, int logM, int logC, St status) {
  using Lay = CauchyLayout<RANK, PACKED>;
  constexpr int NW = Lay::NW, PS = Lay::PS, JT = Lay::JT;
  static_assert(!PACKED || RPT % 2 == 0, "packed roots come in pairs");
  constexpr int NPR = RPT / 2;  // (PACKED) root pairs per thread
  __shared__ __align__(16) float par[JT * PS];
  __shared__ float2 red[T / 32 + 1];

  pdl_wait();  // (a programmatic launch) the previous kernel on the stream is done
  st_record_gen(status);
  pdl_launch_dependents();  // the next kernel may start; it waits for this grid before reading
  const int h = blockIdx.x;
  const int M = 1 << logM;
  const float delta = dt[h];
  const bool bad = !(delta > 0.f) || !(delta <= FLT_MAX);
  const int Mc = M >> logC;
  // a = 2/Delta as an exact fp32 pair a_hi + a_lo
  const float a_hi = bad ? 0.f : __fdiv_rn(2.f, delta);
  const float a_lo = bad ? 0.f : __fdiv_rn(fmaf(-a_hi, delta, 2.f), delta);

  int pos[RPT];
  bool zm1[RPT];
  float shi[RPT], slo[RPT], th[RPT];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    pos[rr] = (blockIdx.y * RPT + rr) * T + threadIdx.x;
    const bool valid = pos[rr] < M;
    const int k = valid ? (pos[rr] % Mc) * (1 << logC) + pos[rr] / Mc : 0;
    const float2 tt = (valid && S4_IN(k << (16 - logM), 65536)) ? __ldg(g_tan + (k << (16 - logM)))
                                                                 : make_float2(0.f, 0.f);
    zm1[rr] = valid && M >= 2 && 2 * k == M;
    const float p = a_hi * tt.x;
    const float perr = fmaf(a_hi, tt.x, -p);
    const float lo = perr + fmaf(a_hi, tt.y, a_lo * tt.x);
    shi[rr] = zm1[rr] ? 0.f : p;
    slo[rr] = zm1[rr] ? 0.f : lo;
    th[rr] = tt.x;
  }

  float2 acc[RPT][NW];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr)
#pragma unroll
    for (int w = 0; w < NW; ++w) acc[rr][w] = make_float2(0.f, 0.f);
  float2 cb = make_float2(0.f, 0.f);
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

  for (int j0 = 0; j0 < N; j0 += JT) {
    const int jn = min(JT, N - j0);
    __syncthreads();
    for (int jj = threadIdx.x; jj < jn; jj += T) {
      const size_t j = (size_t)h * N + j0 + jj;
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
      float2 w = conj_mul(c, b);
      cb = cadd(cb, w);
      put(0, w);
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
    if constexpr (PACKED) {
#pragma unroll kCauchyUnroll
      for (int jj = 0; jj < jn; ++jj) {
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
      continue;
    }
#pragma unroll kCauchyUnroll
    for (int jj = 0; jj < jn; ++jj) {
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

  // C~^* B over all poles, for the root z = -1
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
  const float2 cb_all = red[T / 32];

  unsigned flags = bad ? ST_BAD_STEP : 0u;
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    if (pos[rr] >= M) continue;
    float2 Hk = make_float2(0.f, 0.f);
    if (!bad) {
      if (zm1[rr]) {
        Hk = cscale(cb_all, 0.5f * delta);
      } else {
        bool fin = true;
#pragma unroll
        for (int w = 0; w < NW; ++w) fin = fin && cfinite(acc[rr][w]);
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


template <int RANK, int RPT, bool PACKED = false>
static cudaError_t cauchy_launch(const float2* Lambda, const float2* P, const float2* Q,
                                 const float2* B, const float2* Ct, const float* dt,
                                 float2* Khat, int H, int N, int M, int logC, St status,
                                 cudaStream_t s, bool pdl) {
  constexpr int T = S4_CAUCHY_T;
  const int tiles = (M + T * RPT - 1) / (T * RPT);
  dim3 grid(H, tiles);
  TimedLaunch tl("cauchy", s);
  int logM = 0;
  while ((1 << logM) < M) ++logM;
  // A programmatic launch lets this grid's CTAs become resident while the
  // previous kernel drains; that pays when the grid fits in one wave.  A larger
  // grid's first wave would only sit on the SMs beside the previous kernel's tail.
  static int per_sm = -1;  // resident CTAs per SM (queried once per instantiation)
  if (pdl && per_sm < 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cauchy_kernel<RANK, RPT, T, PACKED>, T, 0) != cudaSuccess)
    per_sm = 0;
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
  return cudaLaunchKernelEx(&cfg, cauchy_kernel<RANK, RPT, T, PACKED>, Lambda, P, Q, B, Ct, dt, Khat, N, logM,
                            logC, status);
}

cudaError_t launch_cauchy(const float2* Lambda, const float2* P, const float2* Q, const float2* B,
                          const float2* Ct, const float* dt, float2* Khat, int H, int N, int r,
                          int M, int logC, St status, cudaStream_t s, bool pdl) {
  // roots per thread: rank 1 takes 2 on every grid (S4_CAUCHY_RPT1_BIG); rank 2
  // takes 4 (512 per CTA) once the grid holds at least two waves of such CTAs
  // and 2 below that, to keep enough warps resident
  const bool small = (long long)H * M < 512LL * 5 * 2 * num_sms();
  switch (r) {
    case 1:
#if S4_CAUCHY_PACKED
      return small ? cauchy_launch<1, S4_CAUCHY_RPT1>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<1, S4_CAUCHY_PRPT1_BIG, true>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s,
                                                               pdl);
#else
      return small ? cauchy_launch<1, S4_CAUCHY_RPT1>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<1, S4_CAUCHY_RPT1_BIG>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl);
#endif
    case 2:  // 4 roots per thread on large grids measured 2 % faster (8 at rank 1 was 11 % slower)
      return small ? cauchy_launch<2, 2>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl)
                   : cauchy_launch<2, 4>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl);
    case 3:
      return cauchy_launch<3, 1>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl);
    case 4:
      return cauchy_launch<4, 1>(Lambda, P, Q, B, Ct, dt, Khat, H, N, M, logC, status, s, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace s4impl
