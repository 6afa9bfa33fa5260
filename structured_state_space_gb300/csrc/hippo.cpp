// HiPPO generators in DPLR form: host float64 routine of libs4.
//
// Page "Recurrent, LSTM, and structured state-space models": the LegS, LegT
// and LagT generators (entry formulas), the LegT diagonal similarity S_0, the
// statement that each similar generator is a normal matrix minus a rank-1
// (LegS, LagT) or rank-2 (LegT) term, and the DPLR / NPLR definitions with
// the unitary state change that maps B, C to V^* B, V^* C.
//
// Steps:
//  1. Gt = S^{-1} G S (S = I, or S_0 for LegT), entry by entry.
//  2. Gt = H - U U^T with U read off the entries:
//       LegS u_n = sqrt(n + 1/2); LagT u_n = sqrt(1/2);
//       LegT u = [r, r z] / sqrt(2 theta), r_n = sqrt(2n+1), z_n = (-1)^n.
//     In each case H = c I + S with S real skew-symmetric (c = -1/2 for LegS
//     and LagT, 0 for LegT); the routine checks this before going on.
//  3. The Hermitian matrix K = -i S (purely imaginary) is diagonalised by
//     cyclic Jacobi rotations, K = W diag(mu) W^*; then H = W diag(c + i mu) W^*.
//  4. P = W^* U, B~ = W^* S^{-1} B, C~ = W^* S C (S real diagonal).
#include <algorithm>
#include <cmath>
#include <complex>
#include <numeric>
#include <vector>

#include "s4.h"

namespace {

using cplx = std::complex<double>;

// Cyclic Jacobi eigen-iteration for a Hermitian n x n matrix A (row-major,
// overwritten).  On success mu holds the eigenvalues and VT (row-major, ROW j
// = eigenvector j) the rows of V^T for a unitary V with A_in = V diag(mu) V^*.
// Each rotation J (identity outside rows/columns p, q) is a phase that makes
// the (p, q) block real, followed by the real rotation that zeroes it; the
// new rows p, q of J^* A J are formed from the old rows and mirrored into the
// columns (A stays Hermitian), so every update streams contiguous rows.
bool jacobi_hermitian(std::vector<cplx>& A, int n, std::vector<double>& mu, std::vector<cplx>& VT) {
  VT.assign((size_t)n * n, cplx(0.0, 0.0));
  for (int i = 0; i < n; ++i) VT[(size_t)i * n + i] = 1.0;
  auto at = [&](int i, int j) -> cplx& { return A[(size_t)i * n + j]; };
  double total = 0.0;
  for (const cplx& v : A) total += std::norm(v);
  const double tol = 1e-28 * std::max(total, 1e-300);  // off-diagonal norm <= 1e-14 of the total
  bool converged = false;
  for (int sweep = 0; sweep < 60 && !converged; ++sweep) {
    double off = 0.0;
    for (int p = 0; p < n; ++p)
      for (int q = p + 1; q < n; ++q) off += std::norm(at(p, q));
    if (2.0 * off <= tol) {
      converged = true;
      break;
    }
    for (int p = 0; p < n - 1; ++p) {
      for (int q = p + 1; q < n; ++q) {
        const cplx b = at(p, q);
        const double babs = std::abs(b);
        if (babs == 0.0) continue;
        const double a = at(p, p).real(), d = at(q, q).real();
        // with e^{i phi} = b/|b|, the phase diag(1, e^{-i phi}) turns the block
        // into [[a, |b|], [|b|, d]]; t = tan(theta) is the smaller root of
        // t^2 + 2 zeta t - 1 = 0, zeta = (d - a)/(2|b|).
        const double zeta = (d - a) / (2.0 * babs);
        const double t = (zeta >= 0.0 ? 1.0 : -1.0) / (std::fabs(zeta) + std::sqrt(1.0 + zeta * zeta));
        const double c = 1.0 / std::sqrt(1.0 + t * t), s = t * c;
        // e = e^{-i phi}; J = [[c, s], [-s e, c e]] on (p, q).  Row p of J^* A is
        // c A_p - s conj(e) A_q, row q is s A_p + c conj(e) A_q.
        const double er = b.real() / babs, ei = -b.imag() / babs;
        cplx* rp = &A[(size_t)p * n];
        cplx* rq = &A[(size_t)q * n];
        for (int k = 0; k < n; ++k) {
          if (k == p || k == q) continue;
          const double xr = rp[k].real(), xi = rp[k].imag(), yr = rq[k].real(), yi = rq[k].imag();
          const double ye_r = yr * er + yi * ei, ye_i = yi * er - yr * ei;  // conj(e) y
          rp[k] = cplx(c * xr - s * ye_r, c * xi - s * ye_i);
          rq[k] = cplx(s * xr + c * ye_r, s * xi + c * ye_i);
          at(k, p) = std::conj(rp[k]);
          at(k, q) = std::conj(rq[k]);
        }
        at(p, p) = a - t * babs;
        at(q, q) = d + t * babs;
        at(p, q) = at(q, p) = 0.0;
        // V J: columns p, q of V are rows p, q of VT; column p of V J is
        // c V_p - s e V_q, column q is s V_p + c e V_q.
        cplx* vp = &VT[(size_t)p * n];
        cplx* vq = &VT[(size_t)q * n];
        for (int k = 0; k < n; ++k) {
          const double xr = vp[k].real(), xi = vp[k].imag(), yr = vq[k].real(), yi = vq[k].imag();
          const double ye_r = yr * er - yi * ei, ye_i = yr * ei + yi * er;  // e y
          vp[k] = cplx(c * xr - s * ye_r, c * xi - s * ye_i);
          vq[k] = cplx(s * xr + c * ye_r, s * xi + c * ye_i);
        }
      }
    }
  }
  if (!converged) return false;
  mu.resize(n);
  for (int i = 0; i < n; ++i) mu[i] = at(i, i).real();
  for (double m : mu)
    if (!std::isfinite(m)) return false;
  return true;
}

}  // namespace

extern "C" s4_status s4_hippo_dplr(int kind, int N, double theta, const double* B, const double* C,
                                   double* Lambda, double* P, double* Bt, double* Ct, int* rank) {
  if (kind < S4_HIPPO_LEGS || kind > S4_HIPPO_LAGT || N < 1 || N > 512 || !Lambda || !P || !rank)
    return S4_ERR_INVALID_ARG;
  if (kind == S4_HIPPO_LEGT && !(theta > 0.0 && std::isfinite(theta))) return S4_ERR_INVALID_ARG;
  if ((B && !Bt) || (C && !Ct)) return S4_ERR_INVALID_ARG;
  const int r = kind == S4_HIPPO_LEGT ? 2 : 1;

  // step 1: similarity diagonal and the similar generator Gt
  std::vector<double> sd(N, 1.0), Gt((size_t)N * N, 0.0);
  for (int n = 0; n < N; ++n)
    if (kind == S4_HIPPO_LEGT) sd[n] = std::sqrt(2.0 * n + 1.0) * ((n & 1) ? -1.0 : 1.0);
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < N; ++k) {
      double g = 0.0;
      if (kind == S4_HIPPO_LEGS) {
        g = n > k ? -std::sqrt((2.0 * n + 1.0) * (2.0 * k + 1.0)) : (n == k ? -(n + 1.0) : 0.0);
      } else if (kind == S4_HIPPO_LEGT) {
        const double sg = ((n - k) & 1) ? -1.0 : 1.0;  // (-1)^(n-k)
        g = n >= k ? -(2.0 * n + 1.0) * sg / theta : -(2.0 * n + 1.0) / theta;
      } else {
        g = n >= k ? -1.0 : 0.0;
      }
      Gt[(size_t)n * N + k] = g * sd[k] / sd[n];
    }
  }
  // step 2: U and H = Gt + U U^T = c I + S
  std::vector<double> U((size_t)N * r);
  for (int n = 0; n < N; ++n) {
    if (kind == S4_HIPPO_LEGS) {
      U[n] = std::sqrt(n + 0.5);
    } else if (kind == S4_HIPPO_LAGT) {
      U[n] = std::sqrt(0.5);
    } else {
      const double rn = std::sqrt(2.0 * n + 1.0) / std::sqrt(2.0 * theta);
      U[(size_t)n * 2] = rn;
      U[(size_t)n * 2 + 1] = (n & 1) ? -rn : rn;
    }
  }
  std::vector<double> Hm((size_t)N * N);
  double hmax = 0.0;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < N; ++k) {
      double uu = 0.0;
      for (int l = 0; l < r; ++l) uu += U[(size_t)n * r + l] * U[(size_t)k * r + l];
      Hm[(size_t)n * N + k] = Gt[(size_t)n * N + k] + uu;
      hmax = std::max(hmax, std::fabs(Hm[(size_t)n * N + k]));
    }
  const double c = kind == S4_HIPPO_LEGT ? 0.0 : -0.5;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k <= n; ++k) {
      const double sym = 0.5 * (Hm[(size_t)n * N + k] + Hm[(size_t)k * N + n]) - (n == k ? c : 0.0);
      if (std::fabs(sym) > 1e-12 * std::max(1.0, hmax)) return S4_ERR_NONFINITE;
    }
  // step 3: K = -i (H - c I), Hermitian, purely imaginary
  std::vector<cplx> K((size_t)N * N);
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < N; ++k) K[(size_t)n * N + k] = cplx(0.0, -(Hm[(size_t)n * N + k] - (n == k ? c : 0.0)));
  std::vector<double> mu;
  std::vector<cplx> VT;
  if (!jacobi_hermitian(K, N, mu, VT)) return S4_ERR_NONFINITE;
  std::vector<int> ord(N);
  std::iota(ord.begin(), ord.end(), 0);
  std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return mu[a] < mu[b]; });
  // step 4: outputs in ascending order of Im Lambda
  for (int j = 0; j < N; ++j) {
    const int e = ord[j];
    Lambda[2 * j] = c;
    Lambda[2 * j + 1] = mu[e];
    for (int l = 0; l < r; ++l) {  // P_jl = sum_n conj(W_ne) U_nl
      cplx acc = 0.0;
      for (int n = 0; n < N; ++n) acc += std::conj(VT[(size_t)e * N + n]) * U[(size_t)n * r + l];
      P[2 * ((size_t)j * r + l)] = acc.real();
      P[2 * ((size_t)j * r + l) + 1] = acc.imag();
    }
    if (B) {
      cplx acc = 0.0;
      for (int n = 0; n < N; ++n) acc += std::conj(VT[(size_t)e * N + n]) * (cplx(B[2 * n], B[2 * n + 1]) / sd[n]);
      Bt[2 * j] = acc.real();
      Bt[2 * j + 1] = acc.imag();
    }
    if (C) {
      cplx acc = 0.0;
      for (int n = 0; n < N; ++n) acc += std::conj(VT[(size_t)e * N + n]) * (cplx(C[2 * n], C[2 * n + 1]) * sd[n]);
      Ct[2 * j] = acc.real();
      Ct[2 * j + 1] = acc.imag();
    }
  }
  *rank = r;
  return S4_OK;
}
