// Host-side plan set-up: the Lloyd-Max codebook and the Haar rotation.
//
// These run once per plan on the CPU and produce inputs of the path (they are
// not steps of it).  Both are written from the mathematics:
//  - "turboquant-pytorch 소개" (discuss.pytorch.kr), "1단계: 랜덤 회전 +
//    Lloyd-Max 양자화": rotate by a random orthogonal matrix, then quantise each
//    coordinate with a precomputed Lloyd-Max codebook for the bell-shaped
//    coordinate distribution (taken as N(0, 1/d)).
//  - Haar-distributed orthogonal matrices: Q of the QR factorisation of a
//    Gaussian matrix, with the column signs fixed so that R has a positive
//    diagonal (Mezzadri, "How to generate random matrices from the classical
//    compact groups", Notices AMS 2007).
#include <cmath>
#include <cstring>
#include <vector>

#include "../../include/tq.h"

namespace {

double normal_pdf(double x) {
  if (std::isinf(x)) return 0.0;
  return std::exp(-0.5 * x * x) * 0.39894228040143267794;  // 1/sqrt(2 pi)
}

// P(a < Z <= b) with the complementary error function taken on the side of the
// tail, so that the outer cells keep their relative precision.
double normal_mass(double a, double b) {
  const double s = 0.70710678118654752440;  // 1/sqrt(2)
  if (a >= 0.0) return 0.5 * (std::erfc(a * s) - std::erfc(b * s));
  if (b <= 0.0) return 0.5 * (std::erfc(-b * s) - std::erfc(-a * s));
  return 1.0 - 0.5 * std::erfc(-a * s) - 0.5 * std::erfc(b * s);
}

double normal_quantile(double p) {  // bisection on the cdf
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (0.5 * std::erfc(-mid * 0.70710678118654752440) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

}  // namespace

extern "C" tq_status tq_lloyd_max_codebook(int levels, int d, float* out) {
  if (!out || d < 1 || !(levels == 2 || levels == 4 || levels == 8 || levels == 16)) return TQ_EINVAL;
  const int L = levels;
  std::vector<double> c(L), next(L), edge(L + 1);
  for (int i = 0; i < L; ++i) c[i] = normal_quantile((i + 0.5) / L);
  for (int it = 0; it < 200000; ++it) {
    edge[0] = -INFINITY;
    edge[L] = INFINITY;
    for (int i = 1; i < L; ++i) edge[i] = 0.5 * (c[i - 1] + c[i]);
    double change = 0.0;
    for (int i = 0; i < L; ++i) {
      // centroid = conditional mean of N(0,1) on its cell
      next[i] = (normal_pdf(edge[i]) - normal_pdf(edge[i + 1])) / normal_mass(edge[i], edge[i + 1]);
      change = std::fmax(change, std::fabs(next[i] - c[i]));
    }
    c.swap(next);
    if (change < 1e-15) break;
  }
  // the N(0,1) quantiser is odd-symmetric; make the rounding noise symmetric too
  for (int i = 0; i < L / 2; ++i) {
    double a = 0.5 * (c[L - 1 - i] - c[i]);
    c[i] = -a;
    c[L - 1 - i] = a;
  }
  const double scale = 1.0 / std::sqrt((double)d);
  for (int i = 0; i < L; ++i) out[i] = (float)(c[i] * scale);
  return TQ_OK;
}

// Parity (Walsh) expansion of a codebook indexed by k = log2(levels) bits:
// with chi_T(idx) = (-1)^popcount(idx & T), the Walsh coefficients are
// w_T = 2^-k sum_idx c[idx] chi_T(idx), and since chi_T = 1 - 2 parity(idx & T),
//   c[idx] = c[0] + sum_{T != 0} (-2 w_T) parity(idx & T).
// Sums of at most 16 fp32 values scaled by a power of two are exact in fp64,
// so a codebook that is exactly odd-symmetric (c[L-1-i] = -c[i]) gets exactly
// zero weight on every even-weight mask and those terms are dropped.
extern "C" tq_status tq_codebook_parity_expansion(int levels, const float* codebook, int* n_terms,
                                                  unsigned* masks, double* coefs, double* c0) {
  if (!codebook || !n_terms || !masks || !coefs || !c0) return TQ_EINVAL;
  if (!(levels == 2 || levels == 4 || levels == 8 || levels == 16)) return TQ_EINVAL;
  int n = 0;
  for (int T = 1; T < levels; ++T) {
    double w = 0.0;
    for (int idx = 0; idx < levels; ++idx) {
      const double c = (double)codebook[idx];
      w += (__builtin_popcount((unsigned)(idx & T)) & 1) ? -c : c;
    }
    w /= (double)levels;
    if (w != 0.0) {
      masks[n] = (unsigned)T;
      coefs[n] = -2.0 * w;
      ++n;
    }
  }
  *n_terms = n;
  *c0 = (double)codebook[0];
  return TQ_OK;
}

extern "C" tq_status tq_haar_rotation(int d, const double* gaussian, float* Pi_out) {
  if (!gaussian || !Pi_out || d < 1 || d > 8192) return TQ_EINVAL;
  const size_t n = (size_t)d;
  std::vector<double> A(gaussian, gaussian + n * n);  // row-major, reduced in place to R
  std::vector<double> V(n * n, 0.0);                  // Householder vectors, V[k] has support k..d-1
  std::vector<double> rdiag(n), w(n);
  for (size_t k = 0; k < n; ++k) {
    // reflect column k (rows k..d-1) onto -sign(a_kk) ||x|| e_k
    double norm2 = 0.0;
    for (size_t i = k; i < n; ++i) norm2 += A[i * n + k] * A[i * n + k];
    double norm = std::sqrt(norm2);
    if (norm == 0.0) return TQ_EINVAL;
    double alpha = A[k * n + k] >= 0.0 ? -norm : norm;
    double* v = &V[k * n];
    for (size_t i = k; i < n; ++i) v[i] = A[i * n + k];
    v[k] -= alpha;
    double vnorm2 = 0.0;
    for (size_t i = k; i < n; ++i) vnorm2 += v[i] * v[i];
    double inv = vnorm2 > 0.0 ? 1.0 / std::sqrt(vnorm2) : 0.0;
    for (size_t i = k; i < n; ++i) v[i] *= inv;
    // A[k:, k:] -= 2 v (v^T A[k:, k:]), row by row so that the inner loops are contiguous
    std::fill(w.begin() + k, w.end(), 0.0);
    for (size_t i = k; i < n; ++i) {
      const double vi = v[i];
      const double* row = &A[i * n];
      for (size_t j = k; j < n; ++j) w[j] += vi * row[j];
    }
    for (size_t i = k; i < n; ++i) {
      const double vi2 = 2.0 * v[i];
      double* row = &A[i * n];
      for (size_t j = k; j < n; ++j) row[j] -= vi2 * w[j];
    }
    rdiag[k] = alpha;
  }
  // Q = H_0 H_1 ... H_{d-1}: accumulate backwards into the identity
  std::vector<double> Q(n * n, 0.0);
  for (size_t i = 0; i < n; ++i) Q[i * n + i] = 1.0;
  for (size_t kk = n; kk-- > 0;) {
    const double* v = &V[kk * n];
    std::fill(w.begin() + kk, w.end(), 0.0);
    for (size_t i = kk; i < n; ++i) {
      const double vi = v[i];
      const double* row = &Q[i * n];
      for (size_t j = kk; j < n; ++j) w[j] += vi * row[j];
    }
    for (size_t i = kk; i < n; ++i) {
      const double vi2 = 2.0 * v[i];
      double* row = &Q[i * n];
      for (size_t j = kk; j < n; ++j) row[j] -= vi2 * w[j];
    }
  }
  // Pi = Q diag(sign R_kk): flip column k where R_kk < 0
  for (size_t i = 0; i < n; ++i)
    for (size_t j = 0; j < n; ++j) {
      double q = Q[i * n + j];
      Pi_out[i * n + j] = (float)(rdiag[j] < 0.0 ? -q : q);
    }
  return TQ_OK;
}
