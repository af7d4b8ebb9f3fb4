// Host-side strategy generation: the covariance a head accumulates, the
// rotation from its eigenvectors, the channel count under a loss threshold,
// and the per-segment channel count of Algorithm 2.  Host code only (fp64);
// no device memory, no context.
//
// Method: "MosaicKV：...阅读笔记" (zhongzhuzhou.org): Eq. (4) and (6) (the
// rotation R from the eigenvectors of K^T K, eigenvalues descending), Eq. (5)
// (Energy(r), the share of the spectrum the first r rotated channels keep),
// Eq. (10)-(11) and Algorithm 2 (per-segment channel count from the
// segment's variance, outlier ratio and magnitude entropy); "MosaicKV:
// Serving Long-Context LLM with Dynamic Two-D KV Cache Compression"
// (paperlayer.ai), sec. 5.5 (the CPU updates the covariance incrementally and
// picks channel parameters under a loss threshold).
//
// The eigen-decomposition is the cyclic Jacobi method for symmetric matrices
// (Golub and Van Loan, "Matrix Computations", sec. 8.5): each step zeroes one
// off-diagonal pair with a plane rotation whose angle comes from the 2x2
// symmetric Schur decomposition; sweeps run over all pairs until the
// off-diagonal mass is negligible.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "../../include/mosaickv.h"

namespace {

inline double bf16_to_double(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

inline const uint16_t* row_ptr(const void* base, int64_t i, int64_t stride) {
  return static_cast<const uint16_t*>(base) + i * stride;
}

}  // namespace

extern "C" mk_status mk_cov_update(double* G, const void* x, int64_t n, int64_t row_stride, int32_t d) {
  if (!G || (!x && n > 0) || d < 1 || n < 0 || (n > 0 && row_stride < d)) return MK_EINVAL;
  std::vector<double> xr((size_t)d);
  for (int64_t i = 0; i < n; ++i) {
    const uint16_t* row = row_ptr(x, i, row_stride);
    for (int32_t c = 0; c < d; ++c) xr[c] = bf16_to_double(row[c]);
    for (int32_t a = 0; a < d; ++a) {
      const double xa = xr[a];
      if (xa == 0.0) continue;
      double* ga = G + (size_t)a * d;
      for (int32_t b = a; b < d; ++b) ga[b] += xa * xr[b];
    }
  }
  // The loop above fills the upper triangle; mirror it.
  for (int32_t a = 0; a < d; ++a)
    for (int32_t b = a + 1; b < d; ++b) G[(size_t)b * d + a] = G[(size_t)a * d + b];
  return MK_OK;
}

extern "C" mk_status mk_rotation_from_cov(const double* G, int32_t d, float* R, double* lambda) {
  if (!G || !R || !lambda || d < 1) return MK_EINVAL;
  const size_t n = (size_t)d;
  double scale = 0.0;
  for (size_t i = 0; i < n * n; ++i) scale = std::max(scale, std::fabs(G[i]));
  for (size_t a = 0; a < n; ++a)
    for (size_t b = a + 1; b < n; ++b)
      if (std::fabs(G[a * n + b] - G[b * n + a]) > 1e-12 * std::max(scale, 1e-300)) return MK_EINVAL;

  std::vector<double> A(G, G + n * n), V(n * n, 0.0);
  for (size_t i = 0; i < n; ++i) V[i * n + i] = 1.0;
  double fro = 0.0;
  for (size_t i = 0; i < n * n; ++i) fro += A[i] * A[i];
  fro = std::sqrt(fro);
  bool converged = fro == 0.0;
  for (int sweep = 0; sweep < 100 && !converged; ++sweep) {
    double off = 0.0;
    for (size_t p = 0; p < n; ++p)
      for (size_t q = p + 1; q < n; ++q) off += A[p * n + q] * A[p * n + q];
    if (std::sqrt(2.0 * off) <= 1e-15 * fro) {
      converged = true;
      break;
    }
    for (size_t p = 0; p + 1 < n; ++p) {
      for (size_t q = p + 1; q < n; ++q) {
        const double apq = A[p * n + q];
        if (apq == 0.0) continue;
        // 2x2 symmetric Schur: (c, s) with [c s; -s c]^T [app apq; apq aqq] [c s; -s c] diagonal.
        const double tau = (A[q * n + q] - A[p * n + p]) / (2.0 * apq);
        const double t = (tau >= 0.0 ? 1.0 : -1.0) / (std::fabs(tau) + std::sqrt(1.0 + tau * tau));
        const double c = 1.0 / std::sqrt(1.0 + t * t), s = t * c;
        // A <- J^T A J with J the rotation in the (p, q) plane: columns, then rows.
        for (size_t k = 0; k < n; ++k) {
          const double akp = A[k * n + p], akq = A[k * n + q];
          A[k * n + p] = c * akp - s * akq;
          A[k * n + q] = s * akp + c * akq;
        }
        for (size_t k = 0; k < n; ++k) {
          const double apk = A[p * n + k], aqk = A[q * n + k];
          A[p * n + k] = c * apk - s * aqk;
          A[q * n + k] = s * apk + c * aqk;
        }
        A[p * n + q] = A[q * n + p] = 0.0;
        // V <- V J (columns of V are the eigenvectors).
        for (size_t k = 0; k < n; ++k) {
          const double vkp = V[k * n + p], vkq = V[k * n + q];
          V[k * n + p] = c * vkp - s * vkq;
          V[k * n + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  // Eigenvalues descending (ties keep the lower index first); row i of R is
  // the eigenvector of lambda[i].
  std::vector<size_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) { return A[a * n + a] > A[b * n + b]; });
  for (size_t i = 0; i < n; ++i) {
    const size_t j = order[i];
    lambda[i] = A[j * n + j];
    for (size_t k = 0; k < n; ++k) R[i * n + k] = (float)V[k * n + j];
  }
  return converged ? MK_OK : MK_ETIMEOUT;
}

extern "C" mk_status mk_choose_r(const double* lambda, int32_t d, double loss_max, int32_t* r) {
  if (!lambda || !r || d < 1 || !(loss_max >= 0.0)) return MK_EINVAL;
  const double tol = 1e-9 * std::fabs(lambda[0]);
  for (int32_t i = 0; i < d; ++i) {
    if (lambda[i] < -tol) return MK_EINVAL;
    if (i > 0 && lambda[i] > lambda[i - 1] + tol) return MK_EINVAL;
  }
  // tail[i] = sum_{j >= i} lambda_j (tiny negative roundoff counts as zero).
  std::vector<double> tail((size_t)d + 1, 0.0);
  for (int32_t i = d - 1; i >= 0; --i) tail[i] = tail[i + 1] + std::max(0.0, lambda[i]);
  const double total = tail[0];
  if (total <= 0.0) {
    *r = 1;
    return MK_OK;
  }
  for (int32_t k = 1; k <= d; ++k) {
    if (tail[k] <= loss_max * total) {
      *r = k;
      return MK_OK;
    }
  }
  *r = d;
  return MK_OK;
}

extern "C" mk_status mk_alg2_segment_r(const void* seg, int64_t s, int64_t row_stride, int32_t d, double budget,
                                       const mk_alg2_params* p, mk_seg_stats* stats, int32_t* r) {
  if (!seg || !p || !r || s < 1 || d < 1 || row_stride < d || p->hist_bins < 1 || p->r_min < 1 ||
      p->r_max < p->r_min || !(budget >= 0.0))
    return MK_EINVAL;
  // Channel means, then the population variance of each channel.
  std::vector<double> mean((size_t)d, 0.0), var((size_t)d, 0.0);
  double amax = 0.0;
  int64_t n_out = 0;
  for (int64_t i = 0; i < s; ++i) {
    const uint16_t* row = row_ptr(seg, i, row_stride);
    for (int32_t c = 0; c < d; ++c) {
      const double x = bf16_to_double(row[c]);
      mean[c] += x;
      amax = std::max(amax, std::fabs(x));
      if (std::fabs(x) > p->outlier_abs) ++n_out;
    }
  }
  for (int32_t c = 0; c < d; ++c) mean[c] /= (double)s;
  std::vector<int64_t> hist((size_t)p->hist_bins, 0);
  for (int64_t i = 0; i < s; ++i) {
    const uint16_t* row = row_ptr(seg, i, row_stride);
    for (int32_t c = 0; c < d; ++c) {
      const double x = bf16_to_double(row[c]);
      const double dx = x - mean[c];
      var[c] += dx * dx;
      int64_t b = 0;
      if (amax > 0.0) b = std::min<int64_t>(p->hist_bins - 1, (int64_t)std::floor(std::fabs(x) / amax * p->hist_bins));
      ++hist[(size_t)b];
    }
  }
  double variance = 0.0;
  for (int32_t c = 0; c < d; ++c) variance += var[c] / (double)s;
  variance /= (double)d;
  const double n_el = (double)s * (double)d;
  const double outlier_ratio = (double)n_out / n_el;
  double entropy = 0.0;
  for (int64_t h : hist)
    if (h > 0) {
      const double q = (double)h / n_el;
      entropy -= q * std::log(q);
    }
  // Algorithm 2: a segment with many outliers is compressed harder.
  const double per_vec = budget / (double)s;
  double rr = outlier_ratio > p->outlier_ratio_max ? per_vec * (1.0 - p->alpha * outlier_ratio)
                                                   : per_vec * (1.0 + p->alpha * (1.0 - outlier_ratio));
  rr = std::min((double)p->r_max, std::max((double)p->r_min, rr));
  *r = (int32_t)std::floor(rr);
  if (stats) {
    stats->variance = variance;
    stats->outlier_ratio = outlier_ratio;
    stats->entropy = entropy;
  }
  return MK_OK;
}
