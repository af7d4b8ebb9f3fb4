// Host-side strategy generation: the covariance a head accumulates, the
// rotation from its eigenvectors, the channel count under a loss threshold,
// and the per-segment channel count of Algorithm 2; and the host side of the
// double-buffered compression (sec. 5.4 of the paperlayer summary): exact
// re-compression of complete blocks into the arena's formats.  Host code only
// (fp64); no device memory, no context.
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

// [S] sec. 5.5: block sizes under a variance threshold.  Per candidate B, the
// mean over the segment's complete blocks of the mean channel variance inside
// each block; the largest B at or under the threshold wins.
extern "C" mk_status mk_choose_block_size(const void* seg, int64_t s, int64_t row_stride, int32_t d,
                                          const int32_t* cands, int32_t n_cands, double threshold,
                                          double* within_var, int32_t* block) {
  if (!seg || !cands || !block || s < 1 || d < 1 || row_stride < d || n_cands < 1 || n_cands > 16 ||
      !(threshold >= 0.0))
    return MK_EINVAL;
  for (int32_t i = 0; i < n_cands; ++i) {
    if (cands[i] < 1) return MK_EINVAL;
    for (int32_t j = 0; j < i; ++j)
      if (cands[j] == cands[i]) return MK_EINVAL;
  }
  int32_t best = -1, smallest = cands[0];
  std::vector<double> mean((size_t)d), var((size_t)d);
  for (int32_t i = 0; i < n_cands; ++i) {
    const int32_t B = cands[i];
    smallest = std::min(smallest, B);
    const int64_t nb = s / B;
    double v = std::nan("");
    if (nb > 0) {
      double tot = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        std::fill(mean.begin(), mean.end(), 0.0);
        std::fill(var.begin(), var.end(), 0.0);
        for (int32_t t = 0; t < B; ++t) {
          const uint16_t* row = row_ptr(seg, b * B + t, row_stride);
          for (int32_t c = 0; c < d; ++c) mean[c] += bf16_to_double(row[c]);
        }
        for (int32_t c = 0; c < d; ++c) mean[c] /= (double)B;
        for (int32_t t = 0; t < B; ++t) {
          const uint16_t* row = row_ptr(seg, b * B + t, row_stride);
          for (int32_t c = 0; c < d; ++c) {
            const double dx = bf16_to_double(row[c]) - mean[c];
            var[c] += dx * dx;
          }
        }
        double blk = 0.0;
        for (int32_t c = 0; c < d; ++c) blk += var[c] / (double)B;
        tot += blk / (double)d;
      }
      v = tot / (double)nb;
      if (v <= threshold && B > best) best = B;
    }
    if (within_var) within_var[i] = v;
  }
  *block = best > 0 ? best : smallest;
  return MK_OK;
}

// ---- Host re-compression of complete blocks ([S] sec. 5.4: the CPU side of
// the double-buffered compression).  Same formats as the device path; the
// rotation is exact fp64 rounded once to bf16.
namespace {

// Nearest bf16 value to x, ties to even (8 significant bits; below the
// smallest normal the spacing stays 2^-133); zero comes back as +0.
double bf16_round(double x) {
  if (x == 0.0) return 0.0;
  int e = 0;
  (void)std::frexp(x, &e);
  if (e < -125) e = -125;
  const double ulp = std::ldexp(1.0, e - 8);
  return std::nearbyint(x / ulp) * ulp + 0.0;
}

inline uint16_t bf16_bits(double y) {
  const float f = (float)y;  // exact: y is a bf16 value
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// Channels [0, keep) of y ordered by magnitude descending (ties to the lower
// channel); the first r, in ascending channel order.
void top_r(const double* y, int keep, int r, int* out) {
  std::vector<int> c((size_t)keep);
  std::iota(c.begin(), c.end(), 0);
  std::stable_sort(c.begin(), c.end(), [&](int a, int b) { return std::fabs(y[a]) > std::fabs(y[b]); });
  std::sort(c.begin(), c.begin() + r);
  std::copy(c.begin(), c.begin() + r, out);
}

// Grouped top-r of the bitmap format ([S] sec. 5.1): the r / g groups of g
// adjacent channels with the largest energy, summed in fp32 in channel order
// (every bf16 square is exact in fp32, and the volatile keeps each sum a
// separate rounding), ties to the lower group, among the first keep / g.
void top_groups(const double* y, int keep, int r, int g, int* out) {
  const int ng = keep / g;
  std::vector<float> e((size_t)ng);
  for (int j = 0; j < ng; ++j) {
    float acc = 0.0f;
    for (int i = 0; i < g; ++i) {
      const float x = (float)y[g * j + i];
      volatile float sq = x * x;
      acc = i == 0 ? sq : acc + sq;
    }
    e[(size_t)j] = acc;
  }
  std::vector<int> c((size_t)ng);
  std::iota(c.begin(), c.end(), 0);
  std::stable_sort(c.begin(), c.end(), [&](int a, int b) { return e[(size_t)a] > e[(size_t)b]; });
  std::sort(c.begin(), c.begin() + r / g);
  for (int k = 0; k < r / g; ++k)
    for (int i = 0; i < g; ++i) out[k * g + i] = c[(size_t)k] * g + i;
}

}  // namespace

extern "C" mk_status mk_host_pack_blocks(const float* R_k, const float* R_v, const void* k, const void* v,
                                         int64_t row_stride, int32_t n_blocks, int32_t block, int32_t r,
                                         int32_t keep_channels, int64_t page_stride, int32_t meta_channels,
                                         int32_t page_format, int32_t elem_group, void* pages, void* meta,
                                         void* cmeta) {
  constexpr int D = MK_HEAD_DIM;
  if (!R_k || !R_v || !k || !v || !pages || !meta || n_blocks < 0 || row_stride < D) return MK_EINVAL;
  if (block != 16 && block != 32 && block != 64) return MK_EINVAL;
  if (r < 1 || r > D || (keep_channels != 0 && (keep_channels < r || keep_channels > D))) return MK_EINVAL;
  if (page_format != MK_PAGES_PACKED && page_format != MK_PAGES_BITMAP) return MK_EINVAL;
  if (page_format == MK_PAGES_PACKED ? elem_group != 0
                                     : (elem_group != 0 && elem_group != 1 && elem_group != 2 && elem_group != 4 &&
                                        elem_group != 8))
    return MK_EINVAL;
  const int g = page_format == MK_PAGES_BITMAP ? (elem_group ? elem_group : 1) : 0;
  if (g > 1 && (r % g || keep_channels % g)) return MK_EINVAL;
  const int pb = g ? D / g / 8 : r;  // position bytes per token: bitmap or uint8 indices
  if (page_stride < (int64_t)block * (4 * r + 2 * pb)) return MK_EINVAL;
  if (meta_channels < 0 || meta_channels > MK_MAX_META_CHANNELS || (meta_channels > 0 && !cmeta)) return MK_EINVAL;
  const int keep = keep_channels ? keep_channels : D;
  const int64_t crow = meta_channels > 0 ? (5 * meta_channels + 15) / 16 * 16 : 0;
  std::memset(pages, 0, (size_t)n_blocks * (size_t)page_stride);
  if (crow) std::memset(cmeta, 0, (size_t)n_blocks * (size_t)crow);
  const int Br = block * r;
  std::vector<double> x(D), y(D), zk(D);
  std::vector<int> kept((size_t)r);
  for (int32_t b = 0; b < n_blocks; ++b) {
    unsigned char* page = static_cast<unsigned char*>(pages) + (int64_t)b * page_stride;
    double mn[D], mx[D];
    for (int t = 0; t < block; ++t) {
      const int64_t row = (int64_t)b * block + t;
      for (int w = 0; w < 2; ++w) {
        const uint16_t* src = row_ptr(w == 0 ? k : v, row, row_stride);
        const float* R = w == 0 ? R_k : R_v;
        for (int j = 0; j < D; ++j) x[j] = bf16_to_double(src[j]);
        for (int c = 0; c < D; ++c) {
          double acc = 0.0;
          for (int j = 0; j < D; ++j) acc += x[j] * (double)R[(size_t)c * D + j];
          y[c] = bf16_round(acc);
        }
        if (g > 1)
          top_groups(y.data(), keep, r, g, kept.data());
        else
          top_r(y.data(), keep, r, kept.data());
        // [K values B r][K positions B pb][V values B r][V positions B pb]
        uint16_t* val = reinterpret_cast<uint16_t*>(page + (w == 0 ? 0 : 2 * Br + block * pb));
        uint8_t* pos = page + (w == 0 ? 2 * Br : 4 * Br + block * pb) + t * pb;
        for (int i = 0; i < r; ++i) {
          val[t * r + i] = bf16_bits(y[kept[i]]);
          if (g) {
            const int j = kept[i] / g;  // bit j of the bitmap: byte j / 8, bit j % 8
            pos[j >> 3] = (uint8_t)(pos[j >> 3] | (1u << (j & 7)));
          } else {
            pos[i] = (uint8_t)kept[i];
          }
        }
        if (w == 0) {
          // min/max over the block of the zero-filled compressed key
          std::fill(zk.begin(), zk.end(), 0.0);
          for (int i = 0; i < r; ++i) zk[kept[i]] = y[kept[i]];
          for (int c = 0; c < D; ++c) {
            mn[c] = t == 0 ? zk[c] : std::min(mn[c], zk[c]);
            mx[c] = t == 0 ? zk[c] : std::max(mx[c], zk[c]);
          }
        }
      }
    }
    uint16_t* mrow = static_cast<uint16_t*>(meta) + (int64_t)b * 2 * D;
    for (int c = 0; c < D; ++c) {
      mn[c] += 0.0;  // a zero bound is +0
      mx[c] += 0.0;
      mrow[c] = bf16_bits(mn[c]);
      mrow[D + c] = bf16_bits(mx[c]);
    }
    if (crow) {
      double wgt[D];
      for (int c = 0; c < D; ++c) wgt[c] = std::max(std::fabs(mn[c]), std::fabs(mx[c]));
      std::vector<int> ck((size_t)meta_channels);
      top_r(wgt, D, meta_channels, ck.data());
      unsigned char* cr = static_cast<unsigned char*>(cmeta) + (int64_t)b * crow;
      uint16_t* cmn = reinterpret_cast<uint16_t*>(cr);
      uint16_t* cmx = cmn + meta_channels;
      uint8_t* cch = reinterpret_cast<uint8_t*>(cmx + meta_channels);
      for (int i = 0; i < meta_channels; ++i) {
        cmn[i] = bf16_bits(mn[ck[i]]);
        cmx[i] = bf16_bits(mx[ck[i]]);
        cch[i] = (uint8_t)ck[i];
      }
    }
  }
  return MK_OK;
}
