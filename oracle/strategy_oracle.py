"""fp64 oracle for MosaicKV's host-side strategy generation.  TEST INFRASTRUCTURE.

This module is test infrastructure, not the product: only the test suite may import
it.  The library's native strategy calls (mk_cov_update, mk_rotation_from_cov,
mk_choose_r, mk_alg2_segment_r, mk_choose_block_size) never do, and this module
imports nothing from them.

Each function writes out the definition it follows in float64, with numpy's
matmul and eigh as the only library steps.

Sources (cited by page title and equation/section):
  [N] "MosaicKV：面向超长上下文LLM服务的动态二维KV缓存压缩——阅读笔记"
      (reading notes on zhongzhuzhou.org): Eq. (4) and (6) (rotation from the
      eigenvectors of K^T K), Eq. (5) (Energy(r)), Eq. (10)-(11) and
      Algorithm 2 (per-segment channel count).
  [S] "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV Cache
      Compression" (paperlayer.ai summary): sec. 5.5 (incremental covariance,
      channel parameters under a loss threshold, block sizes under a variance
      threshold).

Readings where the pages are silent:
  * the covariance is the uncentred second moment sum x^T x ([N] Eq. (4)
    rotates by the eigenvectors of K^T K);
  * the loss of keeping r channels is the discarded energy 1 - Energy(r);
    the chosen r is the smallest in [1, d] with loss <= the threshold;
  * Algorithm 2: "variance" is the mean over channels of each channel's
    population variance; the magnitude histogram has a given number of equal
    bins over [0, max |x|] (a value at the maximum goes to the last bin); the
    entropy uses the natural log; the clamped r is rounded down;
  * block size ([S] sec. 5.5 chooses block sizes under a variance
    threshold): a candidate B cuts the segment into its complete blocks of B
    consecutive tokens; its within-block variance is the mean over those
    blocks of the mean over channels of each channel's population variance
    inside the block (Algorithm 2's statistic, taken per block); the chosen B
    is the largest candidate whose within-block variance is at most the
    threshold, else the smallest candidate.  The statistic is the trace of
    the within-block covariance over d, so it does not change under a
    rotation of the channels.

Parity status: every function is pinned by tests/test_strategy.py (brute
force, closed forms, invariants, a library eigensolver).
"""
import numpy as np


def cov_update(G, X):
    """G + X^T X ([S] sec. 5.5: the covariance grows by each new token's x^T x)."""
    X = np.asarray(X, dtype=np.float64)
    return np.asarray(G, dtype=np.float64) + X.T @ X


def rotation_from_cov(G):
    """([N] Eq. (4), (6)) eigenvalues of the symmetric G in descending order
    and R whose row i is the eigenvector of the i-th, so k' = k R^T."""
    lam, vecs = np.linalg.eigh(np.asarray(G, dtype=np.float64))
    order = np.argsort(-lam, kind="stable")
    return vecs[:, order].T.copy(), lam[order].copy()


def discarded_energy(lam, r):
    """1 - Energy(r) of [N] Eq. (5): the share of the spectrum beyond the first r channels."""
    lam = np.maximum(np.asarray(lam, dtype=np.float64), 0.0)
    total = lam.sum()
    return 0.0 if total <= 0 else lam[r:].sum() / total


def choose_r(lam, loss_max):
    """Smallest r in [1, d] whose discarded energy is at most loss_max ([S] sec. 5.5)."""
    lam = np.asarray(lam, dtype=np.float64)
    d = lam.shape[0]
    if np.maximum(lam, 0.0).sum() <= 0:
        return 1
    for r in range(1, d + 1):
        if discarded_energy(lam, r) <= loss_max:
            return r
    return d


def segment_stats(S, outlier_abs, hist_bins):
    """The statistics [N] Algorithm 2 computes for a rotated segment S (s x d)."""
    S = np.asarray(S, dtype=np.float64)
    s, d = S.shape
    variance = float(np.mean(np.var(S, axis=0)))
    outlier_ratio = float(np.count_nonzero(np.abs(S) > outlier_abs)) / (s * d)
    a = np.abs(S).ravel()
    amax = a.max()
    if amax > 0:
        bins = np.minimum(hist_bins - 1, np.floor(a / amax * hist_bins)).astype(np.int64)
    else:
        bins = np.zeros(a.shape, dtype=np.int64)
    p = np.bincount(bins, minlength=hist_bins) / a.size
    p = p[p > 0]
    entropy = float(-(p * np.log(p)).sum())
    return {"variance": variance, "outlier_ratio": outlier_ratio, "entropy": entropy}


def alg2_segment_r(S, budget, outlier_abs, outlier_ratio_max, alpha, r_min, r_max, hist_bins):
    """[N] Algorithm 2 (and Eq. (10)-(11)): a segment with many outliers keeps
    fewer channels, a uniform one more; the result is clamped to
    [r_min, r_max] and rounded down."""
    st = segment_stats(S, outlier_abs, hist_bins)
    s = np.asarray(S).shape[0]
    u = st["outlier_ratio"]
    if u > outlier_ratio_max:
        r = budget / s * (1.0 - alpha * u)
    else:
        r = budget / s * (1.0 + alpha * (1.0 - u))
    r = min(float(r_max), max(float(r_min), r))
    return int(np.floor(r)), st


def within_block_variance(S, B):
    """Mean over the complete blocks of B consecutive rows of S (s x d) of the
    mean over channels of the population variance inside the block; None when
    S holds no complete block."""
    S = np.asarray(S, dtype=np.float64)
    nb = S.shape[0] // B
    if nb == 0:
        return None
    blocks = S[:nb * B].reshape(nb, B, S.shape[1])
    return float(np.mean(np.var(blocks, axis=1)))


def choose_block_size(S, candidates, threshold):
    """[S] sec. 5.5: the largest candidate block size whose within-block
    variance is at most the threshold, else the smallest candidate.
    Returns (block size, [within-block variance or None per candidate])."""
    cands = sorted(int(c) for c in candidates)
    v = [within_block_variance(S, B) for B in cands]
    ok = [B for B, x in zip(cands, v) if x is not None and x <= threshold]
    return (max(ok) if ok else cands[0]), v

