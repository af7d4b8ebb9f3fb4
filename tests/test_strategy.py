"""Host-side strategy generation: the oracle pinned to closed forms, brute
force and a library eigensolver; the library's native calls checked against
the oracle on seeded inputs.  CPU only (the native calls touch no GPU)."""
import ctypes
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import strategy_oracle as SO  # noqa: E402


def _bf16_words(X):
    """Round X to bf16 (nearest even) and return (words, the bf16 values as float64)."""
    f = np.ascontiguousarray(X, dtype=np.float32).view(np.uint32)
    rounded = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    vals = (rounded.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return rounded, vals


def _lib():
    from compressed_kv_cache_vector_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding


# ---- oracle pins --------------------------------------------------------------

def test_oracle_cov_update_equals_sum_of_outer_products():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((5, 3))
    G0 = rng.standard_normal((3, 3))
    G0 = G0 + G0.T
    want = G0.copy()
    for x in X:                      # brute force: one outer product per row
        for a in range(3):
            for b in range(3):
                want[a, b] += x[a] * x[b]
    assert np.allclose(SO.cov_update(G0, X), want, rtol=0, atol=1e-12)


def test_oracle_rotation_of_a_diagonal_matrix_is_a_permutation():
    diag = np.array([2.0, 7.0, 1.0, 5.0])
    R, lam = SO.rotation_from_cov(np.diag(diag))
    assert np.array_equal(lam, np.array([7.0, 5.0, 2.0, 1.0]))
    assert np.array_equal(np.abs(R), np.eye(4)[[1, 3, 0, 2]])


def test_oracle_rotation_invariants():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((300, 16)) * 0.9 ** np.arange(16)
    G = X.T @ X
    R, lam = SO.rotation_from_cov(G)
    assert np.all(np.diff(lam) <= 0)
    assert np.allclose(R @ R.T, np.eye(16), atol=1e-12)
    assert np.allclose(R @ G @ R.T, np.diag(lam), atol=1e-9 * lam[0])
    # Energy(r) of the rotated keys equals the eigenvalue share ([N] Eq. (5)).
    Xr = X @ R.T
    for r in (1, 4, 9):
        e = (Xr[:, :r] ** 2).sum() / (X ** 2).sum()
        assert abs((1.0 - e) - SO.discarded_energy(lam, r)) < 1e-12


@pytest.mark.parametrize("rho,eps", [(0.5, 0.01), (0.9, 0.05), (0.8, 0.2)])
def test_oracle_choose_r_geometric_spectrum(rho, eps):
    d = 16
    lam = rho ** np.arange(d)
    # closed form: loss(r) = (rho^r - rho^d) / (1 - rho^d)
    want = next(r for r in range(1, d + 1) if (rho ** r - rho ** d) / (1 - rho ** d) <= eps + 1e-15)
    assert SO.choose_r(lam, eps) == want


def test_oracle_choose_r_special_cases():
    assert SO.choose_r(np.zeros(8), 0.1) == 1
    assert SO.choose_r(np.array([3.0, 2.0, 0.0, 0.0]), 0.0) == 2
    assert SO.choose_r(np.array([1.0, 1.0, 1.0, 1.0]), 0.5) == 2
    assert SO.choose_r(np.array([1.0, 1.0, 1.0, 1.0]), 0.49) == 3


def test_oracle_alg2_constant_segment():
    S = np.full((10, 4), 2.0)
    r, st = SO.alg2_segment_r(S, budget=200.0, outlier_abs=1.0, outlier_ratio_max=0.5, alpha=0.5,
                              r_min=1, r_max=64, hist_bins=8)
    assert st == {"variance": 0.0, "outlier_ratio": 1.0, "entropy": 0.0}
    assert r == math.floor(200.0 / 10 * (1 - 0.5 * 1.0))   # many outliers: compressed harder


def test_oracle_alg2_two_level_segment():
    # Channel c alternates 0 and 1 down the tokens: variance 1/4 per channel,
    # half the magnitudes in the first bin and half in the last: entropy ln 2.
    S = np.tile(np.array([[0.0], [1.0]]), (8, 6))
    r, st = SO.alg2_segment_r(S, budget=160.0, outlier_abs=2.0, outlier_ratio_max=0.1, alpha=0.25,
                              r_min=4, r_max=12, hist_bins=4)
    assert st["variance"] == pytest.approx(0.25, abs=1e-15)
    assert st["outlier_ratio"] == 0.0
    assert st["entropy"] == pytest.approx(math.log(2.0), abs=1e-15)
    assert r == 12        # 160/16 * 1.25 = 12.5, clamped to r_max then rounded down


def test_oracle_alg2_clamps_low():
    S = np.full((4, 4), 5.0)
    r, _ = SO.alg2_segment_r(S, budget=4.0, outlier_abs=1.0, outlier_ratio_max=0.5, alpha=0.9,
                             r_min=3, r_max=8, hist_bins=2)
    assert r == 3


# ---- the library's native calls against the oracle ------------------------------

def test_native_cov_update_matches_oracle():
    b = _lib()
    rng = np.random.default_rng(3)
    words, vals = _bf16_words(rng.standard_normal((700, 128)) * 0.92 ** np.arange(128))
    G = np.zeros((128, 128))
    b.cov_update(G, words[:300])
    b.cov_update(G, words[300:])            # incremental: two updates
    want = SO.cov_update(np.zeros((128, 128)), vals)
    assert np.abs(G - want).max() <= 1e-12 * np.abs(want).max()


def test_native_rotation_matches_oracle():
    b = _lib()
    rng = np.random.default_rng(4)
    _, vals = _bf16_words(rng.standard_normal((2000, 128)) * 0.92 ** np.arange(128))
    G = vals.T @ vals
    R, lam = b.rotation_from_cov(G)
    R_o, lam_o = SO.rotation_from_cov(G)
    assert np.abs(lam - lam_o).max() <= 1e-10 * lam_o[0]
    # Rows agree up to sign (the spectrum is distinct): |R R_o^T| = I to fp32 rounding.
    M = np.abs(R.astype(np.float64) @ R_o.T)
    assert np.abs(M - np.eye(128)).max() < 1e-5


def test_native_rotation_diagonal_and_errors():
    b = _lib()
    R, lam = b.rotation_from_cov(np.diag([2.0, 7.0, 1.0, 5.0]))
    assert np.array_equal(lam, np.array([7.0, 5.0, 2.0, 1.0]))
    assert np.array_equal(np.abs(R), np.eye(4, dtype=np.float32)[[1, 3, 0, 2]])
    G = np.array([[1.0, 2.0], [0.0, 1.0]])    # not symmetric
    with pytest.raises(b.MosaicKVError):
        b.rotation_from_cov(G)


@pytest.mark.parametrize("loss", [0.0, 1e-3, 0.01, 0.05, 0.3])
def test_native_choose_r_matches_oracle(loss):
    b = _lib()
    rng = np.random.default_rng(5)
    _, vals = _bf16_words(rng.standard_normal((1500, 128)) * 0.92 ** np.arange(128))
    _, lam = SO.rotation_from_cov(vals.T @ vals)
    lam = np.maximum(lam, 0.0)
    assert b.choose_r(lam, loss) == SO.choose_r(lam, loss)


def test_native_choose_r_errors():
    b = _lib()
    with pytest.raises(b.MosaicKVError):
        b.choose_r(np.array([1.0, 2.0]), 0.1)     # not descending
    with pytest.raises(b.MosaicKVError):
        b.choose_r(np.array([1.0, -0.5]), 0.1)    # negative
    with pytest.raises(b.MosaicKVError):
        b.choose_r(np.array([1.0, 0.5]), -0.1)    # negative threshold


@pytest.mark.parametrize("seed,scale", [(6, 1.0), (7, 0.05), (8, 3.0)])
def test_native_alg2_matches_oracle(seed, scale):
    b = _lib()
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((256, 128)) * 0.92 ** np.arange(128) * scale
    X[rng.random(X.shape) < 0.02] *= 8.0        # outliers
    words, vals = _bf16_words(X)
    args = dict(budget=256 * 38.0, outlier_abs=1.5, outlier_ratio_max=0.01, alpha=0.5, r_min=8, r_max=96,
                hist_bins=32)
    r, st = b.alg2_segment_r(words, **args)
    r_o, st_o = SO.alg2_segment_r(vals, **args)
    assert r == r_o
    for k in st_o:
        assert st[k] == pytest.approx(st_o[k], rel=1e-12, abs=1e-15)


def test_native_alg2_errors():
    b = _lib()
    w, _ = _bf16_words(np.ones((4, 4)))
    with pytest.raises(b.MosaicKVError):
        b.alg2_segment_r(w, budget=10.0, outlier_abs=1.0, outlier_ratio_max=0.1, alpha=0.1, r_min=5, r_max=4,
                         hist_bins=4)
    with pytest.raises(b.MosaicKVError):
        b.alg2_segment_r(w, budget=10.0, outlier_abs=1.0, outlier_ratio_max=0.1, alpha=0.1, r_min=1, r_max=4,
                         hist_bins=0)
    lib = b.load()
    assert lib.mk_cov_update(None, None, 0, 0, 4) == 1     # MK_EINVAL
    r = ctypes.c_int32(0)
    assert lib.mk_choose_r(None, 4, ctypes.c_double(0.1), ctypes.byref(r)) == 1


# ---- block-size choice ([S] sec. 5.5) ------------------------------------------
def _within_loops(S, B):
    """The statistic with explicit loops (per block, per channel, per token)."""
    s, d = len(S), len(S[0])
    nb = s // B
    tot = 0.0
    for b in range(nb):
        acc = 0.0
        for c in range(d):
            col = [S[b * B + t][c] for t in range(B)]
            m = sum(col) / B
            acc += sum((x - m) ** 2 for x in col) / B
        tot += acc / d
    return tot / nb


def test_oracle_within_block_variance_closed_forms_and_loops():
    # Rows constant within 16-token runs, alternating +a / -a between runs:
    # blocks of 16 have variance 0, blocks of 32 or 64 mix the two levels
    # equally, so each channel's variance is a^2.
    a = np.arange(2, 10) / 4.0           # dyadic: block means and variances exact
    S = np.concatenate([np.tile(a if i % 2 == 0 else -a, (16, 1)) for i in range(8)])
    assert SO.within_block_variance(S, 16) == 0.0
    assert SO.within_block_variance(S, 32) == pytest.approx(np.mean(a ** 2), rel=1e-14)
    assert SO.within_block_variance(S, 64) == pytest.approx(np.mean(a ** 2), rel=1e-14)
    assert SO.within_block_variance(S[:10], 16) is None          # no complete block
    rng = np.random.default_rng(40)
    X = rng.standard_normal((70, 5)) * np.arange(1, 6)
    for B in (1, 4, 16, 32):
        assert SO.within_block_variance(X, B) == pytest.approx(_within_loops(X.tolist(), B), rel=1e-12)
    # iid rows of variance sigma^2: the expected population variance of B samples is sigma^2 (1 - 1/B)
    X = rng.standard_normal((64 * 2000, 4)) * 1.5
    for B in (16, 64):
        assert SO.within_block_variance(X, B) == pytest.approx(2.25 * (1 - 1 / B), rel=0.01)


def test_oracle_within_block_variance_rotation_invariant():
    rng = np.random.default_rng(41)
    X = rng.standard_normal((256, 16)) * 0.8 ** np.arange(16)
    Q, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    for B in (16, 32, 64):
        assert SO.within_block_variance(X @ Q.T, B) == pytest.approx(SO.within_block_variance(X, B), rel=1e-12)


def test_oracle_choose_block_size_rule():
    a = np.arange(2, 10) / 4.0           # dyadic: block means and variances exact
    S = np.concatenate([np.tile(a if i % 2 == 0 else -a, (16, 1)) for i in range(8)])
    va2 = float(np.mean(a ** 2))
    assert SO.choose_block_size(S, [16, 32, 64], 0.0)[0] == 16
    assert SO.choose_block_size(S, [64, 16, 32], va2 * 1.001)[0] == 64   # largest under the threshold
    assert SO.choose_block_size(-np.abs(S), [16, 32, 64], 0.0)[0] == 64  # constant rows: every size qualifies
    assert SO.choose_block_size(S + np.arange(128)[:, None], [16, 32, 64], 0.0)[0] == 16  # none: smallest
    B, v = SO.choose_block_size(S[:40], [16, 32, 64], 10.0)
    assert B == 32 and v[2] is None                                      # 64 has no complete block
    # a planted mistake (the smallest qualifying size) fails the rule above
    ok = [Bc for Bc, x in zip([16, 32, 64], SO.choose_block_size(S, [16, 32, 64], va2 * 1.001)[1]) if x <= va2 * 1.001]
    assert min(ok) != SO.choose_block_size(S, [16, 32, 64], va2 * 1.001)[0]


@pytest.mark.parametrize("seed,smooth", [(42, 0.0), (43, 0.9), (44, 0.99)])
def test_native_choose_block_size_matches_oracle(seed, smooth):
    # Keys that drift slowly along the sequence (an AR(1) walk of strength
    # `smooth`) favour large blocks; iid keys favour none.
    b = _lib()
    rng = np.random.default_rng(seed)
    n, d = 1000, 128
    X = np.empty((n, d))
    X[0] = rng.standard_normal(d)
    for t in range(1, n):
        X[t] = smooth * X[t - 1] + math.sqrt(1 - smooth ** 2) * rng.standard_normal(d)
    X *= 0.92 ** np.arange(d)
    words, vals = _bf16_words(X)
    cands = [64, 16, 32, 512, 2048]
    for thr in (0.0, 0.01, 0.05, 0.2, 1.0):
        B, v = b.choose_block_size(words, cands, thr)
        B_o, v_o = SO.choose_block_size(vals, cands, thr)
        assert B == B_o
        order = sorted(cands)
        for i, c in enumerate(cands):
            want = v_o[order.index(c)]
            if want is None:
                assert math.isnan(v[i])
            else:
                assert v[i] == pytest.approx(want, rel=1e-12, abs=1e-15)


def test_native_choose_block_size_errors():
    b = _lib()
    w, _ = _bf16_words(np.ones((64, 8)))
    for cands, thr in (([16, 16], 0.1), ([0, 16], 0.1), ([], 0.1), ([16], -1.0), ([16], float("nan")),
                       (list(range(1, 18)), 0.1)):
        with pytest.raises(b.MosaicKVError):
            b.choose_block_size(w, cands, thr)
    assert b.choose_block_size(w, [128, 16], 0.0)[0] == 16      # 128 has no complete block
