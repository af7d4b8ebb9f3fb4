"""Pins the fp64 oracle to facts fixed outside itself (runs without a GPU).

Each test checks the oracle against a value the pages print, a closed form, a
library routine, an invariant of the mathematics, or brute force on tiny
inputs.  The mutation tests at the end plant plausible mistakes in copies of
oracle functions and check that a pin catches each of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import mosaickv_oracle as O
from compressed_kv_cache_vector_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 ----
def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    # exact halfway cases: a bf16 value plus half its spacing
    base = torch.tensor(rng.standard_normal(2000), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    half = np.ldexp(1.0, np.frexp(base.astype(np.float64))[1] - 9).astype(np.float32)
    ties = np.concatenate([base + half, base - half]).astype(np.float32)
    for v in (x, ties, np.array([0.0, -0.0, 1.0, 2 ** -126, 3 * 2 ** -130], dtype=np.float32)):
        want = torch.tensor(v).to(torch.bfloat16).double().numpy() + 0.0
        got = O.bf16_round(v.astype(np.float64))
        assert np.array_equal(got, want)
        assert np.array_equal(O.bf16_bits(got), (want.astype(np.float32).view(np.uint32) >> 16))


# ----------------------------------------------------- worked example ----
def _read_golden():
    vec, keep, glob = {}, {}, None
    with open(os.path.join(GOLD, "worked_example_d4.txt"), encoding="utf-8") as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "vector":
                vec[p[1]] = np.array([float(t) for t in p[2:]])
            elif p[0] == "keep":
                keep[p[1]] = int(p[2])
            elif p[0] == "global":
                glob = int(p[1])
    return vec, keep, glob


def test_worked_example_per_vector_vs_global_mask():
    vec, keep, glob = _read_golden()
    X = np.stack([vec["k1"], vec["k2"]])
    idx, vals = O.topr_select(X, 1)
    assert idx[0, 0] == keep["k1"] and idx[1, 0] == keep["k2"]
    assert vals[0, 0] == 10 and vals[1, 0] == 9
    # The page's global channel matches the energy (sum of squares) reading.
    assert O.global_mask_energy(X, 1)[0] == glob
    # Literal var(K', axis 0) on just these two vectors would pick channel 2
    # (variance 19.36 against 16): a discrepancy recorded, not a failure.
    assert O.global_mask_variance(X, 1)[0] == 2


# ------------------------------------------------------------- top-r ----
def _brute_topr(x, r):
    d = len(x)
    valid = []
    for S in itertools.combinations(range(d), r):
        out = [c for c in range(d) if c not in S]
        ok = all(abs(x[c]) > abs(x[o]) or (abs(x[c]) == abs(x[o]) and c < o)
                 for c in S for o in out)
        if ok:
            valid.append(S)
    assert len(valid) == 1
    return list(valid[0])


def test_topr_brute_force_small_d_with_ties():
    rng = np.random.default_rng(2)
    for _ in range(400):
        d = int(rng.integers(2, 9))
        r = int(rng.integers(1, d + 1))
        x = rng.integers(-3, 4, size=d).astype(np.float64)
        x[rng.random(d) < 0.2] = -0.0
        idx, vals = O.topr_select(x, r)
        want = _brute_topr(x, r)
        assert list(idx[0]) == want
        assert np.array_equal(vals[0], x[want])


def test_topr_d128_against_python_sort():
    rng = np.random.default_rng(3)
    X = O.bf16_round(rng.standard_normal((64, 128)) * np.exp(-0.05 * np.arange(128)))
    X[:4, :] = 0.0                     # all-zero vectors keep channels 0..r-1
    X[4, ::2] = X[4, 1::2]             # many exact magnitude ties
    X[5, 10:20] = -X[5, 10:20]
    for r in (1, 32, 38, 64, 128):
        idx, vals = O.topr_select(X, r)
        for i in range(X.shape[0]):
            srt = sorted(range(128), key=lambda c: (-abs(X[i, c]), c))
            assert list(idx[i]) == sorted(srt[:r])
    idx, _ = O.topr_select(X[:4], 38)
    assert np.array_equal(idx, np.tile(np.arange(38), (4, 1)))


def test_topr_truncated_bottom_channels_brute_force():
    # [S] sec. 5.2: only the first `keep` channels are candidates.  Brute
    # force over the truncated vector, and (an independent form) the top-r of
    # the vector whose bottom channels are zeroed, which agrees whenever the
    # candidates hold at least r nonzero magnitudes.
    rng = np.random.default_rng(22)
    for _ in range(300):
        d = int(rng.integers(3, 10))
        keep = int(rng.integers(1, d + 1))
        r = int(rng.integers(1, keep + 1))
        x = rng.integers(-3, 4, size=d).astype(np.float64)
        idx, vals = O.topr_select(x, r, keep)
        want = _brute_topr(x[:keep], r)
        assert list(idx[0]) == want and np.array_equal(vals[0], x[want])
        if np.count_nonzero(x[:keep]) >= r:
            z = x.copy()
            z[keep:] = 0.0
            assert list(O.topr_select(z, r)[0][0]) == want


def test_compressed_block_keys_brute_force_and_full_width():
    # [S] sec. 5.2: per block, the m channels with the largest max(|min|, |max|),
    # ties to the lower channel, ascending; brute force over small rows.
    rng = np.random.default_rng(24)
    for _ in range(200):
        d = int(rng.integers(2, 9))
        m = int(rng.integers(1, d + 1))
        mn = rng.integers(-3, 1, size=(3, d)).astype(np.float64)
        mx = mn + rng.integers(0, 4, size=(3, d))
        idx, cmn, cmx = O.compress_key_rows(mn, mx, m)
        for r in range(3):
            w = np.maximum(np.abs(mn[r]), np.abs(mx[r]))
            want = sorted(sorted(range(d), key=lambda c: (-w[c], c))[:m])
            assert list(idx[r]) == want
            assert np.array_equal(cmn[r], mn[r, want]) and np.array_equal(cmx[r], mx[r, want])
    # Keeping every channel gives back the full keys, so the scores are unchanged.
    mn = rng.standard_normal((5, 128))
    mx = mn + rng.random((5, 128))
    fmn, fmx = O.zero_filled_keys(*O.compress_key_rows(mn, mx, 128))
    assert np.array_equal(fmn, mn) and np.array_equal(fmx, mx)
    q = rng.standard_normal((2, 128))
    assert np.array_equal(O.block_scores(q, fmn, fmx)[1], O.block_scores(q, mn, mx)[1])


# ---------------------------------------------------------- rotation ----
def _gen(T, decay, seed, outliers=True):
    x = synth.lowrank_outlier(T, 128, decay, seed, n_outlier_channels=4 if outliers else 0)
    return synth.bf16_values(x)


def test_rotation_orthogonal_and_preserves_dot_products():
    K = _gen(2048, 0.9, 11)
    R, lam = O.rotation_from_keys(K)
    assert np.allclose(R @ R.T, np.eye(128), atol=1e-12)
    assert np.all(np.diff(lam) <= 1e-9 * lam[0])
    q = np.random.default_rng(4).standard_normal((4, 128))
    Kp = O.rotate(K, R, round_bf16=False)
    qp = q @ R.T
    assert np.allclose(qp @ Kp.T, q @ K.T, rtol=0, atol=1e-10)
    assert np.allclose(np.linalg.norm(Kp, axis=1), np.linalg.norm(K, axis=1), rtol=1e-12)


def test_energy_equals_eigenvalue_share_and_closed_form():
    K = _gen(4096, 0.9, 12)
    R, lam = O.rotation_from_keys(K)
    for r in (1, 8, 32, 64):
        assert abs(O.energy(R, K, r) - lam[:r].sum() / lam.sum()) < 1e-12
    # Without outliers K^T K ~ T Q diag(s^2) Q^T, so Energy(r) ~ sum_{i<r} s_i^2 / sum s_i^2.
    s2 = 0.9 ** (2 * np.arange(128))
    K0 = _gen(20000, 0.9, 13, outliers=False)
    R0, _ = O.rotation_from_keys(K0)
    for r in (4, 16, 32):
        assert abs(O.energy(R0, K0, r) - s2[:r].sum() / s2.sum()) < 0.01
    s2b = 0.92 ** (2 * np.arange(128))
    assert abs(s2b[:38].sum() / s2b.sum() - 0.9982) < 1e-3  # the closed form itself


# ---------------------------------------------------------- segments ----
def test_segment_boundaries_and_k_rule():
    st = O.Strategy(4, 128, 16, [(0, 32, 0), (350, 64, 1), (650, 32, 0)], 0, 100)
    assert O.n_middle_blocks(10000, st) == 617            # ceil(9868 / 16)
    assert O.segment_first_blocks(10000, st) == [0, 219, 406]   # ceil(3496/16), ceil(6496/16)
    assert O.n_select(2040, O.Strategy(4, 128, 16, [(0, 38, 0)], 0, 100)) == 204
    assert O.n_select(4088, O.Strategy(4, 256, 32, [(0, 38, 0)], 0, 100)) == 409
    assert O.n_select(16376, O.Strategy(4, 512, 64, [(0, 38, 0)], 0, 50)) == 819
    assert O.n_select(252, O.Strategy(4, 64, 16, [(0, 32, 0)], 64, 0)) == 64
    assert O.n_select(3, O.Strategy(4, 64, 16, [(0, 32, 0)], 0, 100)) == 1
    assert O.n_select(0, O.Strategy(4, 64, 16, [(0, 32, 0)], 0, 100)) == 0


def test_sizes_and_overheads_printed_on_the_pages():
    assert O.meta_overhead(16) == 0.0625                  # Quest keys: 6.25% at block 16
    assert abs(O.speedup_bound(0.10, 0.30) - 33.333) < 1e-3
    assert O.packed_bytes_per_token(38) == 228
    per_layer = (1048576 - 4 - 512) * 8 * O.packed_bytes_per_token(38)
    assert 1.78 < per_layer / 2 ** 30 < 1.79                  # "about 1.8 GB" per layer


# ------------------------------------------------------- cache build ----
def _cache(T, st, seed, G=4, round_bf16=True, prefill=None, steps=()):
    K = _gen(T, 0.9, seed)
    V = _gen(T, 0.9, seed + 1)
    Rk, _ = O.rotation_from_keys(K)
    Rv, _ = O.rotation_from_keys(V)
    c = O.OracleCache(st, T + 8, round_bf16=round_bf16)
    c.set_rotation(Rk, Rv)
    t0 = prefill if prefill is not None else T
    c.append(K[:t0], V[:t0])
    t = t0
    for n in steps:
        c.append(K[t:t + n], V[t:t + n])
        t += n
    assert t == T
    return c, K, V


def test_incremental_append_equals_batch_append():
    st = O.Strategy(4, 64, 16, [(0, 32, 0), (400, 64, 1), (700, 24, 0)], 0, 100)
    a, _, _ = _cache(1500, st, 20, prefill=1400, steps=(100,))
    b, _, _ = _cache(1500, st, 20, prefill=1400, steps=(1,) * 37 + (50, 13))
    assert a.T == b.T == 1500 and a.n_mid == b.n_mid == 1500 - 64 - 4
    for name in ("Kr", "Vr", "Kt", "Vt", "kidx", "vidx", "kval", "vval", "rtok"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    ma, xa = a.meta()
    mb, xb = b.meta()
    assert np.array_equal(ma, mb) and np.array_equal(xa, xb)
    # meta is the min/max of the zero-filled compressed keys of each block
    for bi in range(a.n_blocks_mid()):
        lo, hi = a.block_tokens(bi)
        assert np.array_equal(ma[bi], a.Kt[lo:hi].min(axis=0))
        assert np.array_equal(xa[bi], a.Kt[lo:hi].max(axis=0))
    assert list(a.window_positions()) == list(range(1500 - 64, 1500))


def test_page_byte_layout():
    st = O.Strategy(0, 1, 16, [(0, 2, 0)])
    c = O.OracleCache(st, 64)
    c.set_rotation(np.eye(128), np.eye(128))
    K = np.zeros((5, 128))
    V = np.zeros((5, 128))
    K[0, 7], K[0, 3], K[0, 100] = 1.5, -2.0, 0.25
    V[0, 0], V[0, 127] = 3.0, -1.0
    c.append(K, V)                        # 4 tokens in the middle, 1 in the window
    pg = c.page_bytes(0)
    assert pg.size == 6 * 16 * 2
    kv = pg[:64].view(np.uint16).reshape(16, 2)
    ki = pg[64:96].reshape(16, 2)
    vv = pg[96:160].view(np.uint16).reshape(16, 2)
    vi = pg[160:192].reshape(16, 2)
    assert list(ki[0]) == [3, 7] and list(O.bits_to_value(kv[0])) == [-2.0, 1.5]
    assert list(vi[0]) == [0, 127] and list(O.bits_to_value(vv[0])) == [3.0, -1.0]
    assert list(ki[1]) == [0, 1] and list(kv[1]) == [0, 0]      # all-zero token
    assert not pg[4 * 2 * 2:64].any() and not ki[4:].any()     # unused slots are zero


# ------------------------------------------------------- scoring -------
def test_block_size_one_score_is_exact_eq12():
    st = O.Strategy(4, 16, 1, [(0, 32, 0)], 0, 100)
    c, _, _ = _cache(300, st, 30)
    q = np.random.default_rng(5).standard_normal((1, 128))
    per, grp = c.scores(q)
    qr = c.rotate_query(q)
    for b in range(c.n_blocks_mid()):
        lo, hi = c.block_tokens(b)
        assert abs(grp[b] - O.block_max_exact(qr, c.Kt[lo:hi])) < 1e-12


def test_block_score_bounds_every_token_and_head():
    st = O.Strategy(4, 32, 16, [(0, 38, 0)], 0, 100)
    c, _, _ = _cache(1200, st, 31)
    q = np.random.default_rng(6).standard_normal((4, 128))
    per, grp = c.scores(q)
    qr = c.rotate_query(q)
    for b in range(c.n_blocks_mid()):
        lo, hi = c.block_tokens(b)
        exact = (c.Kt[lo:hi].astype(np.float64) @ qr.T) / math.sqrt(128)
        assert np.all(per[:, b] >= exact.max(axis=0) - 1e-12)
        assert grp[b] == per[:, b].max()


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        s = rng.integers(-4, 5, size=n).astype(np.float64)
        cand = np.sort(rng.choice(n, size=int(rng.integers(1, n + 1)), replace=False))
        k = int(rng.integers(0, len(cand) + 1))
        got = O.topk_blocks(s, cand, k)
        want = sorted(sorted(cand.tolist(), key=lambda b: (-s[b], b))[:k])
        assert got.tolist() == want


# ------------------------------------------------------ attention ------
def _hand_attention_case():
    """Two query heads over three tokens, with every value worked out by hand.

    [N] Eq. (1): o = softmax(q k^T / sqrt(d)) V with d = 128.  Head 0 is
    sqrt(128) e_0, so its logits are the tokens' channel-0 entries, chosen as
    0, ln 2, ln 3: the weights are 1/6, 2/6, 3/6.  Head 1 is 2 sqrt(128) e_1
    over channel-1 entries 0, 0, ln 2 / 2: logits 0, 0, ln 2, weights 1/4,
    1/4, 2/4.  V's rows are 6 e_0, 3 e_1 and 2 e_2 + e_3, so
      head 0: o = (1, 1, 1, 1/2, 0, ...)
      head 1: o = (3/2, 3/4, 1, 1/2, 0, ...).
    """
    d = 128
    q = np.zeros((2, d))
    q[0, 0] = math.sqrt(d)
    q[1, 1] = 2 * math.sqrt(d)
    K = np.zeros((3, d))
    K[:, 0] = [0.0, math.log(2), math.log(3)]
    K[:, 1] = [0.0, 0.0, math.log(2) / 2]
    V = np.zeros((3, d))
    V[0, 0], V[1, 1], V[2, 2], V[2, 3] = 6.0, 3.0, 2.0, 1.0
    want = np.zeros((2, d))
    want[0, :4] = [1.0, 1.0, 1.0, 0.5]
    want[1, :4] = [1.5, 0.75, 1.0, 0.5]
    return q, K, V, want


def _sdpa(q, K, V):
    """torch's scaled_dot_product_attention in float64 (default scale 1/sqrt(E), E = q's last dim)."""
    t = lambda x: torch.as_tensor(np.asarray(x, dtype=np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(K), t(V))[0, 0].numpy()


def _softmax_pins_hold(fn):
    """The two pins of softmax_attention, as a predicate (used on planted mistakes too)."""
    q, K, V, want = _hand_attention_case()
    if not np.allclose(fn(q, K, V), want, rtol=0, atol=1e-14):
        return False
    rng = np.random.default_rng(81)
    for G, T in ((1, 1), (4, 7), (8, 300)):
        q = rng.standard_normal((G, 128))
        K = rng.standard_normal((T, 128)) * 3.0
        V = rng.standard_normal((T, 128))
        ref = _sdpa(q, K, V)
        if not np.allclose(fn(q, K, V), ref, rtol=0, atol=1e-12 * np.abs(ref).max()):
            return False
    return True


def test_softmax_attention_hand_case_and_library_routine():
    # [N] Eq. (1)/(13): a hand-computed case with exact weights, and torch's
    # scaled_dot_product_attention in float64 on random inputs.
    assert _softmax_pins_hold(O.softmax_attention)
    assert _softmax_pins_hold(O.dense_attention)
    # No tokens: the output is zero (a state the kernels see with T = 0).
    assert not O.softmax_attention(np.ones((2, 128)), np.zeros((0, 128)), np.zeros((0, 128))).any()


def test_softmax_pins_catch_planted_mistakes():
    def scaled(c):
        def f(q, K, V):
            lg = q @ K.T * c
            p = np.exp(lg - lg.max(axis=1, keepdims=True))
            return (p / p.sum(axis=1, keepdims=True)) @ V
        return f

    def wrong_axis(q, K, V):
        lg = q @ K.T / math.sqrt(128)
        p = np.exp(lg - lg.max(axis=0, keepdims=True))
        return (p / p.sum(axis=0, keepdims=True)) @ V

    def unnormalised(q, K, V):
        lg = q @ K.T / math.sqrt(128)
        return np.exp(lg - lg.max(axis=1, keepdims=True)) @ V

    assert _softmax_pins_hold(scaled(1 / math.sqrt(128)))          # the right form passes
    for bad in (scaled(1 / 128), scaled(1 / math.sqrt(38)), scaled(1.0), wrong_axis, unnormalised):
        assert not _softmax_pins_hold(bad)


def test_densify_hand_case_and_planted_mistake():
    # Zero-filled k~ from (index, value) pairs, d = 4 worked by hand.
    idx = np.array([[0, 2], [1, 3], [0, 1]], dtype=np.uint8)
    vals = np.array([[1.5, -2.0], [3.0, 0.25], [0.0, 7.0]])
    want = np.array([[1.5, 0.0, -2.0, 0.0], [0.0, 3.0, 0.0, 0.25], [0.0, 7.0, 0.0, 0.0]])
    assert np.array_equal(O.densify(idx, vals, 4), want)
    # A densify that ignored the indices (values into the first r channels) fails it.
    wrong = np.zeros((3, 4))
    wrong[:, :2] = vals
    assert not np.array_equal(wrong, want)


def test_compressed_rows_are_brute_force_top_r_of_rotated_rows():
    # At r < d the zero-filled rows the attention reads (Kt, Vt) hold, for each
    # middle token, exactly its r largest-magnitude rotated channels (a Python
    # sort, ties to the lower channel) and zero elsewhere.
    st = O.Strategy(4, 32, 16, [(0, 38, 0), (500, 17, 0)], 0, 100)
    c, _, _ = _cache(900, st, 70)
    for t in range(4, 4 + c.n_mid, 7):
        r = c.r_of_block((t - 4) // 16)
        for rows, dense in ((c.Kr, c.Kt), (c.Vr, c.Vt)):
            x = rows[t].astype(np.float64)
            keep = sorted(sorted(range(128), key=lambda j: (-abs(x[j]), j))[:r])
            z = np.zeros(128)
            z[keep] = x[keep]
            assert np.array_equal(dense[t].astype(np.float64), z)


def test_compressed_attention_by_explicit_sums_over_packed_pairs():
    # [N] Eq. (13)-(14) at r < d, restated with scalar loops over the packed
    # (index, value) pairs of each page (no zero-filled rows), math.exp for the
    # softmax and an explicit un-rotation; the pages' bytes are pinned by hand
    # in test_page_byte_layout.
    st = O.Strategy(4, 24, 16, [(0, 38, 0)], topk_fixed=3)
    c, _, _ = _cache(170, st, 71, G=2)
    q = np.random.default_rng(72).standard_normal((2, 128))
    ids, _ = c.select(q)
    qr = q @ c.Rk.T
    toks = []                                   # (key pairs, value pairs) per attended token
    for p in list(c.sink_positions()) + list(c.window_positions()):
        toks.append((list(enumerate(c.Kr[p].astype(np.float64))), list(enumerate(c.Vr[p].astype(np.float64)))))
    for b in ids:
        lo, hi = c.block_tokens(int(b))
        kv, ki, vv, vi = _page_rows(c.page_bytes(int(b)), 16, 38, hi - lo)
        for t in range(hi - lo):
            toks.append((list(zip(ki[t].tolist(), O.bits_to_value(kv[t]).tolist())),
                         list(zip(vi[t].tolist(), O.bits_to_value(vv[t]).tolist()))))
    got = np.zeros((2, 128))
    for h in range(2):
        logits = [sum(qr[h, j] * x for j, x in kp) / math.sqrt(128) for kp, _ in toks]
        m = max(logits)
        w = [math.exp(l - m) for l in logits]
        acc = [0.0] * 128
        for wi, (_, vp) in zip(w, toks):
            for j, x in vp:
                acc[j] += wi * x
        o = [a / sum(w) for a in acc]
        for j in range(128):
            got[h, j] = sum(o[i] * c.Rv[i, j] for i in range(128))
    want = c.attention(q, ids)
    assert np.allclose(want, got, rtol=0, atol=1e-12 * np.abs(got).max())


def _page_rows(pg, B, r, n):
    Br = B * r
    return (pg[:2 * Br].view(np.uint16).reshape(B, r)[:n], pg[2 * Br:3 * Br].reshape(B, r)[:n],
            pg[3 * Br:5 * Br].view(np.uint16).reshape(B, r)[:n], pg[5 * Br:].reshape(B, r)[:n])


@pytest.mark.parametrize("G", [1, 4])
def test_full_channels_all_blocks_equals_dense_attention(G):
    st = O.Strategy(4, 40, 16, [(0, 128, 0)], topk_fixed=10 ** 6)
    c, K, V = _cache(700, st, 40, round_bf16=False, prefill=650, steps=(1,) * 50)
    q = np.random.default_rng(8).standard_normal((G, 128))
    ids, _ = c.select(q)
    assert len(ids) == c.n_blocks_mid()
    got = c.attention(q, ids)
    want = _sdpa(q, K, V)                       # [N] Eq. (1) by the library routine
    assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())


def test_always_segment_is_attended_without_selection():
    st = O.Strategy(4, 32, 16, [(0, 128, 0), (300, 128, 1), (600, 128, 0)], topk_fixed=1)
    c, K, V = _cache(1000, st, 41, round_bf16=False)
    q = np.random.default_rng(9).standard_normal((1, 128))
    ids, _ = c.select(q)
    assert len(ids) == 1 and len(c.always_blocks()) > 0
    assert not set(ids.tolist()) & set(c.always_blocks().tolist())
    Kt, _ = c.attend_tokens(ids)
    assert Kt.shape[0] == 4 + 32 + 16 * (1 + len(c.always_blocks()))


# ----------------------------------------------- planted mistakes ------
def test_pins_catch_planted_mistakes():
    K = _gen(4096, 0.9, 50)
    R, lam = O.rotation_from_keys(K)
    # (a) rotation with R instead of R^T breaks the eigenvalue-share pin
    Xp = K @ R
    col = np.sum(Xp * Xp, axis=0)
    assert abs(col[:8].sum() / col.sum() - lam[:8].sum() / lam.sum()) > 1e-3
    # (b) un-rotation by R_v^T instead of R_v breaks the dense-attention pin
    st = O.Strategy(4, 40, 16, [(0, 128, 0)], topk_fixed=10 ** 6)
    c, Kd, Vd = _cache(500, st, 51, round_bf16=False)
    q = np.random.default_rng(10).standard_normal((2, 128))
    ids, _ = c.select(q)
    Kt, Vt = c.attend_tokens(ids)
    wrong = O.softmax_attention(c.rotate_query(q), Kt, Vt) @ c.Rv.T
    assert not np.allclose(wrong, O.dense_attention(q, Kd, Vd), atol=1e-6)
    # (c) ties toward the higher channel break the brute-force pin
    x = np.array([1.0, -1.0, 0.5, 1.0])
    order = np.argsort(-np.abs(x[::-1]), kind="stable")[:2]
    wrong_idx = sorted((3 - order).tolist())
    assert wrong_idx != _brute_topr(x, 2)
    # (d) a min/max swap in the bound breaks the upper-bound pin
    st = O.Strategy(4, 32, 16, [(0, 38, 0)], 0, 100)
    c, _, _ = _cache(800, st, 52)
    qr = c.rotate_query(np.random.default_rng(11).standard_normal((1, 128)))
    mn, mx = c.meta()
    wrong_s = np.sum(np.minimum(qr * mn, qr * mx), axis=1) / math.sqrt(128)
    exact = np.array([O.block_max_exact(qr, c.Kt[slice(*c.block_tokens(b))])
                      for b in range(c.n_blocks_mid())])
    assert np.any(wrong_s < exact - 1e-9)


# ------------------------------------------------------ Quest comparator ----
@pytest.mark.parametrize("segments,G,topk", [([(0, 128, 0)], 4, 0), ([(0, 128, 0), (400, 128, 1)], 1, 0),
                                            ([(0, 128, 0)], 8, 5)])
def test_quest_equals_the_method_with_every_channel_and_no_rotation(segments, G, topk):
    # Quest keeps every channel and does not rotate: the method's oracle with
    # r = d and R = I computes the same block keys, scores, ids and output.
    st = O.Strategy(4, 40, 16, segments, topk, 0 if topk else 100)
    K = _gen(1500, 0.9, 90)
    V = _gen(1500, 0.9, 91)
    c = O.OracleCache(st, 1508)
    c.set_rotation(np.eye(128), np.eye(128))
    c.append(K[:1400], V[:1400])
    for t in range(1400, 1500, 20):
        c.append(K[t:t + 20], V[t:t + 20])
    q = O.bf16_round(np.random.default_rng(92).standard_normal((G, 128)))
    ids, out = O.quest_decode(q, K, V, st, T0=1400)
    want_ids, _ = c.select(q)
    assert np.array_equal(ids, want_ids)
    assert np.allclose(out, c.attention(q, want_ids), rtol=0, atol=1e-12)
    # and with every block kept it is dense attention, [N] Eq. (1)
    st_all = O.Strategy(4, 40, 16, [(0, 128, 0)], 10 ** 6)
    _, out_all = O.quest_decode(q, K, V, st_all)
    ref = _sdpa(q, K, V)
    assert np.allclose(out_all, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


# ------------------------------------- segment re-compressed, own rotation ----
def _seg_cache(round_bf16, r_all, seed, topk_fixed=10 ** 6):
    st = O.Strategy(4, 40, 16, [(0, r_all, 0), (500, r_all, 0)], topk_fixed, 0)
    K = _gen(1200, 0.9, seed)
    V = _gen(1200, 0.9, seed + 1)
    Rk, _ = O.rotation_from_keys(K)
    Rv, _ = O.rotation_from_keys(V)
    c = O.OracleCache(st, 1208, round_bf16=round_bf16)
    c.set_rotation(Rk, Rv)
    c.append(K[:1150], V[:1150])
    c.append(K[1150:], V[1150:])
    return c, K, V


def test_own_rotation_segment_full_channels_equals_dense_attention():
    # [S] sec. 5.4 / [N] Fig. 4: segment 0 re-compressed under its own
    # rotation (eigenvectors of its own K^T K, V^T V).  With every channel
    # kept, every block attended and no rounding, attention is still [N]
    # Eq. (1) on the raw cache: each basis's logits use the query in that
    # basis and its values are un-rotated by its own R_v.
    c, K, V = _seg_cache(False, 128, 60)
    lo = 4
    hi = 4 + c.firsts[1] * 16
    Rk_s, _ = O.rotation_from_keys(K[lo:hi])
    Rv_s, _ = O.rotation_from_keys(V[lo:hi])
    assert np.abs(Rk_s - c.Rk).max() > 0.1          # a genuinely different basis
    c.recompress_segment(0, K, V, 128, 0, Rk_s, Rv_s)
    q = np.random.default_rng(61).standard_normal((4, 128))
    ids, _ = c.select(q)
    got = c.attention(q, ids)
    want = _sdpa(q, K, V)
    assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())
    # a planted mistake: the segment's values un-rotated by the head's R_v
    saved = c.seg_rot[0]
    c.seg_rot[0] = (Rk_s, c.Rv)
    assert not np.allclose(c.attention(q, ids), want, atol=1e-6)
    c.seg_rot[0] = saved


def test_own_rotation_segment_scores_and_storage():
    # B = 1: a block's score is q'_s . k~ / sqrt(d) with q' rotated by the
    # block's own basis ([N] Eq. (12)); the stored rows are the top-r of the
    # raw rows rotated once by the segment's rotation and rounded once.
    st = O.Strategy(4, 16, 1, [(0, 32, 0), (500, 32, 0)], 0, 100)
    K = _gen(400, 0.9, 62)
    V = _gen(400, 0.9, 63)
    Rk, _ = O.rotation_from_keys(K)
    Rv, _ = O.rotation_from_keys(V)
    c = O.OracleCache(st, 408)
    c.set_rotation(Rk, Rv)
    c.append(K, V)
    hi = 4 + c.firsts[1]
    Rk_s, _ = O.rotation_from_keys(K[4:hi])
    Rv_s, _ = O.rotation_from_keys(V[4:hi])
    c.recompress_segment(0, K, V, 24, 0, Rk_s, Rv_s)
    q = np.random.default_rng(64).standard_normal((2, 128))
    _, grp = c.scores(q)
    for b in range(c.n_blocks_mid()):
        lo_t, hi_t = c.block_tokens(b)
        Rq = Rk_s if b < c.firsts[1] else Rk
        assert abs(grp[b] - O.block_max_exact(q @ Rq.T, c.Kt[lo_t:hi_t])) < 1e-12
    for t in range(4, hi):
        x = O.bf16_round(K[t] @ Rk_s.T)
        keep = sorted(sorted(range(128), key=lambda j: (-abs(x[j]), j))[:24])
        z = np.zeros(128)
        z[keep] = x[keep]
        assert np.array_equal(c.Kt[t].astype(np.float64), z)
    assert c.r_of_block(0) == 24 and c.r_of_block(c.firsts[1]) == 32


def test_recompress_with_head_rotation_reproduces_the_cache():
    # Re-compressing a segment with the head's own rotation and strategy gives
    # back exactly what the appends built.
    a, K, V = _seg_cache(True, 38, 65, topk_fixed=0)
    b, _, _ = _seg_cache(True, 38, 65, topk_fixed=0)
    b.recompress_segment(0, K, V, 38)
    for name in ("Kr", "Vr", "Kt", "Vt", "kidx", "vidx", "kval", "vval", "mn", "mx"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name


# ----------------------------------------- bitmap format ([S] sec. 5.1) ----
def _brute_groups(x, r, g):
    """Exact-arithmetic brute force: of all sets of r / g groups, the first (in
    lexicographic order of sorted group ids) with the largest kept energy."""
    e = [sum(float(v) * float(v) for v in x[j * g:(j + 1) * g]) for j in range(len(x) // g)]
    best, best_e = None, -1.0
    for S in itertools.combinations(range(len(e)), r // g):
        tot = sum(e[j] for j in S)
        if tot > best_e:
            best, best_e = S, tot
    return [j * g + i for j in best for i in range(g)]


def test_grouped_topr_brute_force_with_ties():
    # Small integers: every energy is exact in fp32, ties are frequent.
    rng = np.random.default_rng(31)
    for _ in range(400):
        g = int(rng.choice([2, 4]))
        n_groups = int(rng.integers(2, 6))
        d = g * n_groups
        r = g * int(rng.integers(1, n_groups + 1))
        x = rng.integers(-3, 4, size=d).astype(np.float64)
        idx, vals = O.topr_groups(x, r, g)
        want = _brute_groups(x, r, g)
        assert list(idx[0]) == want
        assert np.array_equal(vals[0], x[want])


def test_grouped_topr_with_one_nonzero_per_group_is_the_element_top_r():
    # A group holding a single nonzero element has energy x^2, so taking the
    # r / g best groups is the element top-(r / g) of [N] Eq. (9) by |x|.
    rng = np.random.default_rng(32)
    for g in (2, 4, 8):
        for _ in range(50):
            x = np.zeros(128)
            pos = np.arange(0, 128, g) + rng.integers(0, g, size=128 // g)
            x[pos] = O.bf16_round(rng.standard_normal(128 // g))
            r = g * int(rng.integers(1, 128 // g + 1))
            idx, _ = O.topr_groups(x, r, g)
            el, _ = O.topr_select(x, r // g)
            assert list(np.unique(idx[0] // g)) == sorted((el[0] // g).tolist())


def test_grouped_topr_truncation_and_energy_bounds():
    rng = np.random.default_rng(33)
    X = O.bf16_round(rng.standard_normal((40, 128)) * np.exp(-0.03 * np.arange(128)))
    for g, r, keep in ((2, 38, 96), (4, 40, 96), (8, 32, 128)):
        idx, _ = O.topr_groups(X, r, g, keep)
        assert idx.max() < keep
        el, _ = O.topr_select(X, r, keep)
        for i in range(X.shape[0]):
            got = np.sum(X[i, idx[i]] ** 2)
            # whole groups only, so at most the element top-r's energy
            assert got <= np.sum(X[i, el[i]] ** 2) * (1 + 1e-12)
            groups = np.unique(idx[i] // g)
            assert len(groups) == r // g and np.array_equal(np.sort(idx[i]), idx[i])
            e = [np.sum(X[i, j * g:(j + 1) * g] ** 2) for j in range(keep // g)]
            # every kept group's energy is at least every dropped group's
            dropped = [e[j] for j in range(keep // g) if j not in groups]
            assert min(e[j] for j in groups) >= max(dropped) * (1 - 1e-6)


def test_group_energy_is_fp32_in_channel_order():
    # 4096^2 = 2^24: adding 1 in fp32 rounds back to 2^24 (ties to even), so
    # [4096, 1, 1, 0] sums to 2^24 while [1, 1, 4096, 0] sums to 2^24 + 2.
    e = O.group_energy_f32(np.array([[4096.0, 1, 1, 0, 1, 1, 4096, 0]]), 4)
    assert e[0, 0] == 2.0 ** 24 and e[0, 1] == 2.0 ** 24 + 2
    # The decision follows fp32: groups [4096, 1, 0, 0] and [4096, 1, 1, 0]
    # both sum to 2^24, so the lower group wins, where exact sums would take
    # the upper one.
    x = np.array([4096.0, 1, 0, 0, 4096, 1, 1, 0])
    assert list(O.topr_groups(x, 4, 4)[0][0]) == [0, 1, 2, 3]
    assert _brute_groups(x, 4, 4) == [4, 5, 6, 7]


def test_bitmap_bytes_hand_cases_and_round_trip():
    bm = O.bitmap_bytes(np.array([[0, 1, 33, 127]]), 1)
    want = np.zeros(16, dtype=np.uint8)
    want[0], want[4], want[15] = 0x03, 0x02, 0x80
    assert np.array_equal(bm[0], want)
    bm = O.bitmap_bytes(np.array([[0, 1, 2, 3, 124, 125, 126, 127]]), 4)
    assert list(bm[0]) == [0x01, 0, 0, 0x80]
    bm = O.bitmap_bytes(np.array([[8, 9, 10, 11, 12, 13, 14, 15]]), 8)
    assert list(bm[0]) == [0x02, 0]
    rng = np.random.default_rng(34)
    for g in (1, 2, 4, 8):
        X = O.bf16_round(rng.standard_normal((20, 128)))
        idx, _ = O.topr_groups(X, 8 * g, g)
        bm = O.bitmap_bytes(idx, g)
        assert bm.shape == (20, 16 // g)
        bits = np.unpackbits(bm, axis=1, bitorder="little")
        for i in range(20):
            assert np.array_equal(np.flatnonzero(bits[i]), np.unique(idx[i] // g))


def test_bitmap_page_byte_layout():
    # [Kval B*r][K bitmaps B*d/g/8][Vval B*r][V bitmaps]; g = 2, r = 2.
    st = O.Strategy(0, 1, 16, [(0, 2, 0)], bitmap_group=2)
    c = O.OracleCache(st, 64)
    c.set_rotation(np.eye(128), np.eye(128))
    K = np.zeros((5, 128))
    V = np.zeros((5, 128))
    K[0, 6], K[0, 7], K[0, 100] = 1.5, -2.0, 0.25       # group 3 (energy 6.25) beats group 50
    V[0, 126], V[0, 127] = 3.0, -1.0                     # group 63
    c.append(K, V)
    pg = c.page_bytes(0)
    assert pg.size == 16 * (4 * 2 + 2 * 8)
    kv = pg[:64].view(np.uint16).reshape(16, 2)
    kb = pg[64:192].reshape(16, 8)
    vv = pg[192:256].view(np.uint16).reshape(16, 2)
    vb = pg[256:384].reshape(16, 8)
    assert list(O.bits_to_value(kv[0])) == [1.5, -2.0] and list(kb[0]) == [0x08, 0, 0, 0, 0, 0, 0, 0]
    assert list(O.bits_to_value(vv[0])) == [3.0, -1.0] and list(vb[0]) == [0, 0, 0, 0, 0, 0, 0, 0x80]
    assert list(kb[1]) == [1, 0, 0, 0, 0, 0, 0, 0]       # all-zero token: ties keep group 0
    assert not kb[4:].any() and not kv[4:].any()          # unused slots are zero
    assert O.packed_bytes_per_token(38, 1) == 2 * (76 + 16)
    assert O.packed_bytes_per_token(40, 4) == 2 * (80 + 4)


@pytest.mark.parametrize("g,segs", [(1, [(0, 40, 0), (500, 16, 0)]), (4, [(0, 40, 0), (500, 16, 0)]),
                                    (4, [(0, 40, 0, 0, 8), (400, 16, 0, 96, 2), (700, 40, 0, 0, 1)])],
                         ids=["g1", "g4", "per-segment-g"])
def test_bitmap_cache_rows_and_attention_by_explicit_sums(g, segs):
    # The zero-filled rows hold each token's kept groups (each segment with
    # its own group size where it gives one, [S] sec. 4.3); every page
    # decoded by hand from its bytes gives back those rows.
    st = O.Strategy(4, 32, 16, segs, 0, 100, bitmap_group=g)
    c, _, _ = _cache(900, st, 71)
    assert [c.st.segments[i][4] for i in range(len(segs))] == [sg[4] if len(sg) > 4 else g for sg in segs]
    for t in range(4, 4 + c.n_mid, 5):
        b = (t - 4) // 16
        r = c.r_of_block(b)
        g = c.group_of_block(b)
        kp = c.keep_of_block(b)
        for rows, dense in ((c.Kr, c.Kt), (c.Vr, c.Vt)):
            x = rows[t].astype(np.float64)
            if g > 1:   # a Python sort of scalar fp32 energies, ties to the lower group
                e = []
                for j in range(kp // g):
                    acc = np.float32(0.0)
                    for i in range(g):
                        acc = np.float32(acc + np.float32(x[j * g + i]) * np.float32(x[j * g + i]))
                    e.append(acc)
                best = sorted(sorted(range(kp // g), key=lambda j: (-e[j], j))[:r // g])
                keep = [j * g + i for j in best for i in range(g)]
            else:
                keep = sorted(sorted(range(kp), key=lambda j: (-abs(x[j]), j))[:r])
            z = np.zeros(128)
            z[keep] = x[keep]
            assert np.array_equal(dense[t].astype(np.float64), z)
    # decode every page by hand and compare with Kt / Vt
    for b in range(c.n_blocks_mid()):
        r = c.r_of_block(b)
        g = c.group_of_block(b)
        nb = 16 // g
        lo, hi = c.block_tokens(b)
        pg = c.page_bytes(b)
        Br = 16 * r
        parts = [(pg[:2 * Br], pg[2 * Br:2 * Br + 16 * nb], c.Kt),
                 (pg[2 * Br + 16 * nb:4 * Br + 16 * nb], pg[4 * Br + 16 * nb:], c.Vt)]
        for vals_b, bm_b, dense in parts:
            vals = O.bits_to_value(vals_b.view(np.uint16).reshape(16, r))
            bms = bm_b.reshape(16, nb)
            for t in range(hi - lo):
                row = np.zeros(128)
                k = 0
                for byte in range(nb):
                    for bit in range(8):
                        if bms[t, byte] >> bit & 1:
                            j = 8 * byte + bit
                            row[j * g:(j + 1) * g] = vals[t, k:k + g]
                            k += g
                assert k == r
                assert np.array_equal(row, dense[lo + t].astype(np.float64))


# ------------------------------------ per-segment sequence retention ----
def test_per_segment_retention_brute_force_and_k_rule():
    # [S] sec. 4.3: each segment's strategy has its own sequence retention.
    # Each scored segment keeps its own k_s = ceil(rate * n_s / 1000) best
    # blocks (clamped to [1, n_s]), ties to the lower id; always-attended
    # segments are not scored.  Brute force: a Python sort per segment.
    assert O.n_select(37, O.Strategy(4, 32, 16, [(0, 32, 0)], 0, 100), 150) == 6     # ceil(5.55)
    assert O.n_select(5, O.Strategy(4, 32, 16, [(0, 32, 0)], 0, 100), 1) == 1        # at least one
    assert O.n_select(0, O.Strategy(4, 32, 16, [(0, 32, 0)], 0, 100), 500) == 0
    segs = [(0, 32, 0, 0, 0, 300), (300, 64, 1), (550, 32, 0, 0, 0, 50), (800, 24, 0)]
    st = O.Strategy(4, 32, 16, segs, 0, 100)
    assert st.per_segment_retention()
    c, _, _ = _cache(3000, st, 80)
    rng = np.random.default_rng(81)
    for trial in range(5):
        q = rng.standard_normal((4, 128))
        ids, grp = c.select(q)
        want, total = [], 0
        for s, sg in enumerate(c.st.segments):
            if sg[2]:
                continue
            nb = c.n_blocks_mid()
            lo = min(c.firsts[s], nb)
            hi = min(c.firsts[s + 1], nb) if s + 1 < len(segs) else nb
            blocks = list(range(lo, hi))
            rate = sg[5] or 100
            k = min(max(-(-rate * len(blocks) // 1000), 1), len(blocks)) if blocks else 0
            want += sorted(sorted(blocks, key=lambda b: (-grp[b], b))[:k])
            total += k
        assert list(ids) == sorted(want) and c.n_selected() == total == len(ids)
    # a planted mistake: one top-k over all scored blocks with the same total
    # picks another set (the segments' own rates are not kept)
    cand = c.candidates()
    glob = O.topk_blocks(grp, cand, len(ids))
    assert not np.array_equal(glob, ids)


def test_per_segment_retention_equal_rates_is_the_global_rule():
    # One scored segment at the cache's own rate: the same blocks as the
    # single top-k over the candidates.
    st_g = O.Strategy(4, 32, 16, [(0, 32, 0), (500, 64, 1)], 0, 100)
    st_s = O.Strategy(4, 32, 16, [(0, 32, 0, 0, 0, 100), (500, 64, 1)], 0, 100)
    a, _, _ = _cache(2000, st_g, 82)
    b, _, _ = _cache(2000, st_s, 82)
    q = np.random.default_rng(83).standard_normal((4, 128))
    assert np.array_equal(a.select(q)[0], b.select(q)[0])
