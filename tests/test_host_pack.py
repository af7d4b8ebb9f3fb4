"""Host re-compression of complete blocks (the CPU side of the double-buffered
compression) against the oracle's pages, keys and compressed keys.  CPU only."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import mosaickv_oracle as O  # noqa: E402

D = 128


def _lib():
    from compressed_kv_cache_vector_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding


def _signed_perm(seed):
    rng = np.random.default_rng(seed)
    P = np.zeros((D, D))
    P[np.arange(D), rng.permutation(D)] = rng.choice([-1.0, 1.0], size=D)
    return P


def _bf16_data(T, decay, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, D)) * decay ** np.arange(D)
    X[rng.random(X.shape) < 0.02] *= 8.0
    Xb = O.bf16_round(X)
    return Xb, O.bf16_bits(Xb)


@pytest.mark.parametrize("rot,block,r,keep,mc,fmt,g", [
    ("perm", 16, 32, 0, 0, 0, 0), ("identity", 32, 38, 96, 24, 0, 0), ("perm", 64, 20, 0, 48, 0, 0),
    # bitmap pages ([S] sec. 5.1): one bit per channel, or per group of g channels
    ("perm", 16, 38, 0, 0, 2, 1), ("perm", 32, 38, 96, 0, 2, 2), ("identity", 16, 40, 96, 24, 2, 4),
    ("perm", 64, 24, 0, 0, 2, 8)])
def test_host_pack_matches_oracle_bit_exact(rot, block, r, keep, mc, fmt, g):
    b = _lib()
    S, W = 4, 64
    T = S + W + 5 * block + 7                      # five complete middle blocks and a partial one
    K, Kw = _bf16_data(T, 0.92, 1)
    V, Vw = _bf16_data(T, 0.92, 2)
    Rk = np.eye(D) if rot == "identity" else _signed_perm(3)
    Rv = np.eye(D) if rot == "identity" else _signed_perm(4)
    seg = (0, r, 0, keep)
    bg = max(1, g) if fmt == 2 else 0
    oc = O.OracleCache(O.Strategy(S, W, block, [seg], 0, 100, mc, bitmap_group=bg), T)
    oc.set_rotation(Rk, Rv)
    oc.append(K, V)
    n = 5
    pb = 16 // bg if bg else r
    page_stride = block * (4 * r + 2 * pb) + 32     # any stride at least one page
    pages, meta, cmeta = b.host_pack_blocks(Rk, Rv, Kw[S:S + n * block], Vw[S:S + n * block], block, r, keep,
                                            page_stride, mc, fmt, g)
    mn, mx = oc.meta()
    for blk in range(n):
        want = oc.page_bytes(blk)
        assert np.array_equal(pages[blk, :want.size], want), blk
        assert not pages[blk, want.size:].any()
        assert np.array_equal(meta[blk, 0], O.bf16_bits(mn[blk]))
        assert np.array_equal(meta[blk, 1], O.bf16_bits(mx[blk]))
    if mc:
        idx, cmn, cmx = O.compress_key_rows(mn[:n], mx[:n], mc)
        assert np.array_equal(cmeta[:, :2 * mc].copy().view(np.uint16), O.bf16_bits(cmn))
        assert np.array_equal(cmeta[:, 2 * mc:4 * mc].copy().view(np.uint16), O.bf16_bits(cmx))
        assert np.array_equal(cmeta[:, 4 * mc:5 * mc], idx.astype(np.uint8))


def test_host_pack_eigen_rotation_within_an_ulp():
    # With a dense rotation the fp64 sums run in another order than numpy's,
    # so a rounding boundary may flip rarely; values agree to one bf16 ulp.
    b = _lib()
    S, W, block, r = 4, 64, 32, 38
    T = S + W + 4 * block
    K, Kw = _bf16_data(T, 0.92, 5)
    V, Vw = _bf16_data(T, 0.92, 6)
    Rk, _ = O.rotation_from_keys(K)
    Rv, _ = O.rotation_from_keys(V)
    Rk, Rv = Rk.astype(np.float32).astype(np.float64), Rv.astype(np.float32).astype(np.float64)
    oc = O.OracleCache(O.Strategy(S, W, block, [(0, r, 0)], 0, 100), T)
    oc.set_rotation(Rk, Rv)
    oc.append(K, V)
    pages, meta, _ = b.host_pack_blocks(Rk, Rv, Kw[S:S + 4 * block], Vw[S:S + 4 * block], block, r, 0,
                                        6 * block * r, 0)
    same = total = 0
    for blk in range(4):
        want = oc.page_bytes(blk)
        same += int(np.count_nonzero(pages[blk, :want.size] == want))
        total += want.size
    assert same >= total - total // 1000


def test_host_pack_errors():
    b = _lib()
    k = np.zeros((16, D), dtype=np.uint16)
    R = np.eye(D)
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 24, 8, 0, 6 * 24 * 8)          # block must be 16, 32 or 64
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 4, 6 * 16 * 8)          # keep below r
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 0, 6 * 16 * 8 - 1)      # page too small
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 0, 6 * 16 * 8, 0, 0, 4)  # a group size needs bitmap pages
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 0, 6 * 16 * 8, 0, 2, 3)  # group sizes are 1, 2, 4, 8
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 6, 0, 6 * 16 * 8, 0, 2, 4)  # r a multiple of the group
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 12, 6 * 16 * 8, 0, 2, 8)  # keep a multiple of the group
    with pytest.raises(b.MosaicKVError):
        b.host_pack_blocks(R, R, k, k, 16, 8, 0, 16 * (4 * 8 + 2 * 16) - 1, 0, 2, 1)  # bitmap page too small


@pytest.mark.parametrize("seed", list(range(2000, 2012)))
def test_host_pack_random_formats_bit_exact(seed):
    # Random block size, r, truncation, page format and group size; exact
    # rotations (signed permutations), so the host's pages, block keys and
    # compressed keys equal the oracle's byte for byte.
    b = _lib()
    rng = np.random.default_rng(seed)
    block = int(rng.choice([16, 32, 64]))
    fmt = int(rng.choice([0, 2]))
    g = int(rng.choice([1, 2, 4, 8])) if fmt == 2 else 0
    gg = max(1, g)
    r = gg * int(rng.integers(max(1, 4 // gg), 96 // gg + 1))
    keep = int(rng.choice([0, 96])) if r <= 96 else 0
    mc = int(rng.choice([0, 16]))
    S, W, n = 4, 32, int(rng.integers(1, 5))
    T = S + W + n * block + 3
    K, Kw = _bf16_data(T, 0.9, seed)
    V, Vw = _bf16_data(T, 0.9, seed + 1)
    Rk, Rv = _signed_perm(seed + 2), _signed_perm(seed + 3)
    oc = O.OracleCache(O.Strategy(S, W, block, [(0, r, 0, keep)], 0, 100, mc, bitmap_group=g if fmt == 2 else 0), T)
    oc.set_rotation(Rk, Rv)
    oc.append(K, V)
    pb = 16 // gg if fmt == 2 else r
    page_stride = block * (4 * r + 2 * pb) + 16 * int(rng.integers(0, 3))
    pages, meta, cmeta = b.host_pack_blocks(Rk, Rv, Kw[S:S + n * block], Vw[S:S + n * block], block, r, keep,
                                            page_stride, mc, fmt, g)
    mn, mx = oc.meta()
    for blk in range(n):
        want = oc.page_bytes(blk)
        assert np.array_equal(pages[blk, :want.size], want), (seed, blk)
        assert np.array_equal(meta[blk, 0], O.bf16_bits(mn[blk]))
        assert np.array_equal(meta[blk, 1], O.bf16_bits(mx[blk]))
    if mc:
        idx, cmn, cmx = O.compress_key_rows(mn[:n], mx[:n], mc)
        assert np.array_equal(cmeta[:, 4 * mc:5 * mc], idx.astype(np.uint8))
