"""fp64 oracle for the MosaicKV decode-time hot path.  TEST INFRASTRUCTURE.

This module is test infrastructure, not the product.  Only the test suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import it.  The CUDA library and its Python binding never do, and this
module imports nothing from them: the two sides share only the seeded input
generators, which hold none of the method's arithmetic.

It restates the method step by step, in float64, with library primitives
(matmul, eigh, stable argsort) as the only building blocks.  bf16-exact data
(inputs, rotated vectors) are kept as float32 to save memory; every
arithmetic step upcasts to float64.

Sources (cited by page title and equation/section):
  [N] "MosaicKV：面向超长上下文LLM服务的动态二维KV缓存压缩——阅读笔记"
      (reading notes on zhongzhuzhou.org): Eq. (1), (4)-(9), (12)-(16),
      Algorithm 1, the d=4 worked example of the SVD section.
  [S] "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV Cache
      Compression" (paperlayer.ai summary of arXiv 2607.00760v1):
      sec. 4.2-4.3 (two-stage compression, per-segment strategy),
      sec. 5.1 (packed format), sec. 5.2 (encoding variants), sec. 5.3
      (PackedAttention), sec. 6.3.

Readings where the pages are silent:
  * segments: sinks [0, S), recent window [T-W, T), middle [S, T-W) cut into
    blocks of B tokens from S; the last block may be partial;
  * per-vector top-r: magnitude descending, ties to the lower channel; the
    kept channels are stored in ascending channel order as bf16 values plus
    uint8 indices; a stored zero is +0;
  * block metadata: per-channel min and max over the block of the
    zero-filled compressed key (Quest-style bound on Eq. (12));
  * GQA: a kv head's block score is the max over its query heads;
  * top-k: k largest scores, ties to the lower block id, ids ascending;
    k = min(topk_fixed, n) or ceil(retain * n / 1000) clamped to [1, n];
  * strategy segments start at the first block boundary at or after
    begin_permille/1000 of the prefill length; the last one is open-ended;
  * decode append: the new token enters the window; the window's oldest
    token, once more than W are held, moves into the middle;
  * sec. 5.1 bitmap (off by default): the indices are replaced by a bitmap
    of d / g bits per vector, one bit per group of g adjacent channels; for
    g > 1 the vector keeps the r / g groups of largest energy (fp32, summed
    in channel order), ties to the lower group; g may differ per segment
    (sec. 4.3), and a re-compressed segment keeps its g;
  * sec. 5.2 variants (off by default): "bottom channels truncated" = the
    per-vector top-r picks among the first keep_channels rotated channels
    only; "per-block keys channel-compressed" = each block keeps the m
    channels with the largest max(|min|, |max|), ties to the lower channel,
    and the scores use them with the other channels zero.

Parity status: every public function is pinned by tests/test_oracle_pins.py
(worked example, brute force, closed forms, library routines, invariants).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

D_HEAD = 128


# --------------------------------------------------------------------------
# bf16 rounding (storage precision of K, V and the rotated vectors)
# --------------------------------------------------------------------------
def bf16_round(x):
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits and float32's exponent range, so for
    2**(e-1) <= |x| < 2**e the spacing is 2**(e-8); below the smallest normal
    (2**-126) the spacing stays 2**-133.  Zero is returned as +0.
    """
    x = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(x)), "NaN/Inf inputs are outside the contract"
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    ulp = np.ldexp(1.0, e - 8)
    y = np.round(x / ulp) * ulp
    return y + 0.0


def bf16_bits(y):
    """uint16 bit pattern of bf16-exact float64 values."""
    y = np.asarray(y, dtype=np.float64)
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bits_to_value(b):
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Rotation: [N] Eq. (4), (6)-(8); un-rotation Eq. (14)
# --------------------------------------------------------------------------
def rotation_from_keys(X):
    """R = V^T from the eigendecomposition X^T X = V diag(lambda) V^T.

    Eigenvalues are sorted descending, so row i of R is the i-th principal
    direction.  Returns (R, eigenvalues).
    """
    X = np.asarray(X, dtype=np.float64)
    lam, vecs = np.linalg.eigh(X.T @ X)
    order = np.argsort(-lam, kind="stable")
    return vecs[:, order].T.copy(), lam[order]


def rotate(X, R, round_bf16=True):
    """X' = X R^T ([N] Eq. (7)/(8)); rounded once, fp64 -> bf16, if asked."""
    Y = np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64).T
    return bf16_round(Y) if round_bf16 else Y


def energy(R, X, r):
    """Energy(r) of [N] Eq. (5), measured on the rotated columns of X."""
    Xp = rotate(X, R, round_bf16=False)
    col = np.sum(Xp * Xp, axis=0)
    return col[:r].sum() / col.sum()


# --------------------------------------------------------------------------
# Channel selection: [N] Eq. (9) / Algorithm 1 and the global-mask contrast
# --------------------------------------------------------------------------
def topr_select(X, r, keep=None):
    """Per-vector top-r by magnitude ([N] Eq. (9), Algorithm 1).

    X: [n, d] bf16-exact values.  Order channels by |x| descending, ties to
    the lower channel (a stable sort keeps channel order among equals), keep
    the first r, and return them in ascending channel order.  With `keep`,
    only the first `keep` channels are candidates: the bottom ones are
    truncated ([S] sec. 5.2).
    Returns (idx uint8 [n, r], vals float64 [n, r]).
    """
    X = np.asarray(X, dtype=np.float64)
    if X.ndim == 1:
        X = X[None, :]
    keep = X.shape[1] if keep is None else keep
    assert r <= keep
    order = np.argsort(-np.abs(X[:, :keep]), axis=1, kind="stable")[:, :r]
    idx = np.sort(order, axis=1)
    vals = np.take_along_axis(X, idx, axis=1)
    return idx.astype(np.uint8), vals


def group_energy_f32(X, g):
    """Energy of each group of g adjacent channels, sum_c x_c^2 over the group,
    accumulated from the group's first channel to its last with every product
    and every sum rounded to fp32: the precision the kernels decide the grouped
    selection in (the bf16 inputs make each square exact in fp32).
    X: [n, d]; returns float32 [n, d // g]."""
    X32 = np.asarray(X, dtype=np.float32)
    n, d = X32.shape
    Xg = X32.reshape(n, d // g, g)
    e = (Xg[:, :, 0] * Xg[:, :, 0]).astype(np.float32)
    for i in range(1, g):
        e = (e + (Xg[:, :, i] * Xg[:, :, i]).astype(np.float32)).astype(np.float32)
    return e


def topr_groups(X, r, g, keep=None):
    """Per-vector top-r in groups of g adjacent channels ([S] sec. 5.1: a
    variable-granularity bitmap has one bit per group of adjacent elements,
    so the vector keeps whole groups; [S] sec. 4.3 lists the element-group
    size in each segment's strategy).

    g = 1 is the per-element top-r of [N] Eq. (9) (topr_select).  For g > 1
    the r / g groups with the largest energy are kept (the grouped form of the
    energy the top-r retains, [N] Eq. (5)), ties to the lower group; with
    `keep` (a multiple of g) only the first keep / g groups are candidates.
    Returns (idx uint8 [n, r], vals float64 [n, r]) in ascending channel order,
    as topr_select does.
    """
    X = np.asarray(X, dtype=np.float64)
    if X.ndim == 1:
        X = X[None, :]
    if g == 1:
        return topr_select(X, r, keep)
    d = X.shape[1]
    keep = d if keep is None else keep
    assert r % g == 0 and keep % g == 0 and r <= keep
    e = group_energy_f32(X, g)[:, :keep // g]
    groups = np.sort(np.argsort(-e, axis=1, kind="stable")[:, :r // g], axis=1)
    idx = (groups[:, :, None] * g + np.arange(g)[None, None, :]).reshape(X.shape[0], r)
    vals = np.take_along_axis(X, idx, axis=1)
    return idx.astype(np.uint8), vals


def bitmap_bytes(idx, g, d=D_HEAD):
    """Position bitmap of [S] sec. 5.1 for kept channels idx [n, r]: d / g bits
    per vector, bit j set when group j (channels g j .. g j + g - 1) is kept;
    bit j lives in byte j // 8 at bit j % 8.  Returns uint8 [n, d // g // 8]."""
    idx = np.asarray(idx, dtype=np.int64)
    bits = np.zeros((idx.shape[0], d // g), dtype=np.uint8)
    np.put_along_axis(bits, idx // g, 1, axis=1)
    return np.packbits(bits, axis=1, bitorder="little")


def global_mask_energy(Xp, r):
    """ThinK-style shared mask by channel energy sum_i x_ij^2 (contrast only)."""
    e = np.sum(np.asarray(Xp, dtype=np.float64) ** 2, axis=0)
    return np.sort(np.argsort(-e, kind="stable")[:r])


def global_mask_variance(Xp, r):
    """ThinK-style shared mask argtopk(var(K', axis 0), r) ([N] ThinK formula)."""
    v = np.var(np.asarray(Xp, dtype=np.float64), axis=0)
    return np.sort(np.argsort(-v, kind="stable")[:r])


def densify(idx, vals, d=D_HEAD):
    """Zero-filled dense vectors k~ from (idx, vals) pairs."""
    idx = np.asarray(idx, dtype=np.int64)
    out = np.zeros((idx.shape[0], d), dtype=np.float64)
    np.put_along_axis(out, idx, np.asarray(vals, dtype=np.float64), axis=1)
    return out


# --------------------------------------------------------------------------
# Segments and strategy ([S] sec. 4.3)
# --------------------------------------------------------------------------
@dataclass
class Strategy:
    n_sink: int
    window: int
    block: int
    segments: list            # [(begin_permille, r, always[, keep_channels[, elem_group[, retain_permille]]])]
    topk_fixed: int = 0
    retain_permille: int = 0
    meta_channels: int = 0    # > 0: channel-compressed per-block keys ([S] sec. 5.2)
    bitmap_group: int = 0     # 0: uint8 channel indices; g >= 1: the D-bit (g = 1) or
                              # grouped (one bit per g channels) bitmap of [S] sec. 5.1

    def __post_init__(self):
        # keep_channels: the first channels eligible for the top-r; 0 or
        # absent means all of them ([S] sec. 5.2 truncates the bottom 25%).
        # elem_group (bitmap pages only): the segment's own element-group
        # size ([S] sec. 4.3 lists it in each segment's strategy); 0 or
        # absent means the cache's bitmap_group.
        # retain_permille: the segment's own sequence retention ([S] sec. 4.3:
        # each segment's strategy has one); 0 or absent means the cache's.
        self.segments = [(sg[0], sg[1], sg[2], (sg[3] if len(sg) > 3 and sg[3] else D_HEAD),
                          (sg[4] if len(sg) > 4 and sg[4] else self.bitmap_group) if self.bitmap_group else 0,
                          sg[5] if len(sg) > 5 else 0)
                         for sg in self.segments]

    def per_segment_retention(self):
        """True when some scored segment gives its own retention: then every
        scored segment keeps its own k (its own rate, else the cache's)."""
        return any(sg[5] for sg in self.segments if not sg[2])


def compress_key_rows(mn, mx, m):
    """Channel-compressed per-block keys ([S] sec. 5.2: prefill encoding
    channel-compresses the per-block keys as it does the vectors): in each
    block keep the m channels with the largest bound magnitude
    max(|min|, |max|), ties to the lower channel, in ascending channel order.
    Returns (idx [nb, m], min values, max values)."""
    mn = np.asarray(mn, dtype=np.float64)
    mx = np.asarray(mx, dtype=np.float64)
    w = np.maximum(np.abs(mn), np.abs(mx))
    idx = np.sort(np.argsort(-w, axis=1, kind="stable")[:, :m], axis=1)
    return idx, np.take_along_axis(mn, idx, axis=1), np.take_along_axis(mx, idx, axis=1)


def zero_filled_keys(idx, cmn, cmx, d=D_HEAD):
    """Dense min/max rows of compressed keys: the dropped channels are zero."""
    return densify(idx, cmn, d), densify(idx, cmx, d)


def n_middle_blocks(T, st: Strategy):
    mid = max(0, T - st.window - st.n_sink)
    return (mid + st.block - 1) // st.block


def segment_first_blocks(T0, st: Strategy):
    """First middle block of each strategy segment, fixed at prefill length T0."""
    nb0 = n_middle_blocks(T0, st)
    firsts = []
    prev = 0
    for i, sg in enumerate(st.segments):
        begin = sg[0]
        if i == 0:
            b = 0
        else:
            pos = (begin * T0) // 1000
            b = (max(0, pos - st.n_sink) + st.block - 1) // st.block
            b = min(max(b, prev), nb0)
        firsts.append(b)
        prev = b
    return firsts


def block_segment(b, firsts):
    s = 0
    for i, f in enumerate(firsts):
        if b >= f:
            s = i
    return s


def n_select(n_scored, st: Strategy, retain_permille=None):
    """Number of blocks top-k keeps among n_scored candidates (with a given
    retention, that rate instead of the strategy's rule)."""
    if n_scored <= 0:
        return 0
    if retain_permille is None and st.topk_fixed > 0:
        return min(st.topk_fixed, n_scored)
    ret = st.retain_permille if retain_permille is None else retain_permille
    k = (ret * n_scored + 999) // 1000
    return min(max(k, 1), n_scored)


# --------------------------------------------------------------------------
# Block scoring and top-k ([N] Eq. (12); Quest min/max bound; [S] sec. 4.2)
# --------------------------------------------------------------------------
def block_scores(qr, mn, mx):
    """Quest-style bound per block: (1/sqrt(d)) sum_j max(q'_j mn_j, q'_j mx_j).

    qr: [G, d] rotated queries of one kv head's group; mn, mx: [nblk, d].
    Returns (per_head [G, nblk], group max [nblk]).
    """
    qr = np.asarray(qr, dtype=np.float64)
    mn = np.asarray(mn, dtype=np.float64)
    mx = np.asarray(mx, dtype=np.float64)
    d = qr.shape[1]
    per = np.empty((qr.shape[0], mn.shape[0]))
    for h in range(qr.shape[0]):
        per[h] = np.sum(np.maximum(qr[h][None, :] * mn, qr[h][None, :] * mx), axis=1) / math.sqrt(d)
    return per, per.max(axis=0)


def block_max_exact(qr, Kt_block):
    """[N] Eq. (12) taken literally: (1/sqrt(d)) max_i q' . k~_i over a block."""
    qr = np.asarray(qr, dtype=np.float64)
    return np.max(np.asarray(Kt_block, dtype=np.float64) @ qr.T, axis=0).max() / math.sqrt(qr.shape[1])


def topk_blocks(scores, candidates, k):
    """k highest scores among candidate block ids; ties to the lower id; ascending ids."""
    cand = np.asarray(candidates, dtype=np.int64)
    if k <= 0 or cand.size == 0:
        return np.zeros(0, dtype=np.int64)
    s = np.asarray(scores, dtype=np.float64)[cand]
    order = np.lexsort((cand, -s))
    return np.sort(cand[order[:k]])


# --------------------------------------------------------------------------
# Attention ([N] Eq. (1), (13), (14))
# --------------------------------------------------------------------------
def softmax_attention(qr, Kt, Vt):
    """o = softmax(q' K^T / sqrt(d)) V for each row of qr, exact in fp64."""
    qr = np.asarray(qr, dtype=np.float64)
    if Kt.shape[0] == 0:
        return np.zeros((qr.shape[0], qr.shape[1]))
    logits = qr @ np.asarray(Kt, dtype=np.float64).T / math.sqrt(qr.shape[1])
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return p @ np.asarray(Vt, dtype=np.float64)


def dense_attention(q, K, V):
    """[N] Eq. (1) on the unrotated, uncompressed cache."""
    return softmax_attention(q, np.asarray(K, dtype=np.float64), np.asarray(V, dtype=np.float64))


# --------------------------------------------------------------------------
# The compressed cache of one (layer, sequence, kv head)
# --------------------------------------------------------------------------
class OracleCache:
    """Sinks and window as dense rotated bf16; middle as per-vector top-r.

    Built by appending tokens ([N] the decode-time rotation of each new
    k/v; [S] sec. 4.2 stage 1, sec. 5.3 update buffer read as the window).
    """

    def __init__(self, st: Strategy, capacity: int, d: int = D_HEAD, round_bf16: bool = True):
        self.st = st
        self.d = d
        self.cap = capacity
        self.round = round_bf16
        dt = np.float32 if round_bf16 else np.float64
        self.Kr = np.zeros((capacity, d), dtype=dt)     # rotated tokens
        self.Vr = np.zeros((capacity, d), dtype=dt)
        self.Kt = np.zeros((capacity, d), dtype=dt)     # zero-filled compressed (middle rows)
        self.Vt = np.zeros((capacity, d), dtype=dt)
        rmax = max(sg[1] for sg in st.segments)
        self.kidx = np.zeros((capacity, rmax), dtype=np.uint8)
        self.vidx = np.zeros((capacity, rmax), dtype=np.uint8)
        self.kval = np.zeros((capacity, rmax), dtype=dt)
        self.vval = np.zeros((capacity, rmax), dtype=dt)
        self.rtok = np.zeros(capacity, dtype=np.int64)
        nb = n_middle_blocks(capacity, st) + 1
        self.mn = np.zeros((nb, d), dtype=dt)
        self.mx = np.zeros((nb, d), dtype=dt)
        self.T = 0
        self.T0 = None
        self.firsts = None
        self.n_mid = 0
        self.Rk = None
        self.Rv = None
        self.seg_rot = {}   # segment -> (R_k, R_v) of a segment re-compressed under its own rotation

    def set_rotation(self, Rk, Rv):
        self.Rk = np.asarray(Rk, dtype=np.float64)
        self.Rv = np.asarray(Rv, dtype=np.float64)

    # --- strategy helpers -------------------------------------------------
    def r_of_block(self, b):
        return self.st.segments[block_segment(b, self.firsts)][1]

    def always_of_block(self, b):
        return bool(self.st.segments[block_segment(b, self.firsts)][2])

    def keep_of_block(self, b):
        return self.st.segments[block_segment(b, self.firsts)][3]

    def group_of_block(self, b):
        """The block's element-group size (bitmap pages), 0 for uint8 indices."""
        return self.st.segments[block_segment(b, self.firsts)][4]

    def rotations_of_block(self, b):
        """(R_k, R_v) the block's tokens are stored in: the segment's own after a
        re-compression under its own rotation ([S] sec. 5.4), else the head's."""
        return self.seg_rot.get(block_segment(b, self.firsts), (self.Rk, self.Rv))

    def n_blocks(self):
        return n_middle_blocks(self.T, self.st)

    def block_tokens(self, b):
        S, B = self.st.n_sink, self.st.block
        lo = S + b * B
        hi = min(lo + B, S + self.n_mid)
        return lo, hi

    # --- append -----------------------------------------------------------
    def append(self, K_new, V_new):
        K_new = np.asarray(K_new, dtype=np.float64)
        V_new = np.asarray(V_new, dtype=np.float64)
        n = K_new.shape[0]
        assert self.Rk is not None, "rotation must be set before append"
        assert self.T + n <= self.cap, "capacity exceeded"
        if self.T == 0:
            self.T0 = n
            self.firsts = segment_first_blocks(n, self.st)
        t0 = self.T
        self.Kr[t0:t0 + n] = rotate(K_new, self.Rk, self.round)
        self.Vr[t0:t0 + n] = rotate(V_new, self.Rv, self.round)
        self.T += n
        S, W, B = self.st.n_sink, self.st.window, self.st.block
        target = max(0, self.T - W - S)
        if target > self.n_mid:
            lo, hi = S + self.n_mid, S + target
            self._compress(lo, hi)
            self.n_mid = target
            # Block min/max over the zero-filled compressed keys, recomputed
            # from the definition for every block that gained a token.
            for b in range((lo - S) // B, (hi - 1 - S) // B + 1):
                blo, bhi = self.block_tokens(b)
                blk = self.Kt[blo:bhi].astype(np.float64)
                self.mn[b] = blk.min(axis=0) + 0.0
                self.mx[b] = blk.max(axis=0) + 0.0

    def _compress(self, lo, hi):
        S, B = self.st.n_sink, self.st.block
        pos = np.arange(lo, hi)
        blocks = (pos - S) // B
        for b in np.unique(blocks):
            sel = pos[blocks == b]
            r, keep = self.r_of_block(int(b)), self.keep_of_block(int(b))
            g = max(1, self.group_of_block(int(b)))
            for src, dst_idx, dst_val, dense in ((self.Kr, self.kidx, self.kval, self.Kt),
                                                (self.Vr, self.vidx, self.vval, self.Vt)):
                idx, vals = topr_groups(src[sel].astype(np.float64), r, g, keep)
                dst_idx[sel, :r] = idx
                dst_idx[sel, r:] = 0
                dst_val[sel, :r] = vals
                dst_val[sel, r:] = 0
                dense[sel] = densify(idx, vals, self.d)
            self.rtok[sel] = r

    def n_blocks_mid(self):
        return (self.n_mid + self.st.block - 1) // self.st.block

    # --- re-compression of a closed segment ([S] sec. 5.4) ---------------
    def recompress_segment(self, seg, K_raw, V_raw, r, keep=0, Rk=None, Rv=None):
        """[S] sec. 5.4: the CPU re-compresses a closed segment (not the last,
        open one) with a new strategy and, from the per-segment SVD of [N]
        Fig. 4, possibly its own rotation (rows = eigenvectors of the
        segment's own K^T K and V^T V by descending eigenvalue); the result
        replaces the segment.  K_raw, V_raw: the sequence's unrotated rows
        (float64, at least up to the segment's end).  Its tokens are rotated
        once more and rounded once, compressed to the new r (truncation keep,
        0 = all channels), and its blocks' min/max recomputed."""
        assert 0 <= seg < len(self.st.segments) - 1, "only a closed segment is re-compressed"
        segs = list(self.st.segments)
        begin, _, always, _, g, ret = segs[seg]     # the segment keeps its group size and retention
        segs[seg] = (begin, r, always, keep if keep else self.d, g, ret)
        self.st = Strategy(self.st.n_sink, self.st.window, self.st.block, segs, self.st.topk_fixed,
                           self.st.retain_permille, self.st.meta_channels, self.st.bitmap_group)
        if Rk is not None:
            self.seg_rot[seg] = (np.asarray(Rk, dtype=np.float64), np.asarray(Rv, dtype=np.float64))
        Rk_s, Rv_s = self.seg_rot.get(seg, (self.Rk, self.Rv))
        S, B = self.st.n_sink, self.st.block
        lo = S + self.firsts[seg] * B
        hi = S + self.firsts[seg + 1] * B
        if hi <= lo:
            return
        self.Kr[lo:hi] = rotate(np.asarray(K_raw, dtype=np.float64)[lo:hi], Rk_s, self.round)
        self.Vr[lo:hi] = rotate(np.asarray(V_raw, dtype=np.float64)[lo:hi], Rv_s, self.round)
        self._compress(lo, hi)
        for b in range(self.firsts[seg], self.firsts[seg + 1]):
            blo, bhi = self.block_tokens(b)
            blk = self.Kt[blo:bhi].astype(np.float64)
            self.mn[b] = blk.min(axis=0) + 0.0
            self.mx[b] = blk.max(axis=0) + 0.0

    # --- views used by the tests ------------------------------------------
    def sink_positions(self):
        return np.arange(min(self.st.n_sink, self.T))

    def window_positions(self):
        return np.arange(self.st.n_sink + self.n_mid, self.T)

    def ring_slot(self, p):
        return (p - self.st.n_sink) % self.st.window

    def meta(self):
        nb = self.n_blocks_mid()
        return self.mn[:nb].astype(np.float64), self.mx[:nb].astype(np.float64)

    def page_bytes(self, b):
        """The packed page of block b: [Kval B*r bf16][Kpos][Vval B*r bf16][Vpos].

        Pos is B*r uint8 channel indices (the build's default contract), or
        with bitmap_group g the B bitmaps of d / g bits ([S] sec. 5.1).
        Slots past the last live token are zero ([S] sec. 5.1 contiguous
        packing).
        """
        B = self.st.block
        r = self.r_of_block(b)
        g = self.group_of_block(b)
        lo, hi = self.block_tokens(b)
        n = hi - lo
        kv = np.zeros((B, r), dtype=np.uint16)
        vv = np.zeros((B, r), dtype=np.uint16)
        kv[:n] = bf16_bits(self.kval[lo:hi, :r])
        vv[:n] = bf16_bits(self.vval[lo:hi, :r])
        if g:
            ki = np.zeros((B, self.d // g // 8), dtype=np.uint8)
            vi = np.zeros_like(ki)
            ki[:n] = bitmap_bytes(self.kidx[lo:hi, :r], g, self.d)
            vi[:n] = bitmap_bytes(self.vidx[lo:hi, :r], g, self.d)
        else:
            ki = np.zeros((B, r), dtype=np.uint8)
            vi = np.zeros((B, r), dtype=np.uint8)
            ki[:n] = self.kidx[lo:hi, :r]
            vi[:n] = self.vidx[lo:hi, :r]
        return np.concatenate([kv.reshape(-1).view(np.uint8), ki.reshape(-1),
                               vv.reshape(-1).view(np.uint8), vi.reshape(-1)])

    # --- decode-time select and attention ---------------------------------
    def rotate_query(self, q):
        """q' = q R_k^T, the query side of the rotation ([S] sec. 5.3)."""
        return np.asarray(q, dtype=np.float64) @ self.Rk.T

    def candidates(self):
        nb = self.n_blocks_mid()
        return np.array([b for b in range(nb) if not self.always_of_block(b)], dtype=np.int64)

    def always_blocks(self):
        nb = self.n_blocks_mid()
        return np.array([b for b in range(nb) if self.always_of_block(b)], dtype=np.int64)

    def score_keys(self):
        """The per-block keys the scores use: the min/max rows, or with
        channel-compressed keys their zero-filled dense form."""
        mn, mx = self.meta()
        if self.st.meta_channels:
            mn, mx = zero_filled_keys(*compress_key_rows(mn, mx, self.st.meta_channels), self.d)
        return mn, mx

    def scores(self, q):
        """Group scores over every middle block (always-blocks included).  A
        block stored under its segment's own rotation is scored with the query
        rotated by that rotation."""
        mn, mx = self.score_keys()
        per, grp = block_scores(self.rotate_query(q), mn, mx)
        for seg, (Rk_s, _) in self.seg_rot.items():
            lo, hi = self.firsts[seg], min(self.firsts[seg + 1], self.n_blocks_mid())
            if hi > lo:
                p_s, _ = block_scores(np.asarray(q, dtype=np.float64) @ Rk_s.T, mn[lo:hi], mx[lo:hi])
                per[:, lo:hi] = p_s
        return per, per.max(axis=0)

    def segment_candidates(self, seg):
        """The middle blocks of a scored segment (empty for an always-attended one)."""
        if self.st.segments[seg][2]:
            return np.zeros(0, dtype=np.int64)
        nb = self.n_blocks_mid()
        lo = min(self.firsts[seg], nb)
        hi = min(self.firsts[seg + 1], nb) if seg + 1 < len(self.st.segments) else nb
        return np.arange(lo, max(lo, hi), dtype=np.int64)

    def n_selected(self):
        """How many blocks the selection keeps."""
        if not self.st.per_segment_retention():
            return n_select(len(self.candidates()), self.st)
        return sum(n_select(len(self.segment_candidates(s)), self.st, sg[5] or self.st.retain_permille)
                   for s, sg in enumerate(self.st.segments) if not sg[2])

    def select(self, q):
        """The blocks attended besides the always-attended ones: the k best
        scored blocks; with per-segment retention, each scored segment's own
        k best (each segment its own top-k, [S] sec. 4.3), ids ascending."""
        _, grp = self.scores(q)
        if not self.st.per_segment_retention():
            cand = self.candidates()
            return topk_blocks(grp, cand, n_select(len(cand), self.st)), grp
        ids = []
        for s, sg in enumerate(self.st.segments):
            cand = self.segment_candidates(s)
            if len(cand):
                ids.append(topk_blocks(grp, cand, n_select(len(cand), self.st, sg[5] or self.st.retain_permille)))
        return (np.sort(np.concatenate(ids)) if ids else np.zeros(0, dtype=np.int64)), grp

    def attend_tokens(self, ids):
        """Token rows (rotated K, rotated V) that attention reads for these blocks."""
        rows_k = [self.Kr[self.sink_positions()], self.Kr[self.window_positions()]]
        rows_v = [self.Vr[self.sink_positions()], self.Vr[self.window_positions()]]
        blocks = np.concatenate([np.asarray(ids, dtype=np.int64), self.always_blocks()])
        for b in blocks:
            lo, hi = self.block_tokens(int(b))
            rows_k.append(self.Kt[lo:hi])
            rows_v.append(self.Vt[lo:hi])
        return (np.concatenate(rows_k).astype(np.float64),
                np.concatenate(rows_v).astype(np.float64))

    def attention(self, q, ids):
        """[N] Eq. (13) on the kept tokens, then Eq. (14) output = o R_v."""
        if not self.seg_rot:
            Kt, Vt = self.attend_tokens(ids)
            o = softmax_attention(self.rotate_query(q), Kt, Vt)
            return o @ self.Rv
        # Segments under their own rotation: each token's logit uses the query
        # rotated into its basis, and each basis's weighted values are
        # un-rotated by its own R_v; one softmax over all tokens.
        q = np.asarray(q, dtype=np.float64)
        groups = {}   # basis -> (rows of K~, rows of V~)
        head = (id(self.Rk), id(self.Rv))
        def add(key, k_rows, v_rows):
            kk, vv = groups.setdefault(key, ([], []))
            kk.append(k_rows)
            vv.append(v_rows)
        add(head, self.Kr[self.sink_positions()], self.Vr[self.sink_positions()])
        add(head, self.Kr[self.window_positions()], self.Vr[self.window_positions()])
        rot = {head: (self.Rk, self.Rv)}
        for b in np.concatenate([np.asarray(ids, dtype=np.int64), self.always_blocks()]):
            Rk_b, Rv_b = self.rotations_of_block(int(b))
            key = (id(Rk_b), id(Rv_b))
            rot[key] = (Rk_b, Rv_b)
            lo, hi = self.block_tokens(int(b))
            add(key, self.Kt[lo:hi], self.Vt[lo:hi])
        logits, values = [], []
        for key, (kk, vv) in groups.items():
            Rk_b, Rv_b = rot[key]
            Kb = np.concatenate(kk).astype(np.float64)
            logits.append((q @ Rk_b.T) @ Kb.T / math.sqrt(self.d))
            values.append((np.concatenate(vv).astype(np.float64), Rv_b))
        lg = np.concatenate(logits, axis=1)
        p = np.exp(lg - lg.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out = np.zeros((q.shape[0], self.d))
        c0 = 0
        for Vb, Rv_b in values:
            n = Vb.shape[0]
            out += (p[:, c0:c0 + n] @ Vb) @ Rv_b
            c0 += n
        return out


def quest_decode(q, K, V, st: Strategy, T0=None):
    """The Quest comparator: token-block selection alone on the uncompressed cache.

    Quest is the block-selection baseline the pages compare against ([S]
    sec. 6.1 baselines, sec. 6.3 "over Quest"; [N] describes its per-block
    min/max keys).  With the same segment layout as the method: sink tokens
    [0, S) and the window [T-W, T) are always attended; the middle [S, T-W)
    is cut into blocks of B tokens from S.  Each block keeps the elementwise
    min and max of its raw keys; a block's score is
    max over the group's heads of (1/sqrt(d)) sum_j max(q_j mn_j, q_j mx_j);
    the k best blocks of the scored segments are kept (ties to the lower
    block id; segments marked always are attended whole), and each head
    attends, softmax(q K^T / sqrt(d)) V, over the raw rows of sinks, window,
    kept and always-attended blocks.  Every channel is kept.
    q: [G, d]; K, V: [T, d] (float64 values); T0: the length at which the
    segment boundaries were fixed (default T).  Returns (ids, out [G, d]).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    T, d = K.shape
    S, W, B = st.n_sink, st.window, st.block
    mid = max(0, T - S - W)
    nb = (mid + B - 1) // B
    firsts = segment_first_blocks(T if T0 is None else T0, st)
    always = [bool(st.segments[block_segment(b, firsts)][2]) for b in range(nb)]
    scores = np.empty(nb)
    for b in range(nb):
        rows = K[S + b * B:S + min((b + 1) * B, mid)]
        mn, mx = rows.min(axis=0), rows.max(axis=0)
        scores[b] = max(sum(max(q[h, j] * mn[j], q[h, j] * mx[j]) for j in range(d))
                        for h in range(q.shape[0])) / math.sqrt(d)
    cand = [b for b in range(nb) if not always[b]]
    k = n_select(len(cand), st)
    ids = sorted(sorted(cand, key=lambda b: (-scores[b], b))[:k])
    keep = list(range(min(S, T))) + list(range(S + mid, T))
    for b in sorted(ids + [b for b in range(nb) if always[b]]):
        keep += list(range(S + b * B, S + min((b + 1) * B, mid)))
    logits = q @ K[keep].T / math.sqrt(d)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return np.array(ids, dtype=np.int64), p @ V[keep]


def speedup_bound(alpha, beta):
    """[N] Eq. (15): T d / (s_sel r) = 1 / (alpha beta)."""
    return 1.0 / (alpha * beta)


def meta_overhead(block, d=D_HEAD, elem_bytes=2):
    """Per-block min/max keys relative to the block's uncompressed K+V ([S] sec. 6.3)."""
    return (2 * d * elem_bytes) / (2 * block * d * elem_bytes)


def packed_bytes_per_token(r, bitmap_group=0, d=D_HEAD):
    """K and V: r bf16 values plus r uint8 indices each, or with a bitmap of
    d / g bits in place of the indices ([S] sec. 5.1)."""
    pos = d // bitmap_group // 8 if bitmap_group else r
    return 2 * (2 * r + pos)
