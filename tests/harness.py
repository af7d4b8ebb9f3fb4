"""Builds the same compressed cache on both sides for the parity tests.

The CUDA side goes through the C ABI (compressed_kv_cache_vector_gb300.binding);
the oracle side through oracle.mosaickv_oracle.  Both receive the same seeded
inputs from compressed_kv_cache_vector_gb300.synth and the same rotations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from compressed_kv_cache_vector_gb300 import synth
from compressed_kv_cache_vector_gb300.binding import MosaicKV, make_config
from oracle import mosaickv_oracle as O

D = 128


def signed_permutation(seed):
    rng = np.random.default_rng(seed)
    P = np.zeros((D, D))
    P[np.arange(D), rng.permutation(D)] = rng.choice([-1.0, 1.0], size=D)
    return P


@dataclass
class Case:
    n_q: int = 4
    n_kv: int = 1
    seq_lens: list = field(default_factory=lambda: [1000])
    n_sink: int = 4
    window: int = 64
    block: int = 16
    segments: list = field(default_factory=lambda: [(0, 32, 0)])
    topk_fixed: int = 0
    retain_permille: int = 100
    decay: float = 0.9
    steps: list = field(default_factory=list)     # tokens appended per decode step (all sequences)
    rot: str = "eigh"                             # "eigh", "perm" or "identity"
    seed: int = 0
    n_layers: int = 1
    oracle_units: list = None                     # [(layer, seq, kvh)]; None = all
    meta_channels: int = 0                        # > 0: channel-compressed per-block keys
    page_format: int = 0                          # 1: uncompressed pages (the Quest comparator); 2: bitmaps
    elem_group: int = 0                           # bitmap pages: channels per bitmap bit (0 = 1)

    @property
    def G(self):
        return self.n_q // self.n_kv

    def strategy(self):
        return O.Strategy(self.n_sink, self.window, self.block, list(self.segments),
                          self.topk_fixed, self.retain_permille, self.meta_channels, self.bitmap_group)

    @property
    def bitmap_group(self):
        return max(1, self.elem_group) if self.page_format == 2 else 0

    def pos_bytes(self, r):
        return 16 // self.bitmap_group if self.bitmap_group else r


class Pair:
    """GPU cache + oracle caches for a Case, advanced together."""

    def __init__(self, case: Case, device="cuda"):
        self.c = case
        self.dev = device
        extra = sum(case.steps)
        self.T_total = [t + extra for t in case.seq_lens]
        cfg = make_config(case.n_q, case.n_kv, case.n_layers, len(case.seq_lens), max(self.T_total) + 1,
                          case.n_sink, case.window, case.block, case.segments, case.topk_fixed,
                          case.retain_permille, case.meta_channels, case.page_format, case.elem_group)
        self.mk = MosaicKV(cfg, device)
        self.K, self.V, self.R = {}, {}, {}
        units = case.oracle_units
        if units is None:
            units = [(l, s, h) for l in range(case.n_layers) for s in range(len(case.seq_lens))
                     for h in range(case.n_kv)]
        self.units = units
        self.orc = {}
        for l in range(case.n_layers):
            for s, T in enumerate(self.T_total):
                for h in range(case.n_kv):
                    sd = synth.seed_for("test", case.seed, l, s, h)
                    k = synth.lowrank_outlier(T, D, case.decay, sd, device=device)
                    v = synth.lowrank_outlier(T, D, case.decay, sd + 1, device=device)
                    self.K[(l, s, h)], self.V[(l, s, h)] = k, v
                    t0 = case.seq_lens[s]
                    if case.rot == "identity":
                        Rk, Rv = np.eye(D), np.eye(D)
                    elif case.rot == "perm":
                        Rk, Rv = signed_permutation(sd), signed_permutation(sd + 7)
                    else:
                        Rk, _ = O.rotation_from_keys(synth.bf16_values(k[:t0]))
                        Rv, _ = O.rotation_from_keys(synth.bf16_values(v[:t0]))
                    Rk = Rk.astype(np.float32)
                    Rv = Rv.astype(np.float32)
                    self.R[(l, s, h)] = (Rk, Rv)
                    self.mk.set_rotation(l, s, h, Rk, Rv)
                    if (l, s, h) in units:
                        oc = O.OracleCache(case.strategy(), T + 1)
                        oc.set_rotation(Rk.astype(np.float64), Rv.astype(np.float64))
                        self.orc[(l, s, h)] = oc
        self.T = [0] * len(case.seq_lens)
        self._append_all([t for t in case.seq_lens])

    def _append_all(self, n_new):
        c = self.c
        seqs = [s for s in range(len(c.seq_lens)) if n_new[s] > 0]
        for l in range(c.n_layers):
            ks, vs = [], []
            for s in seqs:
                lo, hi = self.T[s], self.T[s] + n_new[s]
                ks.append(torch.stack([self.K[(l, s, h)][lo:hi] for h in range(c.n_kv)], dim=1))
                vs.append(torch.stack([self.V[(l, s, h)][lo:hi] for h in range(c.n_kv)], dim=1))
            k = torch.cat(ks).contiguous()
            v = torch.cat(vs).contiguous()
            self.mk.append(l, seqs, [n_new[s] for s in seqs], k, v)
            for (ll, s, h), oc in self.orc.items():
                if ll == l and n_new[s] > 0:
                    lo, hi = self.T[s], self.T[s] + n_new[s]
                    oc.append(synth.bf16_values(self.K[(l, s, h)][lo:hi]),
                              synth.bf16_values(self.V[(l, s, h)][lo:hi]))
        for s in seqs:
            self.T[s] += n_new[s]

    def step(self, n):
        self._append_all([n] * len(self.c.seq_lens))

    def run_steps(self):
        for n in self.c.steps:
            self.step(n)

    def query(self, seed):
        c = self.c
        return synth.query(len(c.seq_lens), c.n_q, D, synth.seed_for("q", c.seed, seed), device=self.dev)


def page_rows(page_bytes, B, r, n_live, pb=None):
    """Split one packed page into (kval u16, kpos u8, vval u16, vpos u8) live rows; pb: position bytes per
    token (r uint8 indices by default, or a bitmap's bytes)."""
    p = np.asarray(page_bytes, dtype=np.uint8)
    pb = r if pb is None else pb
    Br, Bp = B * r, B * pb
    kv = p[:2 * Br].view(np.uint16).reshape(B, r)[:n_live]
    ki = p[2 * Br:2 * Br + Bp].reshape(B, pb)[:n_live]
    vv = p[2 * Br + Bp:4 * Br + Bp].view(np.uint16).reshape(B, r)[:n_live]
    vi = p[4 * Br + Bp:4 * Br + 2 * Bp].reshape(B, pb)[:n_live]
    return kv, ki, vv, vi


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def score_tolerance(qr, mn, mx):
    """Bound on |fp32 score - exact score|: 128-term fp32 sums of exact products."""
    terms = np.abs(qr)[:, None, :] * np.maximum(np.abs(mn), np.abs(mx))[None, :, :]
    return (terms.sum(axis=2).max(axis=0) / math.sqrt(D)) * (D + 2) * 2.0 ** -24 + 1e-30


def check_storage(p: Pair, unit):
    """Sinks, window ring, meta and pages bit-exact against the oracle."""
    oc = p.orc[unit]
    l, s, h = unit
    views = p.mk.unit_views(l, s, h)
    S, W, B = p.c.n_sink, p.c.window, p.c.block
    sp = oc.sink_positions()
    if len(sp):
        assert np.array_equal(bits(views["sink_k"])[: len(sp)], O.bf16_bits(oc.Kr[sp]))
        assert np.array_equal(bits(views["sink_v"])[: len(sp)], O.bf16_bits(oc.Vr[sp]))
    wk, wv = bits(views["win_k"]), bits(views["win_v"])
    for pos in oc.window_positions():
        slot = (pos - S) % W
        assert np.array_equal(wk[slot], O.bf16_bits(oc.Kr[pos])), pos
        assert np.array_equal(wv[slot], O.bf16_bits(oc.Vr[pos])), pos
    nb = oc.n_blocks_mid()
    mn, mx = oc.meta()
    meta = bits(views["meta"])[:nb]
    assert np.array_equal(meta[:, 0], O.bf16_bits(mn))
    assert np.array_equal(meta[:, 1], O.bf16_bits(mx))
    if p.c.meta_channels:
        m = p.c.meta_channels
        idx, cmn, cmx = O.compress_key_rows(mn, mx, m)
        rows = views["cmeta"].cpu().numpy()[:nb]
        assert np.array_equal(rows[:, :2 * m].copy().view(np.uint16), O.bf16_bits(cmn))
        assert np.array_equal(rows[:, 2 * m:4 * m].copy().view(np.uint16), O.bf16_bits(cmx))
        assert np.array_equal(rows[:, 4 * m:5 * m], idx.astype(np.uint8))
    pages = views["pages"].cpu().numpy()
    for b in range(nb):
        r = oc.r_of_block(b)
        lo, hi = oc.block_tokens(b)
        g = oc.group_of_block(b)
        pb = 16 // g if g else r
        got = page_rows(pages[b], B, r, hi - lo, pb)
        want = page_rows(oc.page_bytes(b), B, r, hi - lo, pb)
        for g, w_, name in zip(got, want, ("kval", "kidx", "vval", "vidx")):
            assert np.array_equal(g, w_), (b, name)
