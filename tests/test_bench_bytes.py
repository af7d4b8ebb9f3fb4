"""The bench's algorithmic bytes (the roofline's numerator) against the
per-step byte counts written out by hand for the 128K and 1M workloads.
CPU only."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from compressed_kv_cache_vector_gb300 import configs  # noqa: E402

D = 128


def _by_hand(T, S, W, B, r, G, retain_permille, topk_fixed=0):
    mid = T - S - W
    nblk = -(-mid // B)
    k = min(topk_fixed, nblk) if topk_fixed else min(max(1, -(-retain_permille * nblk // 1000)), nblk)
    attn = k * 6 * B * r + (S + W) * 2 * D * 2 + D * D * 4 + G * D * (4 + 2)  # pages, dense rows, R_v, q'/out
    select = nblk * 2 * D * 2 + G * D * 2 + D * D * 4                          # meta, q, R_k^T
    append = 2 * D * 2 + 2 * D * D * 4 + 2 * D * 2 + 2 * D * 2 + 6 * r + 2 * 2 * D * 2
    return {"append": append, "select": select, "attn": attn}, k, nblk


def test_c3_bytes_per_unit():
    wl = configs.get("c3")
    T = wl.seq_lens[0]
    got = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
    want, k, nblk = _by_hand(T, 4, 256, 32, 38, 4, 100)
    assert (k, nblk) == (409, 4088)
    assert got == want
    assert 8 * got["attn"] == 25_486_336      # one attention launch (8 kv heads): the roofline's bytes


def test_c4_bytes_per_unit():
    wl = configs.get("c4")
    T = wl.seq_lens[0]
    got = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
    want, k, nblk = _by_hand(T, 4, 512, 64, 38, 4, 50)
    assert (k, nblk) == (819, 16376)
    assert got == want


def test_compressed_keys_shrink_the_selection_bytes():
    wl = configs.get("c3")
    T = wl.seq_lens[0]
    full = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
    wl.meta_channels = 32
    comp = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
    nblk = 4088
    assert full["select"] - comp["select"] == nblk * (2 * D * 2 - 160)
    assert comp["attn"] == full["attn"]


def test_bitmap_pages_shrink_the_attention_bytes():
    # Bitmap pages: 128 / g bits per vector in place of r index bytes, so a
    # token's K and V cost 2 (2 r + 16 / g) bytes instead of 6 r.
    wl = configs.get("c3")
    T = wl.seq_lens[0]
    base = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
    k, B = 409, 32
    for g, r in ((1, 38), (4, 40), (8, 40)):
        wl.elem_group = g
        wl.segments = [(0, r, 0)]
        got = bench.unit_bytes(wl, T, bench.segment_firsts(wl, T))
        assert got["attn"] - base["attn"] == k * B * (2 * (2 * r + 16 // g) - 6 * 38)
        assert got["append"] - base["append"] == 2 * (2 * r + 16 // g) - 6 * 38
