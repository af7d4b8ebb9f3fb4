"""Parity of the bitmap page format ([S] sec. 5.1: a position bitmap per vector
in place of the channel indices, one bit per channel or per group of g
adjacent channels) with the fp64 oracle, through the C ABI.

Bars as in test_gpu_parity: pages, meta and rows bit-exact under exactly
representable rotations (signed permutations), the grouped selection decided
in fp32 on both sides; attention within 5e-3 relative L2 per head.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import build as Bld
from oracle import mosaickv_oracle as O
from tests.harness import Case, Pair, bits, page_rows, rel_l2, score_tolerance
from tests.harness import check_storage as _check_storage

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    Bld.build()


def _segments(g):
    # r and truncation multiples of g; one r above the prefill's staging limit
    # (68), whose rows go straight to the pages.
    if g == 1:
        return [(0, 38, 0), (400, 17, 1, 96), (700, 80, 0)]
    return [(0, 40, 0), (400, 16, 1, 96), (700, 72, 0)]


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_bitmap_storage_bitexact_bulk_then_decode(g):
    case = Case(n_q=4, n_kv=2, seq_lens=[2000, 700], rot="perm", block=32, window=64, page_format=2, elem_group=g,
                segments=_segments(g), steps=[1] * 20 + [5, 33, 1], seed=60 + g)
    p = Pair(case)
    for u in p.units:
        _check_storage(p, u)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
        oc = p.orc[u]
        if g > 1:   # whole groups: every kept index run is g-aligned
            assert np.all(oc.kidx[4:oc.T, 0] % g == 0)


@pytest.mark.parametrize("g", [1, 4])
def test_bitmap_storage_from_empty_and_compressed_keys(g):
    # Single-token appends through sinks, window and middle, with
    # channel-compressed block keys ([S] sec. 5.2) beside the bitmaps.
    case = Case(n_q=2, n_kv=1, seq_lens=[2], rot="perm", n_sink=4, window=16, block=16, page_format=2,
                elem_group=g, segments=[(0, 40, 0)], meta_channels=24, steps=[1] * 60 + [2, 16, 9], seed=70 + g)
    p = Pair(case)
    p.run_steps()
    _check_storage(p, p.units[0])


@pytest.mark.parametrize("g,seq_lens,topk,G", [(1, [3000, 900], 0, 4), (2, [3000, 900], 0, 4), (4, [3000, 900], 0, 4),
                                               (8, [3000, 900], 0, 4), (4, [42000], 600, 4), (8, [3000, 900], 0, 8),
                                               (2, [3000, 900], 0, 1)],
                         ids=["g1", "g2", "g4", "g8", "g4-long-16warps", "g8-gqa8", "g2-gqa1"])
def test_bitmap_decode_attention_matches_oracle(g, seq_lens, topk, G):
    n_kv = 2 if len(seq_lens) > 1 else 1
    case = Case(n_q=G * n_kv, n_kv=n_kv, seq_lens=seq_lens, rot="eigh",
                block=32 if topk == 0 else 64, window=64 if topk == 0 else 128, page_format=2, elem_group=g,
                segments=_segments(g) if topk == 0 else [(0, 40, 0)], topk_fixed=topk,
                retain_permille=0 if topk else 100, steps=[1, 1, 2], seed=80 + g)
    p = Pair(case)
    p.run_steps()
    q = p.query(3)
    seqs = list(range(len(seq_lens)))
    ids, n_sel = p.mk.block_select(0, seqs, q)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    out = out.cpu().to(torch.float64).numpy()
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    G = case.G
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        want = oc.attention(qs, ids[s, h, :n_sel[s, h]])
        for gi in range(G):
            e = rel_l2(out[s, h * G + gi], want[gi])
            assert e <= ATOL_REL, (s, h, gi, e)


@pytest.mark.parametrize("g", [1, 8])
def test_bitmap_append_select_equals_separate_calls(g):
    """The fused decode append + selection writes the same bitmap pages as the
    separate append, and gives the same ids and attention output."""
    case = Case(n_q=4, n_kv=2, seq_lens=[2500, 700], rot="eigh", block=32, window=64, page_format=2,
                elem_group=g, segments=_segments(g), oracle_units=[], seed=90 + g)
    n_steps = 40
    case.steps = [1] * n_steps
    a, b = Pair(case), Pair(case)
    seqs = [0, 1]
    for step in range(n_steps):
        k = torch.stack([torch.stack([a.K[(0, s, h)][a.T[s]] for h in range(2)]) for s in seqs]).contiguous()
        v = torch.stack([torch.stack([a.V[(0, s, h)][a.T[s]] for h in range(2)]) for s in seqs]).contiguous()
        q = a.query(200 + step)
        a.mk.append(0, seqs, [1, 1], k, v)
        ids_a, ns_a = a.mk.block_select(0, seqs, q)
        ids_b, ns_b = b.mk.append_select(0, seqs, k, v, q)
        out_a = a.mk.decode_attn(0, seqs, ids_a, ns_a)
        out_b = b.mk.decode_attn(0, seqs, ids_b, ns_b)
        torch.cuda.synchronize()
        for s in seqs:
            a.T[s] += 1
        assert np.array_equal(ns_a.cpu().numpy(), ns_b.cpu().numpy()), step
        assert np.array_equal(bits(out_a), bits(out_b)), step
    assert a.mk.poll_error() == (0, 0) and b.mk.poll_error() == (0, 0)
    S, W, B = case.n_sink, case.window, case.block
    for s in seqs:
        T = case.seq_lens[s] + n_steps
        mid = max(0, T - S - W)
        nb = (mid + B - 1) // B
        for h in range(2):
            va, vb = a.mk.unit_views(0, s, h), b.mk.unit_views(0, s, h)
            fb = va["layout"]["seg_first_block"]
            pa, pb_ = va["pages"].cpu().numpy(), vb["pages"].cpu().numpy()
            for blk in range(nb):   # the live rows of every block (the arena is not zeroed)
                seg = [i for i, f in enumerate(fb) if blk >= f][-1]
                r = case.segments[seg][1]
                n_live = min(B, mid - blk * B)
                for x, y in zip(page_rows(pa[blk], B, r, n_live, case.pos_bytes(r)),
                                page_rows(pb_[blk], B, r, n_live, case.pos_bytes(r))):
                    assert np.array_equal(x, y), (s, h, blk)
            assert np.array_equal(bits(va["meta"])[:nb], bits(vb["meta"])[:nb]), (s, h)


@pytest.mark.parametrize("own", [False, True], ids=["head-rotation", "own-rotation"])
def test_bitmap_swap_closed_segment(own):
    """[S] sec. 5.4 in the bitmap format: a closed segment re-packed on the host
    (new r and truncation, multiples of the group) replaces the GPU's version;
    bytes equal the oracle's re-compression, attention follows."""
    from compressed_kv_cache_vector_gb300 import binding, synth
    g = 4
    case = Case(n_q=4, n_kv=2, seq_lens=[3000, 1800], rot="perm", block=32, window=64, page_format=2,
                elem_group=g, segments=[(0, 40, 0), (600, 40, 0)], steps=[1] * 3, seed=95)
    p = Pair(case)
    p.run_steps()
    S, B = case.n_sink, case.block
    r_new, keep = 24, 96
    for (l, s, h) in p.units:
        lay = p.mk.layout(l, s, h)
        fb = lay["seg_first_block"]
        rows = slice(S + fb[0] * B, S + fb[1] * B)
        Kraw = synth.bf16_values(p.K[(l, s, h)])
        Vraw = synth.bf16_values(p.V[(l, s, h)])
        if own:
            Rk_s = O.rotation_from_keys(Kraw[rows])[0].astype(np.float32)
            Rv_s = O.rotation_from_keys(Vraw[rows])[0].astype(np.float32)
        else:
            Rk_s, Rv_s = p.R[(l, s, h)]
        pages, meta, _ = binding.host_pack_blocks(Rk_s, Rv_s, p.K[(l, s, h)][rows].cpu(), p.V[(l, s, h)][rows].cpu(),
                                                  B, r_new, keep, lay["page_stride"], 0, 2, g)
        p.mk.swap_segment(l, s, h, 0, r_new, keep, pages, meta, R_k=Rk_s if own else None,
                          R_v=Rv_s if own else None)
        torch.cuda.synchronize()
        p.orc[(l, s, h)].recompress_segment(0, Kraw, Vraw, r_new, keep,
                                            Rk_s.astype(np.float64) if own else None,
                                            Rv_s.astype(np.float64) if own else None)
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
    q = p.query(11)
    scores = torch.full((2, 2, p.mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.block_select(0, [0, 1], q, scores=scores)
    out = p.mk.decode_attn(0, [0, 1], ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    out, scores = out.cpu().to(torch.float64).numpy(), scores.cpu().numpy()
    G = case.G
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        cand = oc.candidates()
        _, grp = oc.scores(qs)
        mn, mx = oc.score_keys()
        nb = oc.n_blocks_mid()
        tol = np.array([score_tolerance(qs @ oc.rotations_of_block(b)[0].T, mn[b:b + 1], mx[b:b + 1])[0]
                        for b in range(nb)])
        assert np.all(np.abs(scores[s, h, :nb][cand].astype(np.float64) - grp[cand]) <= tol[cand]), (s, h)
        want = oc.attention(qs, ids[s, h, :n_sel[s, h]])
        for gi in range(G):
            assert rel_l2(out[s, h * G + gi], want[gi]) <= ATOL_REL, (s, h, gi)


# Per-segment element-group sizes ([S] sec. 4.3): 8, 2 and 1 in one cache (the
# cache's default, 4, for none of them), one truncated, one above the
# prefill's staging limit.  Prefill tiles and decode warps then hold tokens of
# segments with different group sizes.
_MIXED = [(0, 40, 0, 0, 8), (400, 16, 1, 96, 2), (700, 72, 0, 0, 1)]


def test_bitmap_per_segment_groups_storage_and_attention():
    case = Case(n_q=4, n_kv=2, seq_lens=[2300, 900], rot="perm", block=32, window=64, page_format=2, elem_group=4,
                segments=_MIXED, steps=[1] * 20 + [5, 33, 1], seed=120)
    p = Pair(case)
    for u in p.units:
        _check_storage(p, u)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
        oc = p.orc[u]
        assert [sg[4] for sg in oc.st.segments] == [8, 2, 1]
    q = p.query(13)
    ids, n_sel = p.mk.block_select(0, [0, 1], q)
    out = p.mk.decode_attn(0, [0, 1], ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    out = out.cpu().to(torch.float64).numpy()
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    G = case.G
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        want = oc.attention(qs, ids[s, h, :n_sel[s, h]])
        for gi in range(G):
            assert rel_l2(out[s, h * G + gi], want[gi]) <= ATOL_REL, (s, h, gi)


def test_bitmap_per_segment_groups_swap_own_rotation():
    """Per-segment groups, then a closed segment
    re-packed on the host under its own rotation: it keeps its group size
    (8), takes a new r and truncation."""
    from compressed_kv_cache_vector_gb300 import binding, synth
    case = Case(n_q=4, n_kv=2, seq_lens=[3000, 1800], rot="perm", block=32, window=64, page_format=2, elem_group=4,
                segments=[(0, 40, 0, 0, 8), (600, 38, 0, 0, 1)], steps=[1] * 3, seed=121)
    p = Pair(case)
    p.run_steps()
    S, B = case.n_sink, case.block
    r_new, keep = 24, 96
    for (l, s, h) in p.units:
        lay = p.mk.layout(l, s, h)
        fb = lay["seg_first_block"]
        rows = slice(S + fb[0] * B, S + fb[1] * B)
        Kraw = synth.bf16_values(p.K[(l, s, h)])
        Vraw = synth.bf16_values(p.V[(l, s, h)])
        Rk_s = O.rotation_from_keys(Kraw[rows])[0].astype(np.float32)
        Rv_s = O.rotation_from_keys(Vraw[rows])[0].astype(np.float32)
        pages, meta, _ = binding.host_pack_blocks(Rk_s, Rv_s, p.K[(l, s, h)][rows].cpu(), p.V[(l, s, h)][rows].cpu(),
                                                  B, r_new, keep, lay["page_stride"], 0, 2, 8)
        p.mk.swap_segment(l, s, h, 0, r_new, keep, pages, meta, R_k=Rk_s, R_v=Rv_s)
        torch.cuda.synchronize()
        p.orc[(l, s, h)].recompress_segment(0, Kraw, Vraw, r_new, keep, Rk_s.astype(np.float64),
                                            Rv_s.astype(np.float64))
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
        assert p.orc[u].st.segments[0][4] == 8
    q = p.query(14)
    ids, n_sel = p.mk.block_select(0, [0, 1], q)
    out = p.mk.decode_attn(0, [0, 1], ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    out = out.cpu().to(torch.float64).numpy()
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    G = case.G
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        want = oc.attention(qs, ids[s, h, :n_sel[s, h]])
        for gi in range(G):
            assert rel_l2(out[s, h * G + gi], want[gi]) <= ATOL_REL, (s, h, gi)
    # a swap whose r is not a multiple of the segment's group is refused
    lay = p.mk.layout(0, 0, 0)
    pages = np.zeros((lay["seg_first_block"][1], lay["page_stride"]), dtype=np.uint8)
    meta = np.zeros((lay["seg_first_block"][1], 2, 128), dtype=np.uint16)
    with pytest.raises(binding.MosaicKVError):
        p.mk.swap_segment(0, 0, 0, 0, 20, 0, pages, meta)
