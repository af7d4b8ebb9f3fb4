"""Per-segment sequence retention ([S] sec. 4.3: each segment's strategy has
its own sequence retention rate) through the C ABI, against the fp64 oracle.

When a scored segment gives its own rate, every scored segment keeps its own
ceil(rate * n / 1000) best blocks (ties to the lower id) and the ids of all
segments come in one ascending row.  Rotations are exact in bf16 (signed
permutations), so the stored block keys equal the oracle's.  Bars: scores
within the fp32 bound; ids
bit-exact against the per-segment top-k of the kernel's own scores and equal
to the oracle's own choice except at near-ties; attention per head within
5e-3 relative L2.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import build as Bld
from oracle import mosaickv_oracle as O
from tests.harness import Case, Pair, rel_l2, score_tolerance

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    Bld.build()


def _check(p, seqs, q, ids, n_sel, scores, out):
    near = 0
    G = p.c.G
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        per, grp = oc.scores(qs)
        mn, mx = oc.score_keys()
        nb = oc.n_blocks_mid()
        tol = np.array([score_tolerance(qs @ oc.rotations_of_block(b)[0].T, mn[b:b + 1], mx[b:b + 1])[0]
                        for b in range(nb)])
        cand = oc.candidates()
        got_s = scores[s, h, :nb].astype(np.float64)
        assert np.all(np.abs(got_s[cand] - grp[cand]) <= tol[cand]), (s, h)
        assert n_sel[s, h] == oc.n_selected(), (s, h)
        got = ids[s, h, :n_sel[s, h]]
        # the per-segment top-k of the kernel's own scores, bit for bit
        want_own = []
        for sg, segdef in enumerate(oc.st.segments):
            c = oc.segment_candidates(sg)
            if len(c):
                want_own.append(O.topk_blocks(got_s, c, O.n_select(len(c), oc.st, segdef[5] or oc.st.retain_permille)))
        assert np.array_equal(got, np.sort(np.concatenate(want_own))), (s, h)
        want_ids, _ = oc.select(qs)
        if not np.array_equal(got, want_ids):
            near += 1
        want = oc.attention(qs, got)
        for gi in range(G):
            assert rel_l2(out[s, h * G + gi], want[gi]) <= ATOL_REL, (s, h, gi)
    return near


@pytest.mark.parametrize("case", [
    Case(n_q=4, n_kv=2, seq_lens=[4000, 1500], rot="perm", block=16, window=64,
         segments=[(0, 32, 0, 0, 0, 300), (300, 64, 1), (550, 32, 0, 0, 0, 50), (800, 24, 0)],
         steps=[1, 2], seed=130),
    Case(n_q=8, n_kv=1, seq_lens=[80000], rot="perm", block=16, window=128,
         segments=[(0, 38, 0, 0, 0, 20), (600, 38, 0, 0, 0, 150)], steps=[1], seed=131),   # 2 top-k CTAs
    Case(n_q=2, n_kv=2, seq_lens=[2600], rot="perm", block=32, window=64,
         segments=[(0, 38, 0, 0, 0, 400), (500, 38, 0, 0, 0, 30)], steps=[1], seed=133),    # GQA 1
], ids=["four-segments", "long-unit-two-ctas", "gqa1"])
def test_per_segment_retention_select_and_attend(case):
    p = Pair(case)
    p.run_steps()
    seqs = list(range(len(case.seq_lens)))
    q = p.query(30)
    scores = torch.full((len(seqs), case.n_kv, p.mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.block_select(0, seqs, q, scores=scores)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    near = _check(p, seqs, q, ids.cpu().numpy(), n_sel.cpu().numpy(), scores.cpu().numpy(),
                  out.cpu().to(torch.float64).numpy())
    assert near <= 1


def test_per_segment_retention_fused_and_own_rotation():
    """The fused append + selection, then a closed segment re-packed under its
    own rotation: the per-segment selection also places each segment's ids for
    the attention's rotation classes."""
    from compressed_kv_cache_vector_gb300 import binding, synth
    case = Case(n_q=4, n_kv=2, seq_lens=[3000, 1800], rot="perm", block=32, window=64,
                segments=[(0, 32, 0, 0, 0, 250), (600, 32, 0, 0, 0, 80)], steps=[1] * 4, seed=132)
    p = Pair(case)
    for n in case.steps[:3]:     # the fourth token goes through the fused call below
        p.step(n)
    S, B = case.n_sink, case.block
    for (l, s, h) in p.units:
        lay = p.mk.layout(l, s, h)
        fb = lay["seg_first_block"]
        rows = slice(S + fb[0] * B, S + fb[1] * B)
        Kraw = synth.bf16_values(p.K[(l, s, h)])
        Vraw = synth.bf16_values(p.V[(l, s, h)])
        Rk_s = O.rotation_from_keys(Kraw[rows])[0].astype(np.float32)
        Rv_s = O.rotation_from_keys(Vraw[rows])[0].astype(np.float32)
        pages, meta, _ = binding.host_pack_blocks(Rk_s, Rv_s, p.K[(l, s, h)][rows].cpu(), p.V[(l, s, h)][rows].cpu(),
                                                  B, 24, 0, lay["page_stride"])
        p.mk.swap_segment(l, s, h, 0, 24, 0, pages, meta, R_k=Rk_s, R_v=Rv_s)
        torch.cuda.synchronize()
        p.orc[(l, s, h)].recompress_segment(0, Kraw, Vraw, 24, 0, Rk_s.astype(np.float64), Rv_s.astype(np.float64))
    seqs = [0, 1]
    k = torch.stack([torch.stack([p.K[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
    v = torch.stack([torch.stack([p.V[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
    q = p.query(31)
    scores = torch.full((2, 2, p.mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.append_select(0, seqs, k, v, q, scores=scores)
    for (l, s, h), oc in p.orc.items():
        t = p.T[s]
        oc.append(synth.bf16_values(p.K[(l, s, h)][t:t + 1]), synth.bf16_values(p.V[(l, s, h)][t:t + 1]))
    for s in seqs:
        p.T[s] += 1
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    near = _check(p, seqs, q, ids.cpu().numpy(), n_sel.cpu().numpy(), scores.cpu().numpy(),
                  out.cpu().to(torch.float64).numpy())
    assert near <= 1


def test_per_segment_retention_all_ties_long():
    """Every token carries the same key, so every scored block ties; each
    scored segment then keeps its k_s lowest block ids.  About 12,500 blocks:
    the top-k runs in four CTAs and the segments' histograms hold one bin."""
    from compressed_kv_cache_vector_gb300 import synth
    from compressed_kv_cache_vector_gb300.binding import MosaicKV, make_config
    from tests.harness import D, signed_permutation
    T, S, W, B, G = 200_000, 4, 64, 16, 4
    segments = [(0, 32, 0, 0, 0, 80), (400, 16, 1), (600, 32, 0, 0, 0, 150)]
    st = O.Strategy(S, W, B, list(segments), 0, 100)
    cfg = make_config(G, 1, 1, 1, T + 1, S, W, B, segments, 0, 100)
    mk = MosaicKV(cfg, "cuda")
    Rk, Rv = signed_permutation(41), signed_permutation(43)
    mk.set_rotation(0, 0, 0, Rk.astype(np.float32), Rv.astype(np.float32))
    rows = synth.lowrank_outlier(64, D, 0.9, 321, device="cuda")
    k_row, v_row = rows[3:4], rows[7:8]
    mk.append(0, [0], [T], k_row.expand(T, D).reshape(T, 1, D).contiguous(),
              v_row.expand(T, D).reshape(T, 1, D).contiguous())
    q = synth.query(1, G, D, 78, device="cuda")
    ids, n_sel = mk.block_select(0, [0], q)
    torch.cuda.synchronize()
    assert mk.poll_error()[0] == 0
    nb = O.n_middle_blocks(T, st)
    firsts = O.segment_first_blocks(T, st)
    want, total = [], 0
    for s, sg in enumerate(st.segments):
        if sg[2]:
            continue
        lo, hi = min(firsts[s], nb), (min(firsts[s + 1], nb) if s + 1 < len(firsts) else nb)
        k_s = O.n_select(hi - lo, st, sg[5] or 100)
        want += list(range(lo, lo + k_s))
        total += k_s
    assert int(n_sel[0, 0]) == total
    assert np.array_equal(ids[0, 0, :total].cpu().numpy(), np.array(want))
