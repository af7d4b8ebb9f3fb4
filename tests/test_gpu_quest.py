"""The Quest comparator on the GPU: uncompressed pages, token-block selection alone.

With page_format = MK_PAGES_DENSE the same calls (append, block selection,
attention) run Quest's method ([S] sec. 6.1 baselines, sec. 6.3): the middle
pages keep whole rows, the block keys are the min/max of the raw keys (the
rotation is the identity), and attention reads every channel of the kept
blocks.  Checked against the oracle's quest_decode: stored rows and keys bit
for bit, scores within the fp32 summation bound, ids equal except at a
near-tie inside it, attention relative L2 error per head <= 5e-3.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import synth
from oracle import mosaickv_oracle as O
from tests.harness import Case, Pair, bits, rel_l2, score_tolerance

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


def _check_dense_storage(p, s, h):
    c = p.c
    T = p.T[s]
    S, W, B = c.n_sink, c.window, c.block
    views = p.mk.unit_views(0, s, h)
    K, V = bits(p.K[(0, s, h)][:T]), bits(p.V[(0, s, h)][:T])
    mid = max(0, T - S - W)
    nb = (mid + B - 1) // B
    pages = views["pages"].cpu().numpy()
    for b in range(nb):
        n = min(B, mid - b * B)
        pg = pages[b, :4 * B * 128].copy().view(np.uint16).reshape(2, B, 128)
        assert np.array_equal(pg[0, :n], K[S + b * B:S + b * B + n]), b
        assert np.array_equal(pg[1, :n], V[S + b * B:S + b * B + n]), b
    meta = O.bits_to_value(bits(views["meta"])[:nb])
    Kv = synth.bf16_values(p.K[(0, s, h)][:T])
    for b in range(nb):
        rows = Kv[S + b * B:S + min((b + 1) * B, mid)]
        assert np.array_equal(meta[b, 0], rows.min(axis=0) + 0.0)
        assert np.array_equal(meta[b, 1], rows.max(axis=0) + 0.0)


def _check_decode(p, q, ids, n_sel, out, scores):
    """ids and attention of every (sequence, kv head) against quest_decode;
    returns the number of near-ties met."""
    c = p.c
    G = c.G
    S, W, B = c.n_sink, c.window, c.block
    near = 0
    ids, n_sel, out = ids.cpu().numpy(), n_sel.cpu().numpy(), out.cpu().to(torch.float64).numpy()
    scores = scores.cpu().numpy()
    st = c.strategy()
    for s in range(len(c.seq_lens)):
        T = p.T[s]
        mid = max(0, T - S - W)
        nb = (mid + B - 1) // B
        for h in range(c.n_kv):
            qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
            K = synth.bf16_values(p.K[(0, s, h)][:T])
            V = synth.bf16_values(p.V[(0, s, h)][:T])
            want_ids, want = O.quest_decode(qs, K, V, st, T0=c.seq_lens[s])
            k = len(want_ids)
            assert n_sel[s, h] == k
            got = ids[s, h, :k]
            # the kernel's scores against the raw block keys' exact scores
            mn = np.stack([K[S + b * B:S + min((b + 1) * B, mid)].min(axis=0) for b in range(nb)])
            mx = np.stack([K[S + b * B:S + min((b + 1) * B, mid)].max(axis=0) for b in range(nb)])
            grp = O.block_scores(qs, mn, mx)[1]
            tol = score_tolerance(qs, mn, mx)
            got_s = scores[s, h, :nb].astype(np.float64)
            assert np.all(np.abs(got_s - grp) <= tol), (s, h)
            assert np.array_equal(got, O.topk_blocks(got_s, np.arange(nb), k))
            if not np.array_equal(got, want_ids):
                srt = np.sort(grp)[::-1]
                assert srt[k - 1] - srt[k] <= 2 * tol.max(), (s, h)
                near += 1
                want = _attend(qs, K, V, st, got, T)
            for g in range(G):
                assert rel_l2(out[s, h * G + g], want[g]) <= ATOL_REL, (s, h, g)
    return near


def _attend(qs, K, V, st, ids, T):
    S, W, B = st.n_sink, st.window, st.block
    mid = max(0, T - S - W)
    keep = list(range(min(S, T))) + list(range(S + mid, T))
    for b in ids:
        keep += list(range(S + b * B, S + min((b + 1) * B, mid)))
    return O.softmax_attention(qs, K[keep], V[keep])


@pytest.mark.parametrize("G,block,seq_lens", [(4, 16, [3000, 1700]), (8, 32, [5000]), (1, 64, [4100, 900])])
def test_quest_pages_selection_and_attention(G, block, seq_lens):
    case = Case(n_q=2 * G, n_kv=2, seq_lens=seq_lens, rot="identity", block=block, window=64,
                segments=[(0, 128, 0)], retain_permille=100, page_format=1, oracle_units=[], seed=70 + G,
                steps=[1] * 6 + [3])
    p = Pair(case)
    seqs = list(range(len(seq_lens)))
    for step in range(6):           # the fused decode path: one token per sequence and step
        k = torch.stack([torch.stack([p.K[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
        v = torch.stack([torch.stack([p.V[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
        q = p.query(step)
        scores = torch.full((len(seqs), 2, p.mk.nblk_cap), float("nan"), device="cuda")
        ids, n_sel = p.mk.append_select(0, seqs, k, v, q, scores=scores)
        out = p.mk.decode_attn(0, seqs, ids, n_sel)
        torch.cuda.synchronize()
        for s in seqs:
            p.T[s] += 1
        assert _check_decode(p, q, ids, n_sel, out, scores) <= 1
    p.step(3)                       # and the separate append path, three tokens at once
    q = p.query(9)
    scores = torch.full((len(seqs), 2, p.mk.nblk_cap), float("nan"), device="cuda")
    ids, n_sel = p.mk.block_select(0, seqs, q, scores=scores)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    assert _check_decode(p, q, ids, n_sel, out, scores) <= 1
    for s in seqs:
        for h in range(2):
            _check_dense_storage(p, s, h)
