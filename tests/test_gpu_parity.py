"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bars:
  * integer / byte work bit-exact: selected channel indices, packed pages,
    stored sink/window rows, block min/max keys (both sides fed the same bf16
    rotated vectors by using an exactly representable rotation: identity or a
    signed permutation), and the top-k ids given the kernel's own fp32 scores;
  * rotation with a general orthogonal R: within 1 bf16 ulp of the fp64 value
    rounded once (the kernel accumulates in fp32);
  * block scores: within the fp32 summation bound of the exact value; the
    chosen block set equals the oracle's except at near-ties within that bound;
  * attention output: relative L2 error per head <= 5e-3.
"""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import build as Bld
from compressed_kv_cache_vector_gb300.binding import MosaicKVError, make_config, MosaicKV
from oracle import mosaickv_oracle as O
from tests.harness import D, Case, Pair, bits, page_rows, rel_l2, score_tolerance
from tests.harness import check_storage as _check_storage

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    Bld.build()


@pytest.mark.parametrize("rot", ["identity", "perm"])
def test_append_storage_bitexact_bulk_then_decode(rot):
    case = Case(n_q=4, n_kv=2, seq_lens=[1000, 333], rot=rot, steps=[1] * 20 + [5, 17, 1, 70, 1],
                segments=[(0, 32, 0)], seed=1)
    p = Pair(case)
    for u in p.units:
        _check_storage(p, u)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
    assert p.mk.seq_length(0, 0) == 1000 + sum(case.steps)


def test_append_storage_multisegment_r128_block64():
    case = Case(n_q=8, n_kv=1, seq_lens=[3000], rot="perm", block=64, window=100, n_sink=0,
                segments=[(0, 128, 0), (300, 17, 1), (700, 64, 0)], steps=[1] * 40 + [3], seed=2)
    p = Pair(case)
    p.run_steps()
    for u in p.units:
        _check_storage(p, u)


def test_append_storage_truncated_bottom_channels():
    # [S] sec. 5.2: the bottom rotated channels are truncated before the
    # per-vector top-r (here the first 96 of 128 are eligible).
    case = Case(n_q=4, n_kv=2, seq_lens=[1500, 400], rot="perm", window=64,
                segments=[(0, 38, 0, 96), (500, 64, 1, 96)], steps=[1] * 30 + [7], seed=21)
    p = Pair(case)
    for u in p.units:
        _check_storage(p, u)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
        oc = p.orc[u]
        assert int(oc.kidx[:oc.T].max()) < 96 and int(oc.vidx[:oc.T].max()) < 96


def test_append_storage_compressed_block_keys():
    # [S] sec. 5.2: the per-block keys are channel-compressed too (here 24 of 128).
    case = Case(n_q=4, n_kv=2, seq_lens=[1300, 333], rot="perm", block=32, window=64, meta_channels=24,
                steps=[1] * 40 + [9, 1], seed=23)
    p = Pair(case)
    for u in p.units:
        _check_storage(p, u)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)


def test_append_from_empty_through_sinks_and_window():
    # Starts below S+W; single-token appends walk through sinks, window, middle.
    case = Case(n_q=2, n_kv=1, seq_lens=[2], rot="perm", n_sink=4, window=16, block=16,
                steps=[1] * 60 + [2, 16, 9], seed=3)
    p = Pair(case)
    p.run_steps()
    _check_storage(p, p.units[0])


def test_rotation_within_fp32_accumulation_bound():
    # The kernel sums 128 exact bf16 x fp32 products in fp32, then rounds to
    # bf16 once.  Its result must be the bf16 rounding of some value within
    # the fp32 summation bound of the exact product; away from rounding
    # boundaries it equals the oracle's single fp64 -> bf16 rounding.
    case = Case(n_q=4, n_kv=2, seq_lens=[600], window=600 - 4, rot="eigh", seed=4)
    p = Pair(case)
    flips, total = 0, 0
    for u in p.units:
        oc = p.orc[u]
        X = p.K[u][:600].cpu().to(torch.float64).numpy()
        R = oc.Rk
        exact = X @ R.T
        eps = (D + 2) * 2.0 ** -24 * (np.abs(X) @ np.abs(R).T)
        lo, hi = O.bf16_round(exact - eps), O.bf16_round(exact + eps)
        wk = bits(p.mk.unit_views(*u)["win_k"])
        for pos in oc.window_positions():
            got = O.bits_to_value(wk[(pos - 4) % case.window])
            assert np.all((got >= lo[pos]) & (got <= hi[pos])), pos
            flips += int(np.sum(got != oc.Kr[pos]))
            total += 128
    assert flips <= 0.05 * total


@pytest.mark.parametrize("G,topk_fixed,retain,meta_c", [(4, 0, 100, 0), (1, 64, 0, 0), (8, 0, 300, 0),
                                                       (4, 0, 100, 32), (2, 0, 100, 48)])
def test_block_select_scores_and_ids(G, topk_fixed, retain, meta_c):
    case = Case(n_q=G * 2, n_kv=2, seq_lens=[4096, 2500], rot="perm", topk_fixed=topk_fixed,
                retain_permille=retain, steps=[1, 1, 3], seed=5 + G, meta_channels=meta_c)
    p = Pair(case)
    p.run_steps()
    q = p.query(1)
    nblk_cap = p.mk.nblk_cap
    scores = torch.full((2, 2, nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.block_select(0, [0, 1], q, scores=scores)
    torch.cuda.synchronize()
    ids, n_sel, scores = ids.cpu().numpy(), n_sel.cpu().numpy(), scores.cpu().numpy()
    near_ties = 0
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        per, grp = oc.scores(qs)
        nb = oc.n_blocks_mid()
        got_s = scores[s, h, :nb].astype(np.float64)
        mn, mx = oc.score_keys()
        tol = score_tolerance(oc.rotate_query(qs), mn, mx)
        assert np.all(np.abs(got_s - grp) <= tol)
        cand = oc.candidates()
        k = O.n_select(len(cand), oc.st)
        assert n_sel[s, h] == k
        got_ids = ids[s, h, :k]
        # bit-exact: the kernel's ids are the top-k of the kernel's own scores
        assert np.array_equal(got_ids, O.topk_blocks(got_s, cand, k))
        want_ids, _ = oc.select(qs)
        if not np.array_equal(got_ids, want_ids):
            srt = np.sort(grp[cand])[::-1]
            assert k < len(cand) and srt[k - 1] - srt[k] <= 2 * tol.max()
            near_ties += 1
    assert near_ties <= 1


@pytest.mark.parametrize("T,retain,segments", [
    (480_000, 100, [(0, 32, 0)]),                # ~30K blocks: keys staged, in-bin list too long
    (720_000, 50, [(0, 32, 0)]),                 # ~45K blocks: keys read from global memory
    (200_000, 100, [(0, 32, 0), (500, 16, 1)]),  # always-attended second half: not candidates
])
def test_block_select_all_ties_large(T, retain, segments):
    """Every token carries the same key, so every candidate block has the same
    score and the top-k is the k lowest candidate ids (ties go to the lower id)."""
    from compressed_kv_cache_vector_gb300 import synth
    from tests.harness import signed_permutation
    S, W, B, G = 4, 64, 16, 4
    st = O.Strategy(S, W, B, list(segments), 0, retain)
    cfg = make_config(G, 1, 1, 1, T + 1, S, W, B, segments, 0, retain)
    mk = MosaicKV(cfg, "cuda")
    Rk, Rv = signed_permutation(31), signed_permutation(37)
    mk.set_rotation(0, 0, 0, Rk.astype(np.float32), Rv.astype(np.float32))
    rows = synth.lowrank_outlier(64, D, 0.9, 123, device="cuda")
    k_row, v_row = rows[5:6], rows[9:10]
    mk.append(0, [0], [T], k_row.expand(T, D).reshape(T, 1, D).contiguous(),
              v_row.expand(T, D).reshape(T, 1, D).contiguous())
    q = synth.query(1, G, D, 77, device="cuda")
    scores = torch.full((1, 1, mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = mk.block_select(0, [0], q, scores=scores)
    torch.cuda.synchronize()
    assert mk.poll_error()[0] == 0
    # The oracle's score of one such block, from a short cache of the same tokens.
    Ts = S + W + 3 * B
    oc = O.OracleCache(O.Strategy(S, W, B, [(0, 32, 0)], 0, retain), Ts)
    oc.set_rotation(Rk, Rv)
    oc.append(synth.bf16_values(k_row.expand(Ts, D)), synth.bf16_values(v_row.expand(Ts, D)))
    qs = q[0].cpu().to(torch.float64).numpy()
    _, grp = oc.scores(qs)
    mn, mx = oc.meta()
    tol = score_tolerance(oc.rotate_query(qs), mn, mx)
    assert np.all(grp == grp[0])
    # The long cache's candidates and k, from the oracle's segment rules.
    nb = O.n_middle_blocks(T, st)
    firsts = O.segment_first_blocks(T, st)
    cand = np.array([b for b in range(nb) if not st.segments[O.block_segment(b, firsts)][2]], dtype=np.int64)
    k = O.n_select(len(cand), st)
    got_s = scores[0, 0, :nb].cpu().numpy().astype(np.float64)
    assert np.all(got_s[cand] == got_s[cand[0]])
    assert abs(got_s[cand[0]] - grp[0]) <= tol[0]
    assert int(n_sel[0, 0]) == k
    want = O.topk_blocks(np.full(nb, grp[0]), cand, k)
    assert np.array_equal(ids[0, 0, :k].cpu().numpy(), want)


@pytest.mark.parametrize("case", [
    Case(n_q=4, n_kv=2, seq_lens=[2048, 700], rot="eigh", steps=[1] * 5 + [40], seed=11),
    Case(n_q=8, n_kv=1, seq_lens=[5000], rot="eigh", block=64, window=256, segments=[(0, 38, 0)],
         retain_permille=50, steps=[1, 1], seed=12),
    Case(n_q=4, n_kv=1, seq_lens=[4000, 1200, 300], rot="eigh", block=16, window=128,
         segments=[(0, 32, 0), (350, 64, 1), (650, 32, 0)], steps=[1, 2], seed=13),
    Case(n_q=1, n_kv=1, seq_lens=[4096], rot="eigh", window=64, topk_fixed=64, retain_permille=0,
         segments=[(0, 32, 0)], seed=14),
    Case(n_q=4, n_kv=1, seq_lens=[40], rot="eigh", window=64, seed=15),          # empty middle
    Case(n_q=2, n_kv=1, seq_lens=[3], rot="eigh", n_sink=4, window=8, seed=16),  # T < S
    Case(n_q=4, n_kv=2, seq_lens=[3000], rot="eigh", block=32, segments=[(0, 38, 0, 96)], steps=[1, 1, 2],
         seed=18),                                                                 # bottom 25% truncated
    Case(n_q=4, n_kv=2, seq_lens=[3000], rot="eigh", block=32, meta_channels=32, steps=[1, 1, 2],
         seed=20),                                                                 # compressed block keys
    Case(n_q=4, n_kv=1, seq_lens=[42000], rot="eigh", block=64, window=128, topk_fixed=600, retain_permille=0,
         steps=[1, 1], seed=19),                                                   # long selection: 16-warp plan
    Case(n_q=4, n_kv=1, seq_lens=[1500], rot="eigh", segments=[(0, 128, 0)], topk_fixed=10 ** 6,
         retain_permille=0, seed=17),                                              # r = d, all blocks
], ids=["gqa4-2seq", "b64-5pct", "serving-segments", "single-head-c1", "empty-middle", "below-sinks", "truncated-96", "keys-32ch", "long-16warps",
        "r128-allblocks"])
def test_decode_attention_matches_oracle(case):
    p = Pair(case)
    p.run_steps()
    q = p.query(2)
    seqs = list(range(len(case.seq_lens)))
    ids, n_sel = p.mk.block_select(0, seqs, q)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    out = out.cpu().to(torch.float64).numpy()
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    G = case.G
    worst = 0.0
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        got_ids = ids[s, h, :n_sel[s, h]]
        want = oc.attention(qs, got_ids)
        for g in range(G):
            e = rel_l2(out[s, h * G + g], want[g])
            worst = max(worst, e)
            assert e <= ATOL_REL, (s, h, g, e)
    print("worst relative L2", worst)


def test_swap_closed_segment_with_host_repack():
    """[S] sec. 5.4: the CPU re-compresses a closed segment exactly, here under
    a new strategy (r 32 -> 20, bottom 32 channels truncated), and the result
    replaces the GPU's version while decoding goes on.  The cache then equals,
    byte for byte, the oracle built with the new strategy from the start, and
    attention follows it."""
    import dataclasses
    from compressed_kv_cache_vector_gb300 import binding
    case = Case(n_q=4, n_kv=2, seq_lens=[3000, 1800], rot="perm", block=32, window=64,
                segments=[(0, 32, 0), (600, 32, 0)], steps=[1] * 7, seed=31)
    p = Pair(case)
    for n in case.steps[:6]:
        p.step(n)
    S, B = case.n_sink, case.block
    for (l, s, h) in p.units:
        lay = p.mk.layout(l, s, h)
        fb = lay["seg_first_block"]
        rows = slice(S + fb[0] * B, S + fb[1] * B)
        Rk, Rv = p.R[(l, s, h)]
        pages, meta, _ = binding.host_pack_blocks(Rk, Rv, p.K[(l, s, h)][rows].cpu(), p.V[(l, s, h)][rows].cpu(),
                                                  B, 20, 96, lay["page_stride"])
        p.mk.swap_segment(l, s, h, 0, 20, 96, pages, meta)
        torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    # The oracle of the new strategy, fed the same tokens.
    case2 = dataclasses.replace(case, segments=[(0, 20, 0, 96), (600, 32, 0)])
    ref = Pair(case2)
    for n in case2.steps[:6]:
        ref.step(n)
    p.c, p.orc = case2, ref.orc
    for u in p.units:
        _check_storage(p, u)
    # Decoding goes on (the open segment is untouched; p.step also advances
    # the oracle, now ref's), then attention.
    p.step(case.steps[6])
    for u in p.units:
        _check_storage(p, u)
    q = p.query(5)
    ids, n_sel = p.mk.block_select(0, [0, 1], q)
    out = p.mk.decode_attn(0, [0, 1], ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    out = out.cpu().to(torch.float64).numpy()
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    G = case.G
    for (l, s, h), oc in ref.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        want = oc.attention(qs, ids[s, h, :n_sel[s, h]])
        for g in range(G):
            assert rel_l2(out[s, h * G + g], want[g]) <= ATOL_REL


def test_swap_segment_refuses_open_or_bad_segments():
    from compressed_kv_cache_vector_gb300 import binding
    case = Case(n_q=4, n_kv=1, seq_lens=[2000], rot="perm", block=32, segments=[(0, 32, 0), (600, 32, 0)], seed=32)
    p = Pair(case)
    lay = p.mk.layout(0, 0, 0)
    pages = np.zeros((1, lay["page_stride"]), dtype=np.uint8)
    meta = np.zeros((1, 2, 128), dtype=np.uint16)
    for seg, r, keep in ((1, 20, 0), (0, 40, 0), (0, 20, 10), (2, 20, 0)):
        with pytest.raises(binding.MosaicKVError):
            p.mk.swap_segment(0, 0, 0, seg, r, keep, pages, meta)   # open segment, r above r_max, keep < r, no such
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)


@pytest.mark.parametrize("topk_fixed,retain", [(0, 100), (2100, 0)], ids=["12-warp-plan", "16-warp-plan"])
def test_dense_reference_attention(topk_fixed, retain):
    # The second configuration's longest selection (2100 blocks of 16 tokens)
    # picks the 16-warp, one-stage plan for the context, the reference too.
    torch.manual_seed(0)
    n, Hkv, G, T = 2, 2, 4, 3000
    cfg = make_config(Hkv * G, Hkv, 1, n, 40000, 4, 64, 16, [(0, 32, 0)], topk_fixed, retain)
    mk = MosaicKV(cfg)
    K = torch.randn(n, Hkv, T, 128, device="cuda").to(torch.bfloat16)
    V = torch.randn(n, Hkv, T, 128, device="cuda").to(torch.bfloat16)
    q = torch.randn(n, Hkv * G, 128, device="cuda").to(torch.bfloat16)
    lens = [T, 1777]
    out = mk.dense_attn(lens, q, K, V).cpu().to(torch.float64).numpy()
    for s in range(n):
        for h in range(Hkv):
            Kn = K[s, h, :lens[s]].cpu().to(torch.float64).numpy()
            Vn = V[s, h, :lens[s]].cpu().to(torch.float64).numpy()
            qn = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
            want = O.dense_attention(qn, Kn, Vn)
            for g in range(G):
                assert rel_l2(out[s, h * G + g], want[g]) <= ATOL_REL


def test_gram_and_host_rotation():
    from compressed_kv_cache_vector_gb300 import binding, synth
    x = synth.lowrank_outlier(5000, 128, 0.9, 99, device="cuda")
    G = binding.gram(x, 5000, 128).cpu().numpy().astype(np.float64)
    X = synth.bf16_values(x)
    want = X.T @ X
    assert np.max(np.abs(G - want)) <= 1e-5 * np.abs(want).max()
    R = binding.rotation_from_gram(G)
    Ro, lam = O.rotation_from_keys(X)
    # same principal directions up to sign for well-separated eigenvalues
    for i in range(8):
        assert abs(abs(float(R[i] @ Ro[i])) - 1.0) < 1e-3


def test_host_errors_leave_state_unchanged():
    case = Case(n_q=4, n_kv=1, seq_lens=[200], rot="perm", window=32, seed=21)
    p = Pair(case)
    mk = p.mk
    k = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MosaicKVError) as e:
        mk.append(0, [0, 0], [1, 1], k, k)                  # duplicate sequence
    assert e.value.status == 1
    with pytest.raises(MosaicKVError) as e:
        mk.append(0, [0], [10 ** 6], k, k)                  # past capacity
    assert e.value.status == 2
    q = p.query(3)
    ids, n_sel = mk.alloc_select(1)
    out = torch.empty(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    # attention before any selection on this layer
    with pytest.raises(MosaicKVError) as e:
        mk.decode_attn(0, [0], ids, n_sel, out)
    assert e.value.status == 3
    assert mk.seq_length(0, 0) == 200
    mk.block_select(0, [0], q, ids, n_sel)
    mk.decode_attn(0, [0], ids, n_sel, out)
    torch.cuda.synchronize()
    assert mk.poll_error() == (0, 0)


def test_device_error_word_on_bad_block_id():
    # A corrupted ids row (out-of-range block) is caught by the kernel's own
    # bounds check: it sets the error word and skips the page (no fault).
    case = Case(n_q=4, n_kv=1, seq_lens=[800], rot="perm", window=32, seed=22)
    p = Pair(case)
    q = p.query(4)
    ids, n_sel = p.mk.block_select(0, [0], q)
    ids[0, 0, 0] = 10 ** 6
    p.mk.decode_attn(0, [0], ids, n_sel)
    st, detail = p.mk.poll_error()
    assert st == 5 and detail == 2
    p.mk.clear_error()
    assert p.mk.poll_error() == (0, 0)


def test_repeatable_bytes():
    outs = []
    for _ in range(2):
        case = Case(n_q=4, n_kv=2, seq_lens=[1500], rot="eigh", steps=[1, 1], seed=23)
        p = Pair(case)
        p.run_steps()
        q = p.query(5)
        ids, n_sel = p.mk.block_select(0, [0], q)
        out = p.mk.decode_attn(0, [0], ids, n_sel)
        outs.append(bits(out))
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("case", [
    Case(n_q=8, n_kv=2, seq_lens=[3000, 700], rot="eigh", oracle_units=[], seed=21),
    Case(n_q=4, n_kv=1, seq_lens=[4000, 1200, 300], rot="eigh", block=16, window=128,
         segments=[(0, 32, 0), (350, 64, 1), (650, 32, 0)], oracle_units=[], seed=22),
    Case(n_q=4, n_kv=2, seq_lens=[40, 70], rot="eigh", window=64, oracle_units=[], seed=23),
    Case(n_q=4, n_kv=2, seq_lens=[2500, 900], rot="eigh", block=32, meta_channels=24, oracle_units=[], seed=24),
], ids=["gqa4-2seq", "serving-segments", "filling-window", "keys-24ch"])
def test_append_select_equals_separate_calls(case):
    """The fused decode append + block selection gives the ids, the stored
    state and the attention output of the two calls it replaces, step after
    step (evicted tokens cross block boundaries and fill partial blocks)."""
    n_steps = 40
    case.steps = [1] * n_steps
    a, b = Pair(case), Pair(case)
    seqs = list(range(len(case.seq_lens)))
    for step in range(n_steps):
        rows = [torch.stack([a.K[(0, s, h)][a.T[s]] for h in range(case.n_kv)]) for s in seqs]
        k = torch.stack(rows).contiguous()
        v = torch.stack([torch.stack([a.V[(0, s, h)][a.T[s]] for h in range(case.n_kv)]) for s in seqs]).contiguous()
        q = a.query(100 + step)
        a.mk.append(0, seqs, [1] * len(seqs), k, v)
        ids_a, ns_a = a.mk.block_select(0, seqs, q)
        ids_b, ns_b = b.mk.append_select(0, seqs, k, v, q)
        out_a = a.mk.decode_attn(0, seqs, ids_a, ns_a)
        out_b = b.mk.decode_attn(0, seqs, ids_b, ns_b)
        torch.cuda.synchronize()
        for s in seqs:
            a.T[s] += 1
        ns = ns_a.cpu().numpy()
        assert np.array_equal(ns, ns_b.cpu().numpy()), step
        ia, ib = ids_a.cpu().numpy(), ids_b.cpu().numpy()
        for s in seqs:
            for h in range(case.n_kv):
                assert np.array_equal(ia[s, h, :ns[s, h]], ib[s, h, :ns[s, h]]), (step, s, h)
        assert np.array_equal(bits(out_a), bits(out_b)), step
    assert a.mk.poll_error() == (0, 0) and b.mk.poll_error() == (0, 0)
    a.mk.sync_state()
    b.mk.sync_state()
    for s in seqs:
        T = a.mk.seq_length(0, s)
        assert T == b.mk.seq_length(0, s) == case.seq_lens[s] + n_steps
        for h in range(case.n_kv):
            va, vb = a.mk.unit_views(0, s, h), b.mk.unit_views(0, s, h)
            L = va["layout"]
            S, W, B = case.n_sink, case.window, case.block
            n_sink = min(S, T)
            if n_sink:
                assert np.array_equal(bits(va["sink_k"])[:n_sink], bits(vb["sink_k"])[:n_sink])
            for p in range(max(S, T - W), T):
                sl = (p - S) % W
                assert np.array_equal(bits(va["win_k"])[sl], bits(vb["win_k"])[sl]), p
                assert np.array_equal(bits(va["win_v"])[sl], bits(vb["win_v"])[sl]), p
            mid = max(0, T - S - W)
            nb = (mid + B - 1) // B
            assert np.array_equal(bits(va["meta"])[:nb], bits(vb["meta"])[:nb])
            pa, pb = va["pages"].cpu().numpy(), vb["pages"].cpu().numpy()
            for blk in range(nb):
                seg = [i for i, f in enumerate(L["seg_first_block"]) if blk >= f][-1]
                r = case.segments[seg][1]
                n_live = min(B, mid - blk * B)
                for g, w_ in zip(page_rows(pa[blk], B, r, n_live), page_rows(pb[blk], B, r, n_live)):
                    assert np.array_equal(g, w_), (s, h, blk)


@pytest.mark.parametrize("segments,swaps", [
    ([(0, 32, 0), (600, 32, 0)], [(0, 20, 96)]),
    ([(0, 32, 0), (350, 64, 1), (650, 32, 0)], [(0, 24, 0), (1, 48, 0)]),
], ids=["scored-segment", "scored-and-always-segments"])
def test_swap_segments_under_their_own_rotation(segments, swaps):
    """[S] sec. 5.4 with the per-segment SVD of [N] Fig. 4: closed segments
    re-compressed on the host under their own rotations (eigenvectors of the
    segment's own K^T K and V^T V) and a new r replace the GPU's version.  The
    stored bytes then equal the oracle's re-compression; the scores use the
    query rotated into each block's basis, and attention un-rotates each
    basis's values by its own R_v (each rotation gets its own CTAs)."""
    from compressed_kv_cache_vector_gb300 import binding, synth
    # Head rotations exact in bf16 (signed permutations), so the GPU-rotated
    # rows match the oracle bit for bit; the segments' own rotations are
    # general (eigenvectors), packed exactly on the host as the oracle does.
    case = Case(n_q=4, n_kv=2, seq_lens=[3000, 1800], rot="perm", block=32, window=64, segments=segments,
                steps=[1] * 4, seed=41)
    p = Pair(case)
    for n in case.steps[:3]:
        p.step(n)
    S, B = case.n_sink, case.block
    for (l, s, h) in p.units:
        lay = p.mk.layout(l, s, h)
        fb = lay["seg_first_block"]
        Kraw = synth.bf16_values(p.K[(l, s, h)])
        Vraw = synth.bf16_values(p.V[(l, s, h)])
        for seg, r_new, keep in swaps:
            rows = slice(S + fb[seg] * B, S + fb[seg + 1] * B)
            Rk_s = O.rotation_from_keys(Kraw[rows])[0].astype(np.float32)
            Rv_s = O.rotation_from_keys(Vraw[rows])[0].astype(np.float32)
            pages, meta, _ = binding.host_pack_blocks(Rk_s, Rv_s, p.K[(l, s, h)][rows].cpu(),
                                                      p.V[(l, s, h)][rows].cpu(), B, r_new, keep, lay["page_stride"])
            p.mk.swap_segment(l, s, h, seg, r_new, keep, pages, meta, R_k=Rk_s, R_v=Rv_s)
            torch.cuda.synchronize()
            p.orc[(l, s, h)].recompress_segment(seg, Kraw, Vraw, r_new, keep, Rk_s.astype(np.float64),
                                                Rv_s.astype(np.float64))
    assert p.mk.poll_error() == (0, 0)
    for u in p.units:
        _check_storage(p, u)
    # one more decode step through the fused call, then select and attend
    seqs = [0, 1]
    k = torch.stack([torch.stack([p.K[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
    v = torch.stack([torch.stack([p.V[(0, s, h)][p.T[s]] for h in range(2)]) for s in seqs]).contiguous()
    q = p.query(9)
    p.mk.append_select(0, seqs, k, v, q)
    for (l, s, h), oc in p.orc.items():
        t = p.T[s]
        oc.append(synth.bf16_values(p.K[(l, s, h)][t:t + 1]), synth.bf16_values(p.V[(l, s, h)][t:t + 1]))
    for s in seqs:
        p.T[s] += 1
    q = p.query(10)
    scores = torch.full((2, 2, p.mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.block_select(0, seqs, q, scores=scores)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    out, scores = out.cpu().to(torch.float64).numpy(), scores.cpu().numpy()
    G = case.G
    near = 0
    for (l, s, h), oc in p.orc.items():
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        cand = oc.candidates()
        kk = O.n_select(len(cand), oc.st)
        assert n_sel[s, h] == kk
        per, grp = oc.scores(qs)
        mn, mx = oc.score_keys()
        nb = oc.n_blocks_mid()
        tol = np.zeros(nb)
        for b in range(nb):   # the fp32 bound of each block in its own basis
            Rq = oc.rotations_of_block(b)[0]
            tol[b] = score_tolerance(qs @ Rq.T, mn[b:b + 1], mx[b:b + 1])[0]
        got_s = scores[s, h, :nb].astype(np.float64)
        assert np.all(np.abs(got_s[cand] - grp[cand]) <= tol[cand]), (s, h)
        got_ids = ids[s, h, :kk]
        assert np.array_equal(got_ids, O.topk_blocks(got_s, cand, kk))
        want_ids, _ = oc.select(qs)
        if not np.array_equal(got_ids, want_ids):
            srt = np.sort(grp[cand])[::-1]
            assert srt[kk - 1] - srt[kk] <= 2 * tol.max()
            near += 1
        want = oc.attention(qs, got_ids)
        for g in range(G):
            assert rel_l2(out[s, h * G + g], want[g]) <= ATOL_REL, (s, h, g)
    assert near <= 1

