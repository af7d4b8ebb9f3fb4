"""Parity at the shapes the benchmark times (GPU), through the calls it makes.

The benchmark's decode step is mk_append_select (one new token per sequence,
appended and compressed, then block selection: [N] Eq. (9), (12); [S] sec.
4.2) followed by mk_decode_attn ([N] Eq. (13), (14); [S] sec. 5.3).  Here
that same pair of calls runs after a bulk prefill at four workload shapes,
and a few (sequence, kv head) units are followed by the fp64 oracle:

  * the 32K-token layer at batch 4 (block 16, window 128, 10% of blocks);
  * the 128K-token layer (T = 131072, 8 kv heads, GQA 4, r = 38, block 32,
    window 256, 10% of blocks), rotations exact in bf16 (signed permutations)
    so that every stored byte can be compared;
  * one kv head of the 1M-token layer (T = 1048576, block 64, window 512, 5% of
    blocks), with a signed permutation and with rotations from the
    eigenvectors of K^T K (there the scores are checked on the block keys the
    kernel stored, since a general rotation may round a stored value one bf16
    step away from the oracle's);
  * the serving mix: 64 sequences of log-uniform lengths 8K..128K, the middle
    30% kept at r = 64 and attended in full, the rest r = 32 with 10% of blocks.

Bars, per decode step and followed unit: the kernel's scores within the fp32
summation bound of the oracle's; its ids bit-exact against the top-k of its
own scores, and equal to the oracle's own choice except at a near-tie inside
that bound; attention relative L2 error per head <= 5e-3; and, where the
rotation is exact, every stored sink, window, meta and page byte.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import configs, synth
from oracle import mosaickv_oracle as O
from tests.harness import Case, Pair, bits, check_storage, rel_l2, score_tolerance

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


def _fused_steps(p: Pair, n_steps: int):
    """n_steps decode steps through mk_append_select + mk_decode_attn, each
    checked against the oracle units; returns the number of near-ties met."""
    c = p.c
    exact = c.rot != "eigh"
    G = c.G
    seqs = list(range(len(c.seq_lens)))
    scores = torch.empty(len(seqs), c.n_kv, p.mk.nblk_cap, dtype=torch.float32, device="cuda")
    near = 0
    for step in range(n_steps):
        k = torch.stack([torch.stack([p.K[(0, s, h)][p.T[s]] for h in range(c.n_kv)]) for s in seqs]).contiguous()
        v = torch.stack([torch.stack([p.V[(0, s, h)][p.T[s]] for h in range(c.n_kv)]) for s in seqs]).contiguous()
        q = p.query(500 + step)
        scores.fill_(float("nan"))
        ids, n_sel = p.mk.append_select(0, seqs, k, v, q, scores=scores)
        out = p.mk.decode_attn(0, seqs, ids, n_sel)
        torch.cuda.synchronize()
        assert p.mk.poll_error() == (0, 0), step
        for (l, s, h), oc in p.orc.items():
            t = p.T[s]
            oc.append(synth.bf16_values(p.K[(l, s, h)][t:t + 1]), synth.bf16_values(p.V[(l, s, h)][t:t + 1]))
        for s in seqs:
            p.T[s] += 1
        ids_h, ns_h = ids.cpu().numpy(), n_sel.cpu().numpy()
        sc_h, out_h = scores.cpu().numpy(), out.cpu().to(torch.float64).numpy()
        for (l, s, h), oc in p.orc.items():
            qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
            cand = oc.candidates()
            k_ = O.n_select(len(cand), oc.st)
            assert ns_h[s, h] == k_, (step, s, h)
            got_ids = ids_h[s, h, :k_]
            if len(cand):
                nb = oc.n_blocks_mid()
                if exact:
                    mn, mx = oc.score_keys()
                else:
                    # A general rotation rounds a stored value one bf16 step
                    # away from the oracle's now and then, so the kernel's
                    # block keys are scored as stored.
                    meta = O.bits_to_value(bits(p.mk.unit_views(l, s, h)["meta"])[:nb])
                    mn, mx = meta[:, 0], meta[:, 1]
                grp = O.block_scores(oc.rotate_query(qs), mn, mx)[1]
                tol = score_tolerance(oc.rotate_query(qs), mn, mx)
                got_s = sc_h[s, h, :nb].astype(np.float64)
                assert np.all(np.abs(got_s[cand] - grp[cand]) <= tol[cand]), (step, s, h)
                assert np.array_equal(got_ids, O.topk_blocks(got_s, cand, k_)), (step, s, h)
                want_ids = O.topk_blocks(grp, cand, k_)
                if not np.array_equal(got_ids, want_ids):
                    srt = np.sort(grp[cand])[::-1]
                    assert k_ < len(cand) and srt[k_ - 1] - srt[k_] <= 2 * tol.max(), (step, s, h)
                    near += 1
            want = oc.attention(qs, got_ids)
            for g in range(G):
                e = rel_l2(out_h[s, h * G + g], want[g])
                assert e <= ATOL_REL, (step, s, h, g, e)
    return near


def _case_from(wl, **kw):
    base = dict(n_q=wl.n_q_heads, n_kv=wl.n_kv_heads, seq_lens=list(wl.seq_lens), n_sink=wl.n_sink,
                window=wl.window, block=wl.block, segments=list(wl.segments), topk_fixed=wl.topk_fixed,
                retain_permille=wl.retain_permille, decay=wl.decay)
    base.update(kw)
    return Case(**base)


@pytest.mark.parametrize("rot", ["perm", "eigh"])
def test_32k_layer_batch_4_fused_decode_steps(rot):
    # The 32K-token layer at batch 4 (block 16, window 128, 10% of blocks,
    # 2040 blocks and k = 204 per unit), two units of different sequences
    # followed by the oracle.
    wl = configs.get("c2")
    case = _case_from(wl, rot=rot, steps=[1, 1], seed=201, oracle_units=[(0, 1, 2), (0, 3, 7)])
    p = Pair(case)
    assert _fused_steps(p, 2) <= 1
    if rot == "perm":
        for u in p.units:
            check_storage(p, u)


def test_128k_layer_fused_decode_steps():
    wl = configs.get("c3")
    case = _case_from(wl, rot="perm", steps=[1, 1, 1], seed=301, oracle_units=[(0, 0, 0), (0, 0, 5)])
    p = Pair(case)                                  # bulk prefill of the 131072-token layer, all 8 kv heads
    assert _fused_steps(p, 3) <= 1
    for u in p.units:
        check_storage(p, u)
    p.mk.sync_state()
    assert p.mk.seq_length(0, 0) == 131072 + 3


@pytest.mark.parametrize("rot", ["perm", "eigh"])
def test_1m_layer_one_kv_head_fused_decode_steps(rot):
    wl = configs.get("c4")
    case = _case_from(wl, n_q=wl.group, n_kv=1, rot=rot, steps=[1, 1], seed=401)
    p = Pair(case)                                  # T = 1048576, 16376 middle blocks, k = 819
    assert p.mk.nblk_cap >= 16376
    assert _fused_steps(p, 2) <= 1
    if rot == "perm":
        check_storage(p, p.units[0])


def test_serving_mix_64_sequences_fused_decode_steps():
    wl = configs.get("c5")
    lens = list(wl.seq_lens)
    order = np.argsort(lens, kind="stable")
    follow = [int(order[0]), int(order[21]), int(order[42]), int(order[-1])]   # across the length range
    case = _case_from(wl, rot="perm", steps=[1, 1], seed=501, oracle_units=[(0, s, s % 8) for s in follow])
    p = Pair(case)
    assert len(lens) == 64 and min(lens) >= 8192 and max(lens) <= 131072
    assert _fused_steps(p, 2) <= 1
    for u in p.units:
        check_storage(p, u)
