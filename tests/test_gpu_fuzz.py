"""A seeded sweep of random configurations, each checked against the fp64
oracle through the C ABI.

Every case draws its GQA group, block size, sinks and window, one to three
strategy segments (r, always-attended, truncation, per-segment element-group
size and retention), the page format (uint8 indices or bitmaps), compressed
block keys, two sequences' lengths and a few decode appends.  Rotations are
signed permutations (exact in bf16), so the stored sinks, window, block keys
and pages must equal the oracle's byte for byte; the ids must be the top-k of
the kernel's own scores (per segment where the segments give their own
retention); attention per head within 5e-3 relative L2.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import build as Bld
from oracle import mosaickv_oracle as O
from tests.harness import Case, Pair, check_storage, rel_l2

pytestmark = pytest.mark.gpu
ATOL_REL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    Bld.build()


def _draw(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 8]))
    n_kv = int(rng.choice([1, 2]))
    block = int(rng.choice([16, 32, 64]))
    fmt = int(rng.choice([0, 2]))
    g_cache = int(rng.choice([1, 2, 4, 8])) if fmt == 2 else 0
    per_seg_ret = bool(rng.random() < 0.4)
    n_seg = int(rng.integers(1, 4))
    begins = sorted(int(b) for b in rng.choice(np.arange(100, 900, 50), size=n_seg - 1, replace=False))
    segs = []
    for i, b in enumerate([0] + begins):
        g = int(rng.choice([0, 1, 2, 4, 8])) if fmt == 2 else 0
        gg = (g or g_cache) if fmt == 2 else 1
        r = gg * int(rng.integers(max(1, 8 // gg), 96 // gg + 1))
        keep = int(rng.choice([0, 96])) if r <= 96 else 0
        always = int(i > 0 and i < n_seg - 1 and rng.random() < 0.4)
        ret = int(rng.choice([30, 100, 250])) if per_seg_ret and not always else 0
        segs.append((b, r, always, keep, g, ret))
    if not any(s[5] for s in segs if not s[2]):
        segs = [s[:5] for s in segs]
    lens = [int(x) for x in rng.integers(300, 5000, size=2)]
    steps = [int(x) for x in rng.choice([1, 1, 1, 3, 17], size=int(rng.integers(1, 4)))]
    return Case(n_q=G * n_kv, n_kv=n_kv, seq_lens=lens, rot="perm", n_sink=int(rng.choice([0, 4])),
                window=int(rng.choice([16, 64, 128])), block=block, segments=segs, retain_permille=100,
                page_format=fmt, elem_group=g_cache, meta_channels=int(rng.choice([0, 0, 24])), steps=steps,
                seed=int(seed))


@pytest.mark.parametrize("seed", list(range(1000, 1016)))
def test_random_configuration_matches_oracle(seed):
    case = _draw(seed)
    p = Pair(case)
    p.run_steps()
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0), case
    for u in p.units:
        check_storage(p, u)
    seqs = [0, 1]
    q = p.query(seed)
    scores = torch.full((2, case.n_kv, p.mk.nblk_cap), float("nan"), dtype=torch.float32, device="cuda")
    ids, n_sel = p.mk.block_select(0, seqs, q, scores=scores)
    out = p.mk.decode_attn(0, seqs, ids, n_sel)
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0), case
    ids, n_sel = ids.cpu().numpy(), n_sel.cpu().numpy()
    scores, out = scores.cpu().numpy(), out.cpu().to(torch.float64).numpy()
    G = case.G
    for (l, s, h), oc in p.orc.items():
        nb = oc.n_blocks_mid()
        got_s = scores[s, h, :nb].astype(np.float64)
        assert n_sel[s, h] == oc.n_selected(), (case, s, h)
        got = ids[s, h, :n_sel[s, h]]
        if oc.st.per_segment_retention():
            parts = [O.topk_blocks(got_s, c, O.n_select(len(c), oc.st, sg[5] or oc.st.retain_permille))
                     for i, sg in enumerate(oc.st.segments) for c in [oc.segment_candidates(i)] if len(c)]
            want = np.sort(np.concatenate(parts)) if parts else np.zeros(0, dtype=np.int64)
        else:
            cand = oc.candidates()
            want = O.topk_blocks(got_s, cand, O.n_select(len(cand), oc.st))
        assert np.array_equal(got, want), (case, s, h)
        qs = q[s, h * G:(h + 1) * G].cpu().to(torch.float64).numpy()
        ref = oc.attention(qs, got)
        for gi in range(G):
            e = rel_l2(out[s, h * G + gi], ref[gi])
            assert e <= ATOL_REL, (case, s, h, gi, e)
