"""The allocation-free decode attention entry point (GPU).

mk_dense_decode_attn_noalloc serves callers that cannot allocate device memory
where they run attention (a plugin whose host framework forbids allocation
while it enqueues work, a runtime whose memory plan is fixed before serving
starts), so they cannot hand the library a workspace: its scratch is a static
device array inside the library.  This file runs last (pytest collects it
after the others).  On two calls in a row, with different inputs, it checks
the new entry point bit for bit against the workspace-based
mk_dense_decode_attn (the same kernel with the same split), and against the
fp64 oracle's dense attention within the relative L2 tolerance of the other
attention tests, for every GQA group size and at the size limit.  It also
checks that an oversized call is refused and that the device-side error word
reads clean.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import binding
from compressed_kv_cache_vector_gb300.build import build
from oracle import mosaickv_oracle as O

pytestmark = pytest.mark.gpu
TOL = 5e-3
MAX_Q = 128            # MK_NOALLOC_MAX_QUERY_HEADS


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("n,Hkv,G,t_stride,lens", [
    (2, 8, 4, 6000, ([6000, 3111], [17, 5000])),
    (16, 8, 1, 700, ([700] * 16, [1 + 41 * i for i in range(16)])),    # 128 query heads: the limit
    (3, 4, 2, 2500, ([2500, 1, 999], [64, 2500, 1700])),
    (1, 16, 8, 4100, ([4100], [333])),                                  # 128 query heads at G = 8
])
def test_noalloc_matches_workspace_entry_point_and_oracle(n, Hkv, G, t_stride, lens):
    build()
    Hq = Hkv * G
    assert n * Hq <= MAX_Q
    cfg = binding.make_config(Hq, Hkv, 1, n, t_stride, 4, 64, 16, [(0, 32, 0)], 0, 100)
    mk = binding.MosaicKV(cfg)
    g = torch.Generator(device="cuda")
    rng = np.random.default_rng(n * 100 + G)
    for call, T in enumerate(lens):
        g.manual_seed(1000 * G + call)
        K = torch.randn(n, Hkv, t_stride, 128, generator=g, device="cuda").to(torch.bfloat16)
        V = torch.randn(n, Hkv, t_stride, 128, generator=g, device="cuda").to(torch.bfloat16)
        q = torch.randn(n, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
        want = mk.dense_attn(T, q, K, V)
        got = torch.full_like(want, float("nan"))
        binding.dense_attn_noalloc(Hq, Hkv, T, q, K, V, got)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), call
        # oracle: [N] Eq. (1) in fp64 on a few (sequence, kv head) pairs
        for s, h in {(int(rng.integers(n)), int(rng.integers(Hkv))) for _ in range(3)}:
            Kh = K[s, h, :T[s]].double().cpu().numpy()
            Vh = V[s, h, :T[s]].double().cpu().numpy()
            qh = q[s, h * G:(h + 1) * G].double().cpu().numpy()
            ref = O.dense_attention(qh, Kh, Vh)
            out = got[s, h * G:(h + 1) * G].double().cpu().numpy()
            for j in range(G):
                assert _rel(out[j], ref[j]) <= TOL, (call, s, h, j)
    assert binding.noalloc_poll_error() == (0, 0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build()
    n, Hkv, G = 5, 8, 4            # 160 query heads: more than the scratch holds
    K = torch.zeros(n, Hkv, 32, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(n, Hkv * G, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(binding.MosaicKVError) as e:
        binding.dense_attn_noalloc(Hkv * G, Hkv, [32] * n, q, K, K, out)
    assert e.value.status == 2
    # a misaligned (odd-offset) view is refused before any launch
    flat = torch.zeros(Hkv * 32 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    Kodd = flat[1:1 + Hkv * 32 * 128].view(1, Hkv, 32, 128)
    with pytest.raises(binding.MosaicKVError) as e:
        binding.dense_attn_noalloc(Hkv * G, Hkv, [32], q[:1], Kodd, Kodd, out[:1])
    assert e.value.status == 1
    assert binding.noalloc_poll_error() == (0, 0)
