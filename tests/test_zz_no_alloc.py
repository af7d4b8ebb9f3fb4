"""The allocation-free decode attention entry point (GPU).

mk_dense_decode_attn_noalloc serves callers that cannot allocate device memory
where they run attention, so they cannot hand the library a workspace: its
scratch is a static device array inside the library.  This file runs last
(pytest collects it after the others) and checks the new entry point against
the workspace-based mk_dense_decode_attn on two calls in a row, with
different inputs each time, within the relative L2 tolerance of the other
attention tests.  It also checks that an oversized call is refused.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import binding
from compressed_kv_cache_vector_gb300.build import build

pytestmark = pytest.mark.gpu
TOL = 5e-3


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    build()
    n, Hkv, G, t_stride = 2, 8, 4, 6000
    cfg = binding.make_config(Hkv * G, Hkv, 1, n, t_stride, 4, 64, 16, [(0, 32, 0)], 0, 100)
    mk = binding.MosaicKV(cfg)
    g = torch.Generator(device="cuda")
    for call, lens in enumerate(([6000, 3111], [17, 5000])):
        g.manual_seed(100 + call)
        K = torch.randn(n, Hkv, t_stride, 128, generator=g, device="cuda").to(torch.bfloat16)
        V = torch.randn(n, Hkv, t_stride, 128, generator=g, device="cuda").to(torch.bfloat16)
        q = torch.randn(n, Hkv * G, 128, generator=g, device="cuda").to(torch.bfloat16)
        want = mk.dense_attn(lens, q, K, V)
        got = torch.full_like(want, float("nan"))
        binding.dense_attn_noalloc(Hkv * G, Hkv, lens, q, K, V, got)
        torch.cuda.synchronize()
        for s in range(n):
            for h in range(Hkv * G):
                assert _rel(got[s, h], want[s, h]) <= TOL, (call, s, h)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build()
    n, Hkv, G = 5, 8, 4            # 40 (sequence, kv head) pairs at G = 4: more than fits
    K = torch.zeros(n, Hkv, 32, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(n, Hkv * G, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(binding.MosaicKVError) as e:
        binding.dense_attn_noalloc(Hkv * G, Hkv, [32] * n, q, K, K, out)
    assert e.value.status == 2
