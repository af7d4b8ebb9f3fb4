"""Memory-safety checks on the GPU, in place of a memory checker.

* The checked build (libmosaickv_checks.so: every kernel's bounds checks
  compiled in; a failed check records its site and index in the error word
  and skips the access) runs the parity suites and the random sweep.  Those
  suites assert a clean error word after every call, so a check that fires
  fails them; their results are compared with the oracle as in the default
  build.
* mk_swap_segment checks the positions of the pages it is given before any
  copy, since the attention trusts them.
"""
import os
import re
import subprocess
import sys

import numpy as np
import pytest
import torch

from compressed_kv_cache_vector_gb300 import build as Bld

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_bitmap.py", "tests/test_gpu_retention.py",
          "tests/test_gpu_quest.py", "tests/test_gpu_fuzz.py"]


def test_checked_build_runs_the_parity_suites_clean():
    lib = Bld.build(checks=True)
    env = dict(os.environ, MOSAICKV_LIB=lib)
    probe = subprocess.run([sys.executable, "-c", "from compressed_kv_cache_vector_gb300 import binding as b; "
                            "b.load(); print(b.LIB_PATH)"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == lib, probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 60, r.stdout[-2000:]     # the suites ran (about 70 tests)
    print(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("fmt", ["uint8", "bitmap"])
def test_swap_refuses_pages_with_bad_positions(fmt):
    from compressed_kv_cache_vector_gb300 import binding
    from tests.harness import Case, Pair
    g = 4 if fmt == "bitmap" else 0
    case = Case(n_q=4, n_kv=1, seq_lens=[1500], rot="perm", block=16, window=64, segments=[(0, 32, 0), (600, 32, 0)],
                page_format=2 if g else 0, elem_group=g, seed=140)
    p = Pair(case)
    lay = p.mk.layout(0, 0, 0)
    fb = lay["seg_first_block"]
    n = fb[1] - fb[0]
    S, B = case.n_sink, case.block
    rows = slice(S + fb[0] * B, S + fb[1] * B)
    Rk, Rv = p.R[(0, 0, 0)]
    pages, meta, _ = binding.host_pack_blocks(Rk, Rv, p.K[(0, 0, 0)][rows].cpu(), p.V[(0, 0, 0)][rows].cpu(), B, 32, 0,
                                              lay["page_stride"], 0, 2 if g else 0, g)
    before = p.mk.unit_views(0, 0, 0)["pages"].cpu().numpy().copy()
    bad = pages.copy()
    Br = B * 32
    if g:
        bad[n - 1, 2 * Br + 3] ^= 0x10          # one bitmap row with one bit too many or too few
    else:
        bad[n - 1, 2 * Br + 5] = 200            # an index past the head dimension
    with pytest.raises(binding.MosaicKVError) as e:
        p.mk.swap_segment(0, 0, 0, 0, 32, 0, bad, meta)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert np.array_equal(p.mk.unit_views(0, 0, 0)["pages"].cpu().numpy(), before)   # nothing copied
    p.mk.swap_segment(0, 0, 0, 0, 32, 0, pages, meta)                                  # the packer's own pages pass
    torch.cuda.synchronize()
    assert p.mk.poll_error() == (0, 0)
