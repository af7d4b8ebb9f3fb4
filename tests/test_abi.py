"""The C ABI library builds, loads and exports what include/mosaickv.h declares.

CPU only: the calls made here do no device work (size queries, status text,
configuration checks).
"""
import ctypes

import pytest

from compressed_kv_cache_vector_gb300 import build as B
from compressed_kv_cache_vector_gb300 import binding as K


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.load()


def test_exports_every_declared_symbol(lib):
    names = K.header_symbols()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert set(K._SIGS) | {"mk_status_str"} == set(names)


def test_status_strings(lib):
    assert lib.mk_status_str(0) == b"ok"
    assert lib.mk_status_str(2).startswith(b"buffer too small")


def _cfg(**kw):
    base = dict(n_q_heads=32, n_kv_heads=8, n_layers=1, max_seqs=1, max_tokens=131072 + 64,
                n_sink=4, window=256, block=32, segments=[(0, 38, 0)], retain_permille=100)
    base.update(kw)
    return K.make_config(**base)


def test_sizes_follow_the_layout(lib):
    a, w, k = K.sizes(_cfg())
    nblk = (131072 + 64 - 4 - 256 + 31) // 32
    assert k == (100 * nblk + 999) // 1000
    per_unit_pages = nblk * 6 * 32 * 38
    assert a > 8 * per_unit_pages and a < 8 * per_unit_pages * 1.5
    # the 1M configuration: about 1.8 GB of packed pages per layer
    a4, _, k4 = K.sizes(_cfg(max_tokens=1048576, window=512, block=64, retain_permille=50))
    assert 1.9e9 < a4 < 2.2e9 and k4 == 819


@pytest.mark.parametrize("bad", [
    dict(block=24), dict(n_q_heads=24), dict(segments=[(100, 38, 0)]), dict(segments=[(0, 0, 0)]),
    dict(segments=[(0, 129, 0)]), dict(retain_permille=0), dict(window=0),
    dict(segments=[(0, 32, 0), (500, 64, 1), (400, 32, 0)]),
    dict(segments=[(0, 38, 0, 30)]), dict(segments=[(0, 38, 0, 129)]),   # truncation below r, above d
    dict(meta_channels=-1), dict(meta_channels=49),                      # compressed keys out of range
])
def test_bad_configs_rejected(lib, bad):
    with pytest.raises(K.MosaicKVError) as e:
        K.sizes(_cfg(**bad))
    assert e.value.status == 1


def test_head_dim_must_be_128(lib):
    c = _cfg()
    c.head_dim = 64
    sz = ctypes.c_size_t()
    assert lib.mk_arena_bytes(ctypes.byref(c), ctypes.byref(sz)) == 1


def test_variant_options_change_the_arena(lib):
    a0, _, _ = K.sizes(_cfg())
    a_trunc, _, _ = K.sizes(_cfg(segments=[(0, 38, 0, 96)]))
    assert a_trunc == a0                                   # truncation only changes which channels are kept
    a_keys, _, _ = K.sizes(_cfg(meta_channels=32))
    nblk = (131072 + 64 - 4 - 256 + 31) // 32
    # one compressed key row per block and head: 5 * 32 = 160 bytes
    assert 8 * nblk * 160 <= a_keys - a0 <= 8 * (nblk * 160 + 256)


def test_noalloc_refuses_misaligned_pointers_before_any_launch(lib):
    # The pointers are never dereferenced: the 16-byte check comes first.
    T = (ctypes.c_int32 * 1)(64)
    good, odd = 1 << 20, (1 << 20) + 2
    for q, k, v, o in ((odd, good, good, good), (good, odd, good, good), (good, good, odd, good),
                       (good, good, good, odd)):
        st = lib.mk_dense_decode_attn_noalloc(4, 1, 1, T, ctypes.c_void_p(q), ctypes.c_void_p(k),
                                              ctypes.c_void_p(v), 64, ctypes.c_void_p(o), None)
        assert st == 1


def test_quest_comparator_config_rules(lib):
    # Uncompressed pages keep every channel: r = 128, no truncation, no
    # compressed block keys; the pages are 2 x B x 128 bf16.
    ok = _cfg(segments=[(0, 128, 0)], page_format=1)
    a, _, _ = K.sizes(ok)
    nblk = (131072 + 64 - 4 - 256 + 31) // 32
    assert a > 8 * nblk * 4 * 32 * 128
    for bad in (dict(segments=[(0, 38, 0)]), dict(segments=[(0, 128, 0)], meta_channels=16),
                dict(segments=[(0, 128, 0, 96)]), dict(segments=[(0, 128, 0)], page_format=3)):
        bad.setdefault("page_format", 1)
        with pytest.raises(K.MosaicKVError) as e:
            K.sizes(_cfg(**bad))
        assert e.value.status == 1


def test_bitmap_format_config_rules_and_page_size(lib):
    # [S] sec. 5.1: a bitmap of 128 / g bits per vector in place of r uint8
    # indices: pages of B (4 r + 2 * 16 / g) bytes instead of 6 B r.
    nblk = (131072 + 64 - 4 - 256 + 31) // 32
    a0, _, _ = K.sizes(_cfg())
    for g, r in ((0, 38), (1, 38), (2, 38), (4, 40), (8, 40)):
        a, _, _ = K.sizes(_cfg(segments=[(0, r, 0)], page_format=2, elem_group=g))
        pb = 16 // max(1, g)
        base = a0 - 8 * nblk * 6 * 32 * 38
        assert abs(a - base - 8 * nblk * 32 * (4 * r + 2 * pb)) <= 8 * 4096
    K.sizes(_cfg(segments=[(0, 40, 0, 96), (500, 16, 1)], page_format=2, elem_group=8, meta_channels=16))
    # per segment: group sizes 8 and 2, the page sized for the largest bitmap (g = 2: 8 bytes)
    a, _, _ = K.sizes(_cfg(segments=[(0, 40, 0, 0, 8), (500, 16, 0, 96, 2)], page_format=2, elem_group=4))
    base = a0 - 8 * nblk * 6 * 32 * 38
    own_rot = 8 * 2 * 128 * 128 * 4                   # room for the closed segment's own rotations
    assert abs(a - base - own_rot - 8 * nblk * 32 * (4 * 40 + 2 * 8)) <= 8 * 4096
    for bad in (dict(segments=[(0, 40, 0, 0, 3)]), dict(segments=[(0, 36, 0, 0, 8)]),     # g, r per segment
                dict(segments=[(0, 40, 0, 98, 4)]), dict(page_format=0, segments=[(0, 40, 0, 0, 4)])):
        bad.setdefault("page_format", 2)
        with pytest.raises(K.MosaicKVError) as e:
            K.sizes(_cfg(**bad))
        assert e.value.status == 1
    for bad in (dict(elem_group=3), dict(elem_group=16), dict(elem_group=-1),
                dict(elem_group=4, segments=[(0, 38, 0)]),           # r not a multiple of g
                dict(elem_group=8, segments=[(0, 40, 0, 100)]),      # truncation not a multiple of g
                dict(elem_group=2, page_format=0),                   # a group size needs bitmap pages
                dict(elem_group=1, page_format=1, segments=[(0, 128, 0)])):
        bad.setdefault("page_format", 2)
        bad.setdefault("segments", [(0, 40, 0)])
        with pytest.raises(K.MosaicKVError) as e:
            K.sizes(_cfg(**bad))
        assert e.value.status == 1


def test_per_segment_retention_config_rules(lib):
    # [S] sec. 4.3: a scored segment may give its own sequence retention;
    # then each scored segment keeps its own k, and k_max bounds their sum.
    nblk = (131072 + 64 - 4 - 256 + 31) // 32
    segs = [(0, 38, 0, 0, 0, 200), (500, 38, 1), (700, 38, 0, 0, 0, 50)]
    _, _, k = K.sizes(_cfg(segments=segs))
    assert k == -(-200 * nblk // 1000) + -(-50 * nblk // 1000)
    for bad in (dict(segments=[(0, 38, 0, 0, 0, 1001)]), dict(segments=[(0, 38, 0, 0, 0, -1)]),
                dict(segments=[(0, 38, 0), (500, 38, 1, 0, 0, 100)]),          # always-attended: no rate
                dict(segments=[(0, 38, 0, 0, 0, 100)], topk_fixed=64)):         # not with a fixed k
        with pytest.raises(K.MosaicKVError) as e:
            K.sizes(_cfg(**bad))
        assert e.value.status == 1
