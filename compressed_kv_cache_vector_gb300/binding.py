"""ctypes binding of libmosaickv.so (declared in include/mosaickv.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch provides device memory (the arena and workspace the
library asks for, inputs, outputs) and the CUDA stream.  There is no CPU
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import torch

PKG = os.path.dirname(os.path.abspath(__file__))
# MOSAICKV_LIB names another build of the library to load (the tests use it
# for the checked build, libmosaickv_checks.so).
LIB_PATH = os.environ.get("MOSAICKV_LIB") or os.path.join(PKG, "libmosaickv.so")
HEADER = os.path.join(PKG, "..", "include", "mosaickv.h")

MK_HEAD_DIM = 128
MK_MAX_SEGMENTS = 4
MK_MAX_SPLITS = 64
MK_PAGES_PACKED, MK_PAGES_DENSE, MK_PAGES_BITMAP = 0, 1, 2
STATUS = {0: "MK_OK", 1: "MK_EINVAL", 2: "MK_ENOMEM", 3: "MK_ESTATE", 4: "MK_ECUDA",
          5: "MK_EDEVICE", 6: "MK_ETIMEOUT", 7: "MK_ENOTSUP"}
c_i32, c_i64, c_size, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p


class MosaicKVError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class MkSegment(ctypes.Structure):
    _fields_ = [("begin_permille", c_i32), ("r", c_i32), ("always", c_i32), ("keep_channels", c_i32),
                ("elem_group", c_i32), ("retain_permille", c_i32)]


class MkConfig(ctypes.Structure):
    _fields_ = [("head_dim", c_i32), ("n_q_heads", c_i32), ("n_kv_heads", c_i32), ("n_layers", c_i32),
                ("max_seqs", c_i32), ("max_tokens", c_i32), ("n_sink", c_i32), ("window", c_i32),
                ("block", c_i32), ("topk_fixed", c_i32), ("retain_permille", c_i32),
                ("n_segments", c_i32), ("seg", MkSegment * MK_MAX_SEGMENTS), ("meta_channels", c_i32),
                ("page_format", c_i32), ("elem_group", c_i32)]


class MkAlg2Params(ctypes.Structure):
    _fields_ = [("outlier_abs", ctypes.c_double), ("outlier_ratio_max", ctypes.c_double),
                ("alpha", ctypes.c_double), ("r_min", c_i32), ("r_max", c_i32), ("hist_bins", c_i32)]


class MkSegStats(ctypes.Structure):
    _fields_ = [("variance", ctypes.c_double), ("outlier_ratio", ctypes.c_double), ("entropy", ctypes.c_double)]


class MkLayoutInfo(ctypes.Structure):
    _fields_ = [("rkt", c_i64), ("rvt", c_i64), ("rv", c_i64), ("sink_k", c_i64), ("sink_v", c_i64),
                ("win_k", c_i64), ("win_v", c_i64), ("meta", c_i64), ("pages", c_i64),
                ("page_stride", c_i64), ("nblk_cap", c_i32), ("T", c_i32),
                ("seg_first_block", c_i32 * MK_MAX_SEGMENTS), ("n_segments", c_i32), ("reserved", c_i32),
                ("cmeta", c_i64), ("cmeta_row", c_i32), ("meta_channels", c_i32)]


_SIGS = {
    "mk_arena_bytes": [ctypes.POINTER(MkConfig), ctypes.POINTER(c_size)],
    "mk_workspace_bytes": [ctypes.POINTER(MkConfig), ctypes.POINTER(c_size)],
    "mk_max_select": [ctypes.POINTER(MkConfig), ctypes.POINTER(c_i32)],
    "mk_create": [ctypes.POINTER(MkConfig), c_vp, c_size, c_vp, c_size, ctypes.POINTER(c_vp)],
    "mk_destroy": [c_vp],
    "mk_set_rotation": [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp],
    "mk_append_compress": [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp],
    "mk_block_select": [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp],
    "mk_append_select": [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp],
    "mk_decode_attn": [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp],
    "mk_dense_decode_attn": [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_vp],
    "mk_gram": [c_vp, c_i64, c_i64, c_vp, c_vp],
    "mk_poll_error": [c_vp, ctypes.POINTER(c_i32)],
    "mk_clear_error": [c_vp],
    "mk_sync_state": [c_vp],
    "mk_seq_length": [c_vp, c_i32, c_i32, ctypes.POINTER(c_i32)],
    "mk_layout": [c_vp, c_i32, c_i32, c_i32, ctypes.POINTER(MkLayoutInfo)],
    "mk_record_event": [c_vp, c_vp],
    "mk_dense_decode_attn_noalloc": [c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_vp],
    "mk_noalloc_poll_error": [ctypes.POINTER(c_i32)],
    "mk_cov_update": [c_vp, c_vp, c_i64, c_i64, c_i32],
    "mk_rotation_from_cov": [c_vp, c_i32, c_vp, c_vp],
    "mk_choose_r": [c_vp, c_i32, ctypes.c_double, ctypes.POINTER(c_i32)],
    "mk_alg2_segment_r": [c_vp, c_i64, c_i64, c_i32, ctypes.c_double, ctypes.POINTER(MkAlg2Params),
                          ctypes.POINTER(MkSegStats), ctypes.POINTER(c_i32)],
    "mk_choose_block_size": [c_vp, c_i64, c_i64, c_i32, c_vp, c_i32, ctypes.c_double, c_vp, ctypes.POINTER(c_i32)],
    "mk_host_pack_blocks": [c_vp, c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_i64, c_i32, c_i32, c_i32,
                            c_vp, c_vp, c_vp],
    "mk_swap_segment": [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp],
}

_lib = None


def header_symbols():
    """Names of the functions include/mosaickv.h declares."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^\s*(?:mk_status|const char\*)\s+(mk_\w+)\s*\(", txt, re.M)))


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with compressed_kv_cache_vector_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = c_i32
    lib.mk_status_str.argtypes = [c_i32]
    lib.mk_status_str.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(fn, st):
    if st != 0:
        raise MosaicKVError(fn, st)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _i32(xs):
    a = (c_i32 * len(xs))(*[int(x) for x in xs])
    return a


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(n_q_heads, n_kv_heads, n_layers, max_seqs, max_tokens, n_sink, window, block,
                segments, topk_fixed=0, retain_permille=0, meta_channels=0, page_format=0,
                elem_group=0) -> MkConfig:
    c = MkConfig()
    c.head_dim = MK_HEAD_DIM
    c.n_q_heads, c.n_kv_heads, c.n_layers = n_q_heads, n_kv_heads, n_layers
    c.max_seqs, c.max_tokens = max_seqs, max_tokens
    c.n_sink, c.window, c.block = n_sink, window, block
    c.topk_fixed, c.retain_permille = topk_fixed, retain_permille
    c.meta_channels = meta_channels
    c.page_format = page_format
    c.elem_group = elem_group
    c.n_segments = len(segments)
    for i, sg in enumerate(segments):
        b, r, a = sg[:3]
        keep = sg[3] if len(sg) > 3 else 0
        c.seg[i].begin_permille, c.seg[i].r, c.seg[i].always, c.seg[i].keep_channels = b, r, a, keep
        c.seg[i].elem_group = sg[4] if len(sg) > 4 else 0   # bitmap pages: the segment's own group size
        c.seg[i].retain_permille = sg[5] if len(sg) > 5 else 0   # the segment's own sequence retention
    return c


def sizes(cfg: MkConfig):
    lib = load()
    a, w, k = c_size(), c_size(), c_i32()
    _check("mk_arena_bytes", lib.mk_arena_bytes(ctypes.byref(cfg), ctypes.byref(a)))
    _check("mk_workspace_bytes", lib.mk_workspace_bytes(ctypes.byref(cfg), ctypes.byref(w)))
    _check("mk_max_select", lib.mk_max_select(ctypes.byref(cfg), ctypes.byref(k)))
    return a.value, w.value, k.value


class MosaicKV:
    """One compressed KV cache (all layers, sequence slots and kv heads) on one GPU."""

    def __init__(self, cfg: MkConfig, device="cuda"):
        self.lib = load()
        self.cfg = cfg
        self.device = torch.device(device)
        self.arena_bytes, self.ws_bytes, self.k_max = sizes(cfg)
        self.arena = torch.empty(self.arena_bytes, dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        h = c_vp()
        _check("mk_create", self.lib.mk_create(ctypes.byref(cfg), _ptr(self.arena), self.arena_bytes,
                                               _ptr(self.workspace), self.ws_bytes, ctypes.byref(h)))
        self.h = h
        self.G = cfg.n_q_heads // cfg.n_kv_heads
        info = self.layout(0, 0, 0)
        self.nblk_cap = info["nblk_cap"]

    def close(self):
        if getattr(self, "h", None):
            self.lib.mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- calls ------------------------------------------------------------
    def set_rotation(self, layer, seq, kvh, Rk, Rv, stream=None):
        Rk = np.ascontiguousarray(Rk, dtype=np.float32)
        Rv = np.ascontiguousarray(Rv, dtype=np.float32)
        _check("mk_set_rotation", self.lib.mk_set_rotation(
            self.h, layer, seq, kvh, Rk.ctypes.data_as(c_vp), Rv.ctypes.data_as(c_vp), _stream(stream)))

    def append(self, layer, seq_ids, n_new, k, v, stream=None):
        _check("mk_append_compress", self.lib.mk_append_compress(
            self.h, layer, len(seq_ids), _i32(seq_ids), _i32(n_new), _ptr(k), _ptr(v), _stream(stream)))

    def alloc_select(self, n_seqs):
        ids = torch.empty(n_seqs, self.cfg.n_kv_heads, self.k_max, dtype=torch.int32, device=self.device)
        n_sel = torch.empty(n_seqs, self.cfg.n_kv_heads, dtype=torch.int32, device=self.device)
        return ids, n_sel

    def block_select(self, layer, seq_ids, q, ids=None, n_sel=None, scores=None, stream=None):
        if ids is None:
            ids, n_sel = self.alloc_select(len(seq_ids))
        _check("mk_block_select", self.lib.mk_block_select(
            self.h, layer, len(seq_ids), _i32(seq_ids), _ptr(q), _ptr(ids), _ptr(n_sel), _ptr(scores),
            _stream(stream)))
        return ids, n_sel

    def append_select(self, layer, seq_ids, k, v, q, ids=None, n_sel=None, scores=None, stream=None):
        """One new token per sequence (k, v: [n_seqs, n_kv, 128] bf16) appended, then blocks selected for q."""
        if ids is None:
            ids, n_sel = self.alloc_select(len(seq_ids))
        _check("mk_append_select", self.lib.mk_append_select(
            self.h, layer, len(seq_ids), _i32(seq_ids), _ptr(k), _ptr(v), _ptr(q), _ptr(ids), _ptr(n_sel),
            _ptr(scores), _stream(stream)))
        return ids, n_sel

    def decode_attn(self, layer, seq_ids, ids, n_sel, out=None, stream=None):
        if out is None:
            out = torch.empty(len(seq_ids), self.cfg.n_q_heads, MK_HEAD_DIM, dtype=torch.bfloat16,
                              device=self.device)
        _check("mk_decode_attn", self.lib.mk_decode_attn(
            self.h, layer, len(seq_ids), _i32(seq_ids), _ptr(ids), _ptr(n_sel), _ptr(out), _stream(stream)))
        return out

    def dense_attn(self, T, q, K, V, out=None, stream=None):
        if out is None:
            out = torch.empty(q.shape[0], self.cfg.n_q_heads, MK_HEAD_DIM, dtype=torch.bfloat16,
                              device=self.device)
        _check("mk_dense_decode_attn", self.lib.mk_dense_decode_attn(
            self.h, len(T), _i32(T), _ptr(q), _ptr(K), _ptr(V), K.shape[2], _ptr(out), _stream(stream)))
        return out

    def swap_segment(self, layer, seq, kvh, segment, r, keep_channels, pages, meta, cmeta=None, stream=None,
                     R_k=None, R_v=None):
        """Replace a closed segment's pages and keys with host-packed ones (host_pack_blocks), under r from
        then on, and under the segment's own rotations R_k, R_v if given (the pages must be packed with
        them).  The host arrays must live until the stream has run the copies."""
        pg = np.ascontiguousarray(pages, dtype=np.uint8)
        mt = np.ascontiguousarray(meta, dtype=np.uint16)
        cm = None if cmeta is None else np.ascontiguousarray(cmeta, dtype=np.uint8)
        rk = None if R_k is None else np.ascontiguousarray(R_k, dtype=np.float32)
        rv = None if R_v is None else np.ascontiguousarray(R_v, dtype=np.float32)
        self._swap_keep = (pg, mt, cm)   # kept alive until the next swap
        _check("mk_swap_segment", self.lib.mk_swap_segment(
            self.h, layer, seq, kvh, segment, r, keep_channels,
            _np_ptr(rk) if rk is not None else ctypes.c_void_p(0), _np_ptr(rv) if rv is not None else ctypes.c_void_p(0),
            _np_ptr(pg), _np_ptr(mt), _np_ptr(cm) if cm is not None else ctypes.c_void_p(0), _stream(stream)))

    def poll_error(self):
        d = c_i32()
        st = self.lib.mk_poll_error(self.h, ctypes.byref(d))
        return st, d.value

    def clear_error(self):
        _check("mk_clear_error", self.lib.mk_clear_error(self.h))

    def sync_state(self):
        _check("mk_sync_state", self.lib.mk_sync_state(self.h))

    def seq_length(self, layer, seq):
        t = c_i32()
        _check("mk_seq_length", self.lib.mk_seq_length(self.h, layer, seq, ctypes.byref(t)))
        return t.value

    def layout(self, layer, seq, kvh):
        info = MkLayoutInfo()
        _check("mk_layout", self.lib.mk_layout(self.h, layer, seq, kvh, ctypes.byref(info)))
        d = {f: getattr(info, f) for f, _ in MkLayoutInfo._fields_ if f not in ("seg_first_block", "reserved")}
        d["seg_first_block"] = list(info.seg_first_block)[: info.n_segments]
        return d

    # --- raw views into the arena (tests and tools) -----------------------
    def unit_views(self, layer, seq, kvh):
        """Byte/word views of one head's stored state (no copies)."""
        L = self.layout(layer, seq, kvh)
        a = self.arena
        D = MK_HEAD_DIM
        S, W = self.cfg.n_sink, self.cfg.window

        def words(off, n):
            return a[off:off + 2 * n].view(torch.int16)

        return {
            "sink_k": words(L["sink_k"], S * D).view(S, D) if S else None,
            "sink_v": words(L["sink_v"], S * D).view(S, D) if S else None,
            "win_k": words(L["win_k"], W * D).view(W, D),
            "win_v": words(L["win_v"], W * D).view(W, D),
            "meta": words(L["meta"], L["nblk_cap"] * 2 * D).view(L["nblk_cap"], 2, D),
            "pages": a[L["pages"]:L["pages"] + L["nblk_cap"] * L["page_stride"]].view(
                L["nblk_cap"], L["page_stride"]),
            "cmeta": (a[L["cmeta"]:L["cmeta"] + L["nblk_cap"] * L["cmeta_row"]].view(L["nblk_cap"], L["cmeta_row"])
                      if L["meta_channels"] else None),
            "layout": L,
        }


def dense_attn_noalloc(n_q_heads, n_kv_heads, T, q, K, V, out, stream=None):
    """Uncompressed decode attention with no context and no workspace: the
    library's static scratch array stands in for it (for callers that cannot
    allocate device memory where they run attention)."""
    _check("mk_dense_decode_attn_noalloc", load().mk_dense_decode_attn_noalloc(
        n_q_heads, n_kv_heads, len(T), _i32(T), _ptr(q), _ptr(K), _ptr(V), K.shape[2], _ptr(out),
        _stream(stream)))
    return out


def noalloc_poll_error():
    """(status, detail) of the allocation-free call's device-side error word on
    the current device (waits for the device; clears the word)."""
    d = c_i32(0)
    st = load().mk_noalloc_poll_error(ctypes.byref(d))
    return st, d.value


def record_event(ev, stream=None):
    """Records a torch.cuda.Event (timing enabled) so it also works under graph capture."""
    if ev.cuda_event == 0:
        ev.record()            # creates the underlying event
    _check("mk_record_event", load().mk_record_event(ctypes.c_void_p(ev.cuda_event), _stream(stream)))


def gram(x, n_rows, row_stride, out=None, stream=None):
    """X^T X (fp32) of bf16 rows of 128 values on the GPU (set-up helper)."""
    lib = load()
    if out is None:
        out = torch.empty(MK_HEAD_DIM, MK_HEAD_DIM, dtype=torch.float32, device=x.device)
    _check("mk_gram", lib.mk_gram(_ptr(x), n_rows, row_stride, _ptr(out), _stream(stream)))
    return out


def rotation_from_gram(G):
    """Host eigensolve of a Gram matrix (the library's native Jacobi, fp64):
    rows of R are the eigenvectors by descending eigenvalue, so k' = k R^T."""
    Gd = np.asarray(G, dtype=np.float64)
    R, _ = rotation_from_cov(0.5 * (Gd + Gd.T))
    return R


# ---- host-side strategy generation (host arrays; no GPU) ----------------------

def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _bf16_words(x):
    """A 2-D array of bf16 words (uint16) from a uint16 array or a CPU bf16 tensor."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.uint16)


def cov_update(G, x):
    """G += X^T X in fp64 (G: d x d float64, updated in place; x: n x d bf16 rows)."""
    w = _bf16_words(x)
    assert G.dtype == np.float64 and G.flags.c_contiguous and G.shape == (w.shape[1], w.shape[1])
    _check("mk_cov_update", load().mk_cov_update(_np_ptr(G), _np_ptr(w), w.shape[0], w.shape[1], w.shape[1]))
    return G


def rotation_from_cov(G):
    """Native Jacobi eigen-decomposition: (R float32 d x d, rows = eigenvectors; lambda descending)."""
    Gd = np.ascontiguousarray(G, dtype=np.float64)
    d = Gd.shape[0]
    R = np.empty((d, d), dtype=np.float32)
    lam = np.empty(d, dtype=np.float64)
    _check("mk_rotation_from_cov", load().mk_rotation_from_cov(_np_ptr(Gd), d, _np_ptr(R), _np_ptr(lam)))
    return R, lam


def choose_r(lam, loss_max):
    """Smallest r whose discarded energy is at most loss_max."""
    l = np.ascontiguousarray(lam, dtype=np.float64)
    r = c_i32(0)
    _check("mk_choose_r", load().mk_choose_r(_np_ptr(l), l.shape[0], float(loss_max), ctypes.byref(r)))
    return r.value


def alg2_segment_r(seg, budget, outlier_abs, outlier_ratio_max, alpha, r_min, r_max, hist_bins):
    """Algorithm 2 on one rotated segment: (r, {variance, outlier_ratio, entropy})."""
    w = _bf16_words(seg)
    p = MkAlg2Params(outlier_abs, outlier_ratio_max, alpha, r_min, r_max, hist_bins)
    st = MkSegStats()
    r = c_i32(0)
    _check("mk_alg2_segment_r", load().mk_alg2_segment_r(_np_ptr(w), w.shape[0], w.shape[1], w.shape[1],
                                                         float(budget), ctypes.byref(p), ctypes.byref(st),
                                                         ctypes.byref(r)))
    return r.value, {"variance": st.variance, "outlier_ratio": st.outlier_ratio, "entropy": st.entropy}


def choose_block_size(seg, candidates, threshold):
    """[S] sec. 5.5 block-size choice for one segment (seg: bf16 words as uint16, or a CPU bf16 tensor):
    (block size, within-block variance per candidate, NaN where no complete block)."""
    w = _bf16_words(seg)
    cands = np.ascontiguousarray(candidates, dtype=np.int32)
    var = np.empty(cands.shape[0], dtype=np.float64)
    b = c_i32(0)
    _check("mk_choose_block_size", load().mk_choose_block_size(
        _np_ptr(w), w.shape[0], w.shape[1], w.shape[1], _np_ptr(cands), cands.shape[0], float(threshold),
        _np_ptr(var), ctypes.byref(b)))
    return b.value, var


def host_pack_blocks(Rk, Rv, k, v, block, r, keep_channels, page_stride, meta_channels=0, page_format=0,
                     elem_group=0):
    """Exact host re-compression of complete blocks (raw bf16 rows k, v: n_blocks * block rows of 128):
    (pages uint8 [n, page_stride], meta uint16 [n, 2, 128], compressed keys uint8 [n, row] or None)."""
    kw, vw = _bf16_words(k), _bf16_words(v)
    n = kw.shape[0] // block
    Rk32 = np.ascontiguousarray(Rk, dtype=np.float32)
    Rv32 = np.ascontiguousarray(Rv, dtype=np.float32)
    pages = np.empty((n, page_stride), dtype=np.uint8)
    meta = np.empty((n, 2, MK_HEAD_DIM), dtype=np.uint16)
    crow = (5 * meta_channels + 15) // 16 * 16 if meta_channels else 0
    cmeta = np.empty((n, crow), dtype=np.uint8) if meta_channels else None
    _check("mk_host_pack_blocks", load().mk_host_pack_blocks(
        _np_ptr(Rk32), _np_ptr(Rv32), _np_ptr(kw), _np_ptr(vw), kw.shape[1], n, block, r, keep_channels, page_stride,
        meta_channels, page_format, elem_group, _np_ptr(pages), _np_ptr(meta),
        _np_ptr(cmeta) if cmeta is not None else ctypes.c_void_p(0)))
    return pages, meta, cmeta
