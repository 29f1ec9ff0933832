"""GB300 (sm_103a) CSA2 compressed sparse attention.

Thin ctypes binding over the C ABI in ``include/csa2.h`` (libcsa2.so, built
in-tree from ``csrc/``).  PyTorch only provides device memory and streams:
every step of the path runs in the library's CUDA kernels, and the binding
raises if the library cannot be built or loaded -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import math
import threading

import torch

from . import build as _build

__all__ = [
    "Cfg", "PagedCache", "GroupState", "load", "compress", "index_workspace_bytes", "index_topk", "attend",
    "gather_dequant", "layer", "status_string", "CsaError", "CACHE_FP4", "CACHE_BF16", "MODE_FULL",
    "MODE_REINDEX", "MODE_REUSE", "PAGE", "library_path", "capture", "swa_encode", "CACHE_FP4_S32",
    "FMT_IDX_68B", "FMT_SWA_FP8", "FMT_IDX_QFP4", "SWA_FP8_ROW",
]

CACHE_FP4, CACHE_BF16, CACHE_FP4_S32 = 0, 1, 2
FMT_IDX_68B, FMT_SWA_FP8, FMT_IDX_QFP4 = 1, 2, 4
SWA_FP8_ROW = 528  # bytes of one MXFP8 window row
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
PAGE = 64


class CsaError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, status_string(code) if _lib else code, code))
        self.code = code


class Cfg(C.Structure):
    """csa2_cfg: defaults are the model's sizes (64 x 512 latent, 64 RoPE
    dims, indexer 32 x 128, top-512, window 128, HSI 2048 x 8); `formats`
    takes FMT_IDX_68B (indexer entries with one scale per 32 channels),
    FMT_SWA_FP8 (MXFP8 window rows) and FMT_IDX_QFP4 (FP4 indexer queries)."""
    _fields_ = [("dim", C.c_int32), ("rope_dims", C.c_int32), ("n_heads", C.c_int32), ("idx_heads", C.c_int32),
                ("idx_dim", C.c_int32), ("topk", C.c_int32), ("window", C.c_int32), ("ratio", C.c_int32),
                ("hsi_blocks", C.c_int32), ("hsi_block", C.c_int32), ("cache_dtype", C.c_int32),
                ("formats", C.c_int32), ("rope_theta", C.c_double)]

    def __init__(self, ratio=2, cache_dtype=CACHE_FP4, topk=512, window=128, hsi_blocks=0, rope_theta=1e4,
                 formats=0):
        super().__init__(512, 64, 64, 32, 128, topk, window, ratio, hsi_blocks, 8, cache_dtype, formats, rope_theta)

    @property
    def idx_dtype(self) -> int:
        """Format of the indexer cache under this configuration."""
        return CACHE_FP4_S32 if (self.cache_dtype == CACHE_FP4 and self.formats & FMT_IDX_68B) else self.cache_dtype


class _CacheDesc(C.Structure):
    _fields_ = [("data", C.c_void_p), ("scales", C.c_void_p), ("block_table", C.c_void_p), ("max_pages", C.c_int32),
                ("num_pages", C.c_int32), ("channels", C.c_int32), ("reserved", C.c_int32)]


class _GroupState(C.Structure):
    _fields_ = [("main_cache", _CacheDesc), ("idx_cache", _CacheDesc), ("n_entries", C.c_void_p),
                ("max_entries", C.c_int32), ("reserved", C.c_int32), ("topk", C.c_void_p), ("pool", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("status", C.c_void_p)]


class _LayerIO(C.Structure):
    _fields_ = [("B", C.c_int32), ("Tq", C.c_int32), ("q_pos", C.c_void_p), ("T", C.c_int32), ("x", C.c_void_p),
                ("pos0", C.c_void_p), ("merge_w", C.c_void_p), ("w_idx", C.c_void_p), ("q_idx", C.c_void_p),
                ("head_w", C.c_void_p), ("q", C.c_void_p), ("swa", C.c_void_p), ("S", C.c_int32),
                ("swa_len", C.c_void_p), ("swa_pos0", C.c_void_p), ("scale", C.c_float), ("out", C.c_void_p),
                ("lse", C.c_void_p)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Build (if stale) and load libcsa2.so; raises when that is impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        L = C.CDLL(path)
        vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
        L.csa2_page_bytes.restype = sz
        L.csa2_page_bytes.argtypes = [i32, i32, i32]
        L.csa2_status_string.restype = C.c_char_p
        L.csa2_status_string.argtypes = [i32]
        L.csa2_compress.restype = i32
        L.csa2_compress.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.csa2_index_workspace_bytes.restype = sz
        L.csa2_index_workspace_bytes.argtypes = [vp, i32, i32, i32, i32]
        L.csa2_index_topk.restype = i32
        L.csa2_index_topk.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp, vp]
        L.csa2_index_score.restype = i32
        L.csa2_index_score.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, i32, vp, sz, vp, vp]
        L.csa2_index_select.restype = i32
        L.csa2_index_select.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp, vp]
        L.csa2_attend.restype = i32
        L.csa2_attend.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, C.c_float, vp, vp, vp, vp]
        L.csa2_gather_dequant.restype = i32
        L.csa2_gather_dequant.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.csa2_layer.restype = i32
        L.csa2_layer.argtypes = [vp, i32, vp, vp, vp]
        L.csa2_swa_encode.restype = i32
        L.csa2_swa_encode.argtypes = [i32, i32, vp, vp, vp, i32, vp, vp]
        _lib = L
        return L


def status_string(code: int) -> str:
    return load().csa2_status_string(int(code)).decode()


def _check(fn, rc):
    if rc != 0:
        raise CsaError(fn, rc)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _bf16(t, name):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return _ptr(t, None, name)
    return _ptr(t, torch.int16, name) if t.dtype == torch.int16 else _ptr(t, torch.uint16, name)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class PagedCache:
    """Device pages for one cache (main KV: 512 channels; indexer K: 128) of
    `batch` sequences with `capacity` entries each.  Pages are handed out in
    `page_order` (a permutation of range(num_pages); identity by default)."""

    def __init__(self, batch: int, capacity: int, channels: int, cache_dtype: int, device="cuda",
                 page_order=None, spare_pages: int = 0):
        lib = load()
        self.batch, self.channels, self.cache_dtype = batch, channels, cache_dtype
        self.max_pages = max(1, math.ceil(capacity / PAGE))
        self.capacity = self.max_pages * PAGE
        self.num_pages = batch * self.max_pages + spare_pages
        db = lib.csa2_page_bytes(channels, cache_dtype, 0)
        sb = lib.csa2_page_bytes(channels, cache_dtype, 1)
        if db == 0:
            raise ValueError("unsupported cache (channels=%d dtype=%d)" % (channels, cache_dtype))
        self.data = torch.zeros((self.num_pages, db), dtype=torch.uint8, device=device)
        self.scales = torch.zeros((self.num_pages, sb), dtype=torch.uint8, device=device) if sb else None
        order = torch.arange(batch * self.max_pages) if page_order is None else torch.as_tensor(page_order)
        self.block_table = order[: batch * self.max_pages].reshape(batch, self.max_pages).to(
            device=device, dtype=torch.int32).contiguous()

    def desc(self) -> _CacheDesc:
        return _CacheDesc(self.data.data_ptr(), self.scales.data_ptr() if self.scales is not None else None,
                          self.block_table.data_ptr(), self.max_pages, self.num_pages, self.channels, 0)


def compress(cfg: Cfg, x, pos0, merge_w, w_idx, main: PagedCache, idx: PagedCache, n_entries, status=None,
             stream=None):
    """a1: x [B][T][512] bf16, pos0 [B] int64, merge_w [r][512] fp32, w_idx [512][128] bf16."""
    B, T, _ = x.shape
    md, idd = main.desc(), idx.desc()
    _check("csa2_compress", load().csa2_compress(
        C.byref(cfg), B, T, _bf16(x, "x"), _ptr(pos0, torch.int64, "pos0"), _ptr(merge_w, torch.float32, "merge_w"),
        _bf16(w_idx, "w_idx"), C.byref(md), C.byref(idd), _ptr(n_entries, torch.int32, "n_entries"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def index_workspace_bytes(cfg: Cfg, B: int, Tq: int, max_entries: int, reindex: bool = False) -> int:
    return int(load().csa2_index_workspace_bytes(C.byref(cfg), B, Tq, max_entries, int(reindex)))


def index_topk(cfg: Cfg, q_idx, q_pos, idx: PagedCache, n_entries, max_entries: int, topk_out, workspace,
               head_w=None, pool=None, pool_out=None, status=None, stream=None):
    """a3-a6: q_idx [B][Tq][32][128] bf16, q_pos [B][Tq] int64 -> topk_out [B][Tq][k] int32
    (and pool_out [B][Tq][hsi_blocks] for an HSI Full layer; `pool` selects Reindex)."""
    B, Tq = q_idx.shape[:2]
    d = idx.desc()
    _check("csa2_index_topk", load().csa2_index_topk(
        C.byref(cfg), B, Tq, _bf16(q_idx, "q_idx"), _ptr(head_w, torch.float32, "head_w"),
        _ptr(q_pos, torch.int64, "q_pos"), C.byref(d), _ptr(n_entries, torch.int32, "n_entries"), int(max_entries),
        _ptr(pool, torch.int32, "pool"), _ptr(topk_out, torch.int32, "topk_out"),
        _ptr(pool_out, torch.int32, "pool_out"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(status, torch.int32, "status"), _stream(stream)))


def index_score(cfg: Cfg, q_idx, q_pos, idx: PagedCache, n_entries, max_entries: int, workspace, head_w=None,
                pool=None, hsi=False, status=None, stream=None):
    """a3/a5/a6 scores of every query into `workspace` (which holds them all), for index_select."""
    B, Tq = q_idx.shape[:2]
    d = idx.desc()
    _check("csa2_index_score", load().csa2_index_score(
        C.byref(cfg), B, Tq, _bf16(q_idx, "q_idx"), _ptr(head_w, torch.float32, "head_w"),
        _ptr(q_pos, torch.int64, "q_pos"), C.byref(d), _ptr(n_entries, torch.int32, "n_entries"), int(max_entries),
        _ptr(pool, torch.int32, "pool"), 1 if hsi else 0, _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(status, torch.int32, "status"), _stream(stream)))


def index_select(cfg: Cfg, q_pos, idx: PagedCache, n_entries, max_entries: int, topk_out, workspace, pool=None,
                 pool_out=None, status=None, stream=None):
    """a4/a5 from the scores index_score left in `workspace` -> topk_out (and pool_out)."""
    B, Tq = q_pos.shape[:2]
    d = idx.desc()
    _check("csa2_index_select", load().csa2_index_select(
        C.byref(cfg), B, Tq, _ptr(q_pos, torch.int64, "q_pos"), C.byref(d), _ptr(n_entries, torch.int32, "n_entries"),
        int(max_entries), _ptr(pool, torch.int32, "pool"), _ptr(topk_out, torch.int32, "topk_out"),
        _ptr(pool_out, torch.int32, "pool_out"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _ptr(status, torch.int32, "status"), _stream(stream)))


def _swa(cfg: Cfg, swa):
    """Window rows: bf16 [B][S][512], or uint8 MXFP8 rows [B][S][528] under FMT_SWA_FP8."""
    if swa is None:
        return None
    if cfg.formats & FMT_SWA_FP8:
        if swa.shape[-1] != SWA_FP8_ROW:
            raise ValueError("MXFP8 window rows must be [B][S][%d] uint8" % SWA_FP8_ROW)
        return _ptr(swa, torch.uint8, "swa")
    return _bf16(swa, "swa")


def swa_encode(x, row0, rows, status=None, stream=None):
    """FP8 window rows: x [B][T][512] bf16 -> rows[b][row0[b] + i] of rows [B][S][528] uint8 (MXFP8)."""
    B, T = x.shape[:2]
    _check("csa2_swa_encode", load().csa2_swa_encode(
        B, T, _bf16(x, "x"), _ptr(row0, torch.int64, "row0"), _ptr(rows, torch.uint8, "rows"), rows.shape[1],
        _ptr(status, torch.int32, "status"), _stream(stream)))


def attend(cfg: Cfg, q, main: PagedCache, n_entries, topk, swa, swa_len, swa_pos0, q_pos, out, lse=None,
           scale=None, status=None, stream=None):
    """a7: q [B][Tq][64][512] bf16, topk [B][Tq][k], swa [B][S][512] bf16 (or [B][S][528] uint8 MXFP8 rows
    under FMT_SWA_FP8) -> out [B][Tq][64][512] fp32."""
    B, Tq = q.shape[:2]
    S = swa.shape[1] if swa is not None else 0
    d = main.desc()
    scale = 1.0 / math.sqrt(512) if scale is None else float(scale)
    _check("csa2_attend", load().csa2_attend(
        C.byref(cfg), B, Tq, _bf16(q, "q"), C.byref(d), _ptr(n_entries, torch.int32, "n_entries"),
        _ptr(topk, torch.int32, "topk"), _swa(cfg, swa), S, _ptr(swa_len, torch.int32, "swa_len"),
        _ptr(swa_pos0, torch.int64, "swa_pos0"), _ptr(q_pos, torch.int64, "q_pos"), scale,
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(status, torch.int32, "status"),
        _stream(stream)))


def gather_dequant(cache: PagedCache, ids, out, status=None, stream=None):
    """Decode entries ids [B][n] of `cache` into out [B][n][channels] fp32."""
    B, n = ids.shape
    d = cache.desc()
    _check("csa2_gather_dequant", load().csa2_gather_dequant(
        C.byref(d), cache.cache_dtype, B, n, _ptr(ids, torch.int32, "ids"), _ptr(out, torch.float32, "out"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


class GroupState:
    """Shared state of one cross-layer group: caches, entry counts, the latest
    published top-k, the HSI pool and the indexer workspace."""

    def __init__(self, main: PagedCache, idx: PagedCache, n_entries, max_entries: int, topk, pool, workspace,
                 status):
        self.main, self.idx, self.n_entries, self.max_entries = main, idx, n_entries, max_entries
        self.topk, self.pool, self.workspace, self.status = topk, pool, workspace, status
        self._c = _GroupState(main.desc(), idx.desc(), _ptr(n_entries, torch.int32, "n_entries"), int(max_entries), 0,
                              _ptr(topk, torch.int32, "topk"), _ptr(pool, torch.int32, "pool"),
                              _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                              _ptr(status, torch.int32, "status"))


def layer(cfg: Cfg, mode: int, state: GroupState, q_pos, q, swa, swa_len, swa_pos0, out, lse=None, q_idx=None,
          head_w=None, x=None, pos0=None, merge_w=None, w_idx=None, scale=None, stream=None):
    """a8: one CSA2 layer in mode MODE_FULL / MODE_REINDEX / MODE_REUSE."""
    B, Tq = q.shape[:2]
    io = _LayerIO(B, Tq, _ptr(q_pos, torch.int64, "q_pos"), x.shape[1] if x is not None else 0, _bf16(x, "x"),
                  _ptr(pos0, torch.int64, "pos0"), _ptr(merge_w, torch.float32, "merge_w"), _bf16(w_idx, "w_idx"),
                  _bf16(q_idx, "q_idx"), _ptr(head_w, torch.float32, "head_w"), _bf16(q, "q"), _swa(cfg, swa),
                  swa.shape[1] if swa is not None else 0, _ptr(swa_len, torch.int32, "swa_len"),
                  _ptr(swa_pos0, torch.int64, "swa_pos0"), 1.0 / math.sqrt(512) if scale is None else float(scale),
                  _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"))
    _check("csa2_layer", load().csa2_layer(C.byref(cfg), int(mode), C.byref(state._c), C.byref(io), _stream(stream)))


class Captured:
    """A sequence of library calls (and the caller's copies) recorded once as
    a CUDA graph and replayed with one launch: the same kernels on the same
    buffers, without the host-side cost of issuing them call by call.  Every
    buffer the calls touch must stay alive and in place; a call's host-side
    arguments (sizes, configs, pointers) are those of the capture."""

    def __init__(self, fn, warmup: int = 1):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()

    def __call__(self):
        self.graph.replay()


def capture(fn, warmup: int = 1) -> Captured:
    """Record ``fn`` (library calls on the current stream) for replay."""
    return Captured(fn, warmup)

