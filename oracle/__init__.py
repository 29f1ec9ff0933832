"""CSA2 CPU oracle (fp64 C, loaded through ctypes) -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The CUDA library never links it, and
it imports nothing from the CUDA package.  See ``csa2_oracle.h`` for the
sources, readings and canonical layouts.

Every numpy-level function below marshals arrays and calls the C code; no
arithmetic of the method is done here.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libcsa2_oracle.so")
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_lock = threading.Lock()
_lib = None

CACHE_FP4 = 0
CACHE_BF16 = 1
CACHE_FP4_G32 = 2   # FP4 main cache, indexer entries with one scale per 32 channels (68 B)
SWA_BF16 = 0
SWA_MXFP8 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction so x86 and Arm agree)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "csa2_oracle.h"))):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            vp, i, d = C.c_void_p, C.c_int, C.c_double
            L.orc_bf16_value.restype = d
            L.orc_bf16_value.argtypes = [C.c_uint16]
            L.orc_bf16_round.restype = C.c_uint16
            L.orc_bf16_round.argtypes = [d]
            L.orc_e2m1_value.restype = d
            L.orc_e2m1_value.argtypes = [i]
            L.orc_e4m3_value.restype = d
            L.orc_e4m3_value.argtypes = [i]
            L.orc_e4m3_nearest_code.restype = i
            L.orc_e4m3_nearest_code.argtypes = [d]
            L.orc_e2m1_nearest_code.restype = i
            L.orc_e2m1_nearest_code.argtypes = [d, d]
            L.orc_fp4_encode.argtypes = [vp, i, vp, vp]
            L.orc_fp4_decode.argtypes = [vp, vp, i, vp]
            L.orc_fp4_encode_g.argtypes = [vp, i, i, vp, vp]
            L.orc_fp4_decode_g.argtypes = [vp, vp, i, i, vp]
            L.orc_e8m0_value.restype = d
            L.orc_e8m0_value.argtypes = [i]
            L.orc_mxfp8_encode.argtypes = [vp, i, vp]
            L.orc_mxfp8_decode.argtypes = [vp, i, vp]
            L.orc_compress.restype = i
            L.orc_compress.argtypes = [i, i, i, i, i, i, d, i, vp, vp, vp, vp, i,
                                       vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            L.orc_index_topk.restype = i
            L.orc_index_topk.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, i, i, i,
                                         vp, vp, vp, vp]
            L.orc_index_topk_q.restype = i
            L.orc_index_topk_q.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, vp, i, vp, vp, i, i, i,
                                           vp, vp, vp, vp]
            L.orc_attend.restype = i
            L.orc_attend.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, i, vp, i, i, vp, vp, vp,
                                     i, d, vp, vp]
            L.orc_attend_dense.restype = i
            L.orc_attend_dense.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, i, i, vp, vp,
                                           vp, i, d, vp]
            L.orc_threads.restype = i
            _lib = L
    return _lib


def threads() -> int:
    return lib().orc_threads()


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codecs ----

def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def bf16_round(x: float) -> int:
    return lib().orc_bf16_round(float(x))


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(int(byte))


def e4m3_nearest_code(y: float) -> int:
    return lib().orc_e4m3_nearest_code(float(y))


def e2m1_nearest_code(x: float, scale: float) -> int:
    return lib().orc_e2m1_nearest_code(float(x), float(scale))


def fp4_encode(x: np.ndarray, group: int = 16):
    """x [..., C] fp64 -> (codes [..., C/2] u8, scales [..., C/group] u8)."""
    x = _c(x, np.float64)
    Cn = x.shape[-1]
    rows = x.reshape(-1, Cn)
    codes = np.zeros((rows.shape[0], Cn // 2), np.uint8)
    scales = np.zeros((rows.shape[0], Cn // group), np.uint8)
    L = lib()
    for n in range(rows.shape[0]):
        L.orc_fp4_encode_g(_p(rows[n]), Cn, group, _p(codes[n]), _p(scales[n]))
    return codes.reshape(x.shape[:-1] + (Cn // 2,)), scales.reshape(x.shape[:-1] + (Cn // group,))


def fp4_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse of fp4_encode; the scale group (16 or 32) follows from the shapes."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    Cn = codes.shape[-1] * 2
    group = Cn // scales.shape[-1]
    cr = codes.reshape(-1, Cn // 2)
    sr = scales.reshape(-1, Cn // group)
    out = np.zeros((cr.shape[0], Cn), np.float64)
    L = lib()
    for n in range(cr.shape[0]):
        L.orc_fp4_decode_g(_p(cr[n]), _p(sr[n]), Cn, group, _p(out[n]))
    return out.reshape(codes.shape[:-1] + (Cn,))


def e8m0_value(byte: int) -> float:
    return lib().orc_e8m0_value(int(byte))


def mxfp8_encode(x: np.ndarray) -> np.ndarray:
    """x [..., C] fp64 -> MXFP8 rows [..., C + C/32] u8 (elements, then scales)."""
    x = _c(x, np.float64)
    Cn = x.shape[-1]
    rows = x.reshape(-1, Cn)
    out = np.zeros((rows.shape[0], Cn + Cn // 32), np.uint8)
    L = lib()
    for n in range(rows.shape[0]):
        L.orc_mxfp8_encode(_p(rows[n]), Cn, _p(out[n]))
    return out.reshape(x.shape[:-1] + (Cn + Cn // 32,))


def mxfp8_decode(rows: np.ndarray) -> np.ndarray:
    rows = _c(rows, np.uint8)
    Cn = rows.shape[-1] * 32 // 33
    rr = rows.reshape(-1, rows.shape[-1])
    out = np.zeros((rr.shape[0], Cn), np.float64)
    L = lib()
    for n in range(rr.shape[0]):
        L.orc_mxfp8_decode(_p(rr[n]), Cn, _p(out[n]))
    return out.reshape(rows.shape[:-1] + (Cn,))


def swa_encode(bits: np.ndarray) -> np.ndarray:
    """bf16 window rows [..., C] (bit patterns) -> MXFP8 rows [..., C + C/32]."""
    return mxfp8_encode(bf16_bits_to_f64(bits))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (_c(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------- the path ----

class Cache:
    """Canonical (unpaged) cache of B sequences x n_cap entries of `channels`:
    "fp4" (one scale per 16 channels), "fp4g32" (one per 32: the 68-byte
    indexer entry) or "bf16"."""

    def __init__(self, B: int, n_cap: int, channels: int, dtype: str):
        self.B, self.n_cap, self.channels, self.dtype = B, n_cap, channels, dtype
        if dtype in ("fp4", "fp4g32"):
            self.codes = np.zeros((B, n_cap, channels // 2), np.uint8)
            self.scales = np.zeros((B, n_cap, channels // (16 if dtype == "fp4" else 32)), np.uint8)
            self.bf16 = None
        elif dtype == "bf16":
            self.codes = self.scales = None
            self.bf16 = np.zeros((B, n_cap, channels), np.uint16)
        else:
            raise ValueError(dtype)

    @property
    def dtype_code(self) -> int:
        return {"fp4": CACHE_FP4, "fp4g32": CACHE_FP4_G32, "bf16": CACHE_BF16}[self.dtype]

    def values(self) -> np.ndarray:
        """Decoded fp64 entries [B][n_cap][channels]."""
        if self.dtype != "bf16":
            return fp4_decode(self.codes, self.scales)
        return (self.bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def compress(x, pos0, w, w_idx, main: Cache, idx: Cache, r: int, theta: float, rope_dims: int = 64,
             diagnostics: bool = False):
    """a1: merge + RoPE + encode into `main`, then project + encode into `idx`.
    x [B][T][D] bf16 bits, pos0 [B] int64, w [r][D] fp32, w_idx [D][Ci] bf16 bits."""
    x = _c(x, np.uint16)
    pos0 = _c(pos0, np.int64)
    w = _c(w, np.float32)
    w_idx = _c(w_idx, np.uint16)
    B, T, D = x.shape
    Ci = w_idx.shape[1]
    M = T // r
    diag = {}
    if diagnostics:
        for k, n in (("pre_main", D), ("mag_main", D), ("pre_idx", Ci), ("mag_idx", Ci)):
            diag[k] = np.zeros((B, M, n), np.float64)
    if idx.dtype == "fp4g32" and main.dtype != "fp4":
        raise ValueError("the 68-byte indexer entry goes with an FP4 main cache")
    code = idx.dtype_code if idx.dtype == "fp4g32" else main.dtype_code
    rc = lib().orc_compress(B, T, D, Ci, rope_dims, r, float(theta), code,
                            _p(x), _p(pos0), _p(w), _p(w_idx), main.n_cap,
                            _p(main.codes), _p(main.scales), _p(main.bf16),
                            _p(idx.codes), _p(idx.scales), _p(idx.bf16),
                            _p(diag.get("pre_main")), _p(diag.get("mag_main")),
                            _p(diag.get("pre_idx")), _p(diag.get("mag_idx")))
    if rc != 0:
        raise ValueError("orc_compress rejected its arguments (%d)" % rc)
    return diag


def index_topk(idx: Cache, n_entries, q_idx, q_pos, r: int, k: int, head_w=None, hsi_blocks: int = 0,
               hsi_block: int = 8, pool=None, want_pool: bool = False, want_scores: bool = False,
               q_fp4: bool = False):
    """a3-a6.  q_idx [B][Tq][H][Ci] bf16 bits, q_pos [B][Tq] int64; q_fp4: score with
    each head's query encoded to FP4 (E2M1, E4M3 per 16 channels) and read back.
    Returns (topk [B][Tq][k] int32, pool [B][Tq][hsi_blocks] or None, scores or None)."""
    q_idx = _c(q_idx, np.uint16)
    B, Tq, H, Ci = q_idx.shape
    n_entries = _c(n_entries, np.int32)
    q_pos = _c(q_pos, np.int64)
    hw = None if head_w is None else _c(head_w, np.float32)
    pl = None if pool is None else _c(pool, np.int32)
    topk = np.zeros((B, Tq, k), np.int32)
    pool_out = np.zeros((B, Tq, hsi_blocks), np.int32) if want_pool else None
    scores = np.zeros((B, Tq, idx.n_cap), np.float64) if want_scores else None
    rc = lib().orc_index_topk_q(B, Tq, H, Ci, r, idx.dtype_code, idx.n_cap, _p(idx.codes),
                                _p(idx.scales), _p(idx.bf16), _p(n_entries), _p(q_idx), int(bool(q_fp4)), _p(hw),
                                _p(q_pos), k, hsi_blocks, hsi_block, _p(pl), _p(topk), _p(pool_out),
                                _p(scores))
    if rc != 0:
        raise ValueError("orc_index_topk rejected its arguments (%d)" % rc)
    return topk, pool_out, scores


def _swa(swa):
    """Window rows: uint16 [B][S][D] bf16 bits, or uint8 [B][S][D + D/32] MXFP8 rows."""
    if swa.dtype == np.uint8:
        return _c(swa, np.uint8), SWA_MXFP8
    return _c(swa, np.uint16), SWA_BF16


def attend(main: Cache, n_entries, q, topk, swa, swa_len, swa_pos0, q_pos, window: int, scale: float,
           want_lse: bool = False):
    """a7.  q [B][Tq][Hm][D] bf16 bits, topk [B][Tq][k], swa [B][S][D] bf16 bits (uint16) or
    [B][S][D + D/32] MXFP8 rows (uint8).  Returns out [B][Tq][Hm][D] fp64 (and lse [B][Tq][Hm])."""
    q = _c(q, np.uint16)
    B, Tq, Hm, D = q.shape
    topk = _c(topk, np.int32)
    k = topk.shape[-1]
    swa, fmt = _swa(swa)
    S = swa.shape[1]
    out = np.zeros((B, Tq, Hm, D), np.float64)
    lse = np.zeros((B, Tq, Hm), np.float64) if want_lse else None
    rc = lib().orc_attend(B, Tq, Hm, D, main.dtype_code, main.n_cap, _p(main.codes), _p(main.scales),
                          _p(main.bf16), _p(_c(n_entries, np.int32)), _p(q), _p(topk), k, _p(swa), fmt, S,
                          _p(_c(swa_len, np.int32)), _p(_c(swa_pos0, np.int64)), _p(_c(q_pos, np.int64)),
                          window, float(scale), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("orc_attend rejected its arguments (%d)" % rc)
    return (out, lse) if want_lse else out


def attend_dense(main: Cache, n_entries, q, swa, swa_len, swa_pos0, q_pos, r: int, window: int,
                 scale: float):
    q = _c(q, np.uint16)
    B, Tq, Hm, D = q.shape
    swa, fmt = _swa(swa)
    S = swa.shape[1]
    out = np.zeros((B, Tq, Hm, D), np.float64)
    rc = lib().orc_attend_dense(B, Tq, Hm, D, r, main.dtype_code, main.n_cap, _p(main.codes),
                                _p(main.scales), _p(main.bf16), _p(_c(n_entries, np.int32)), _p(q),
                                _p(swa), fmt, S, _p(_c(swa_len, np.int32)), _p(_c(swa_pos0, np.int64)),
                                _p(_c(q_pos, np.int64)), window, float(scale), _p(out))
    if rc != 0:
        raise ValueError("orc_attend_dense rejected its arguments (%d)" % rc)
    return out


# ------------------------------------------------------ cross-layer modes ----

def layer_modes(schedule):
    """a8: for a [(layer, mode)] schedule, map each layer to (mode, index source
    layer).  A Reuse layer reads the top-k of the latest earlier Full/Reindex
    layer; Full/Reindex layers publish their own."""
    out, latest = {}, None
    for layer, mode in schedule:
        if mode in ("full", "reindex"):
            latest = layer
            out[layer] = (mode, layer)
        elif mode == "reuse":
            if latest is None:
                raise ValueError("Reuse layer %d has no earlier indexing layer" % layer)
            out[layer] = (mode, latest)
        else:
            raise ValueError(mode)
    return out


class GroupState:
    """State shared by the layers of one cross-layer group (hn.213312.xyz
    sec. 2.3.2 and the access table of sec. 3.2): the main-KV and indexer-K
    caches the Full layer writes, the entry counts, and the latest published
    top-k and HSI pool."""

    def __init__(self, main: Cache, idx: Cache, n_entries, r: int, k: int, hsi_blocks: int = 0,
                 theta: float = 1e4):
        self.main, self.idx = main, idx
        self.n_entries = np.array(n_entries, np.int32)
        self.r, self.k, self.hsi_blocks, self.theta = r, k, hsi_blocks, theta
        self.topk = None
        self.pool = None


def layer(mode: str, st: GroupState, q_pos, q, swa, swa_len, swa_pos0, window: int, scale: float,
          q_idx=None, x=None, pos0=None, w=None, w_idx=None):
    """a8, one layer under its mode, following the access table:
    full    -- compress the step's tokens (when x is given), index every
               visible entry, publish top-k (and the HSI pool when the group
               has one), attend;
    reindex -- index the published pool's entries with this layer's q_idx,
               publish top-k, attend; no cache writes;
    reuse   -- attend with the latest published top-k; reads no indexer and
               writes nothing.
    Returns the attention output [B][Tq][Hm][D]."""
    if mode == "full":
        if x is not None:
            compress(x, pos0, w, w_idx, st.main, st.idx, st.r, st.theta)
            T = np.asarray(x).shape[1]
            st.n_entries = (np.asarray(pos0, np.int64) // st.r + T // st.r).astype(np.int32)
        st.topk, st.pool, _ = index_topk(st.idx, st.n_entries, q_idx, q_pos, st.r, st.k,
                                         hsi_blocks=st.hsi_blocks, want_pool=st.hsi_blocks > 0)
    elif mode == "reindex":
        if st.pool is None:
            raise ValueError("Reindex needs a published HSI pool")
        st.topk, _, _ = index_topk(st.idx, st.n_entries, q_idx, q_pos, st.r, st.k, hsi_blocks=st.hsi_blocks,
                                   pool=st.pool)
    elif mode == "reuse":
        if st.topk is None:
            raise ValueError("Reuse needs a published top-k")
    else:
        raise ValueError(mode)
    return attend(st.main, st.n_entries, q, st.topk, swa, swa_len, swa_pos0, q_pos, window, scale)
