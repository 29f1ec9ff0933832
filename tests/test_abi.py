"""Host-side checks of the C ABI: the library builds and exports every symbol
declared in include/*.h, page sizes follow the documented layout, and bad
arguments are rejected before any launch (no GPU needed: every call below
fails validation, so nothing is launched)."""
import ctypes as C
import glob
import os
import re

import numpy as np
import pytest
import torch

import compressed_sparse_attention_07_gb300 as csa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"CSA2_API\s+[\w\s\*]+?\b(csa2_\w+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = csa.load()
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_page_bytes_follow_layout():
    lib = csa.load()
    assert lib.csa2_page_bytes(512, csa.CACHE_FP4, 0) == 64 * 256
    assert lib.csa2_page_bytes(512, csa.CACHE_FP4, 1) == 64 * 32
    assert lib.csa2_page_bytes(128, csa.CACHE_FP4, 0) == 64 * 64
    assert lib.csa2_page_bytes(128, csa.CACHE_FP4, 1) == 64 * 8
    assert lib.csa2_page_bytes(512, csa.CACHE_BF16, 0) == 64 * 1024
    assert lib.csa2_page_bytes(512, csa.CACHE_BF16, 1) == 0
    # 288 B per main entry and 72 B per indexer entry in FP4
    assert (lib.csa2_page_bytes(512, 0, 0) + lib.csa2_page_bytes(512, 0, 1)) // 64 == 288
    assert (lib.csa2_page_bytes(128, 0, 0) + lib.csa2_page_bytes(128, 0, 1)) // 64 == 72


def test_status_strings():
    for code in (0, 1, 2, 3, 4, 16, 17, 18, 19):
        assert csa.status_string(code) != "unknown status"
    assert csa.status_string(999) == "unknown status"


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fake_cache(channels, dtype=csa.CACHE_FP4):
    return csa._CacheDesc(FAKE, FAKE if dtype == csa.CACHE_FP4 else None, FAKE, 4, 8, channels, 0)


def test_validation_rejects_before_launch():
    lib = csa.load()
    cfg = csa.Cfg(ratio=2)
    m, i = _fake_cache(512), _fake_cache(128)
    # no configuration
    assert lib.csa2_compress(None, 1, 2, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None, None) == 1
    # unsupported model size
    bad = csa.Cfg(ratio=2)
    bad.dim = 256
    assert lib.csa2_compress(C.byref(bad), 1, 2, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None,
                             None) == 2
    bad = csa.Cfg(ratio=3)
    assert lib.csa2_attend(C.byref(bad), 1, 1, FAKE, C.byref(m), FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 1.0, FAKE,
                           None, None, None) == 2
    # T not a multiple of r
    assert lib.csa2_compress(C.byref(cfg), 1, 3, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None,
                             None) == 1
    # wrong channel count for the indexer cache
    assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(m), FAKE, None,
                             None) == 1
    # workspace too small for one query
    need = lib.csa2_index_workspace_bytes(C.byref(cfg), 1, 1, 256, 0)
    assert need >= 256 * 4
    assert lib.csa2_index_topk(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, 256, None, FAKE, None, FAKE,
                               need - 1, None, None) == 4
    # more entries than the cache can hold
    assert lib.csa2_index_topk(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, 4 * 64 + 1, None, FAKE, None,
                               FAKE, 1 << 30, None, None) == 4
    # pool and pool_out together, or HSI outputs without HSI blocks
    hcfg = csa.Cfg(ratio=1, hsi_blocks=16)
    assert lib.csa2_index_topk(C.byref(hcfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, 256, FAKE, FAKE, FAKE, FAKE,
                               1 << 30, None, None) == 1
    assert lib.csa2_index_topk(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, 256, None, FAKE, FAKE, FAKE,
                               1 << 30, None, None) == 1
    # unaligned workspace
    assert lib.csa2_index_topk(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, 256, None, FAKE, None,
                               FAKE + 4, 1 << 30, None, None) == 1
    # window rows required when window > 0
    assert lib.csa2_attend(C.byref(cfg), 1, 1, FAKE, C.byref(m), FAKE, FAKE, None, 0, None, None, FAKE, 1.0, FAKE,
                           None, None, None) == 1
    # NaN scale
    assert lib.csa2_attend(C.byref(cfg), 1, 1, FAKE, C.byref(m), FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE,
                           float("nan"), FAKE, None, None, None) == 1
    # Reindex without a pool
    st = csa._GroupState(m, i, FAKE, 256, 0, FAKE, None, FAKE, 1 << 30, None)
    io = csa._LayerIO()
    assert lib.csa2_layer(C.byref(hcfg), csa.MODE_REINDEX, C.byref(st), C.byref(io), None) == 1
    assert lib.csa2_layer(C.byref(hcfg), 7, C.byref(st), C.byref(io), None) == 1
    # empty batches are a no-op
    assert lib.csa2_compress(C.byref(cfg), 0, 2, None, None, None, None, None, None, None, None, None) == 0


def test_paged_round_trip_on_host():
    """upload / download through the documented layout (CPU tensors)."""
    import oracle
    import synth
    from tests import _paged

    for dtype, chans in (("fp4", 512), ("fp4", 128), ("bf16", 512), ("bf16", 128)):
        cd = csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16
        order = _paged.page_order(1, 3 * 3 + 2)[:9]
        pc = csa.PagedCache(3, 150, chans, cd, device="cpu", page_order=order, spare_pages=2)
        oc = oracle.Cache(3, 150, chans, dtype)
        g = synth.rng(1, "rt")
        if dtype == "fp4":
            oc.codes[:], oc.scales[:] = g.integers(0, 256, oc.codes.shape), g.integers(0, 256, oc.scales.shape)
        else:
            oc.bf16[:] = g.integers(0, 65536, oc.bf16.shape)
        _paged.upload(pc, oc)
        a, b = _paged.download(pc, 150)
        if dtype == "fp4":
            np.testing.assert_array_equal(a, oc.codes)
            np.testing.assert_array_equal(b, oc.scales)
            # spot-check the documented address of one entry
            bj, j = 2, 131
            page = int(pc.block_table[bj, j // 64])
            slot = j % 64
            if chans == 512:
                got = pc.data[page, slot * 256:(slot + 1) * 256].numpy()
            else:
                got = np.concatenate([pc.data[page, (c * 64 + slot) * 16:(c * 64 + slot + 1) * 16].numpy()
                                      for c in range(4)])
            np.testing.assert_array_equal(got, oc.codes[bj, j])
        else:
            np.testing.assert_array_equal(a, oc.bf16)


def test_page_bytes_of_the_68_byte_indexer_entry():
    lib = csa.load()
    assert lib.csa2_page_bytes(128, csa.CACHE_FP4_S32, 0) == 64 * 64
    assert lib.csa2_page_bytes(128, csa.CACHE_FP4_S32, 1) == 64 * 4
    assert (lib.csa2_page_bytes(128, csa.CACHE_FP4_S32, 0) + lib.csa2_page_bytes(128, csa.CACHE_FP4_S32, 1)) // 64 == 68
    assert lib.csa2_page_bytes(16, csa.CACHE_FP4_S32, 0) == 0  # channels not a multiple of 32


def test_format_flags_are_validated():
    lib = csa.load()
    m, i = _fake_cache(512), _fake_cache(128)
    # an unknown flag, or the 68-byte indexer entry on a bf16 cache
    for cfg in (csa.Cfg(formats=8), csa.Cfg(cache_dtype=csa.CACHE_BF16, formats=csa.FMT_IDX_68B)):
        assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None,
                                 None) == 1
    # 68-byte entries need the indexer cache's scale pages
    cfg = csa.Cfg(formats=csa.FMT_IDX_68B)
    i_noscale = csa._CacheDesc(FAKE, None, FAKE, 4, 8, 128, 0)
    assert lib.csa2_index_topk(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i_noscale), FAKE, 256, None, FAKE,
                               None, FAKE, 1 << 30, None, None) == 1
    # MXFP8 window rows go through the row-tile attention only (top-k + window <= 6 tiles of 128)
    big = csa.Cfg(topk=1024, window=128, formats=csa.FMT_SWA_FP8)
    assert lib.csa2_attend(C.byref(big), 1, 1, FAKE, C.byref(m), FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 1.0, FAKE,
                           None, None, None) == 2
    # swa_encode: rows must be 16-byte aligned and T <= S; empty is a no-op
    assert lib.csa2_swa_encode(1, 4, FAKE, FAKE, FAKE + 8, 8, None, None) == 1
    assert lib.csa2_swa_encode(1, 9, FAKE, FAKE, FAKE, 8, None, None) == 1
    assert lib.csa2_swa_encode(0, 4, None, None, None, 8, None, None) == 0


def test_misaligned_pointers_are_rejected_before_launch():
    lib = csa.load()
    cfg = csa.Cfg(ratio=2)
    m, i = _fake_cache(512), _fake_cache(128)
    # compressor: x needs 4 bytes, w_idx 8, pos0 8
    assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE + 2, FAKE, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None,
                             None) == 1
    assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE, FAKE, FAKE, FAKE + 4, C.byref(m), C.byref(i), FAKE, None,
                             None) == 1
    assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE, FAKE + 4, FAKE, FAKE, C.byref(m), C.byref(i), FAKE, None,
                             None) == 1
    # a block table off its 4-byte boundary
    bt = csa._CacheDesc(FAKE, FAKE, FAKE + 2, 4, 8, 128, 0)
    assert lib.csa2_compress(C.byref(cfg), 1, 2, FAKE, FAKE, FAKE, FAKE, C.byref(m), C.byref(bt), FAKE, None,
                             None) == 1
    # indexer: q_idx needs 16 bytes, q_pos 8, the outputs 4
    args = dict(q_idx=FAKE, head_w=None, q_pos=FAKE, topk_out=FAKE, status=None)
    def index(**kw):
        a = dict(args, **kw)
        return lib.csa2_index_topk(C.byref(cfg), 1, 1, a["q_idx"], a["head_w"], a["q_pos"], C.byref(i), FAKE, 256,
                                   None, a["topk_out"], None, FAKE, 1 << 30, a["status"], None)
    for kw in (dict(q_idx=FAKE + 8), dict(q_pos=FAKE + 4), dict(head_w=FAKE + 2), dict(topk_out=FAKE + 2),
               dict(status=FAKE + 1)):
        assert index(**kw) == 1, kw
    # attention: q and out need 16 bytes, swa_pos0 8
    def attend(q=FAKE, out=FAKE, swa_pos0=FAKE):
        return lib.csa2_attend(C.byref(cfg), 1, 1, q, C.byref(m), FAKE, FAKE, FAKE, 1, FAKE, swa_pos0, FAKE, 1.0,
                               out, None, None, None)
    assert attend(q=FAKE + 8) == 1
    assert attend(out=FAKE + 4) == 1
    assert attend(swa_pos0=FAKE + 4) == 1
    # gather: ids and out need 4 bytes
    assert lib.csa2_gather_dequant(C.byref(m), csa.CACHE_FP4, 1, 1, FAKE + 2, FAKE, None, None) == 1
    assert lib.csa2_gather_dequant(C.byref(m), csa.CACHE_FP4, 1, 1, FAKE, FAKE + 2, None, None) == 1


def test_paged_round_trip_of_68_byte_indexer_entries():
    import oracle
    import synth
    from tests import _paged

    order = _paged.page_order(2, 3 * 3 + 2)[:9]
    pc = csa.PagedCache(3, 150, 128, csa.CACHE_FP4_S32, device="cpu", page_order=order, spare_pages=2)
    oc = oracle.Cache(3, 150, 128, "fp4g32")
    g = synth.rng(2, "rt32")
    oc.codes[:], oc.scales[:] = g.integers(0, 256, oc.codes.shape), g.integers(0, 256, oc.scales.shape)
    _paged.upload(pc, oc)
    a, b = _paged.download(pc, 150)
    np.testing.assert_array_equal(a, oc.codes)
    np.testing.assert_array_equal(b, oc.scales)
    bj, j = 1, 77  # documented address of one entry's scales: slot s at s*4
    page, slot = int(pc.block_table[bj, j // 64]), j % 64
    np.testing.assert_array_equal(pc.scales[page, slot * 4:slot * 4 + 4].numpy(), oc.scales[bj, j])


def test_layer_checks_every_stage_before_the_first_launch():
    """csa2_layer in Full mode: a bad indexer or attention argument is found
    before the compressor is launched (no GPU here, so a launch would come
    back as CSA2_ERR_CUDA instead of the argument error)."""
    lib = csa.load()
    cfg = csa.Cfg(ratio=1, hsi_blocks=16)
    m, i = _fake_cache(512), _fake_cache(128)
    st = csa._GroupState(m, i, FAKE, 256, 0, FAKE, FAKE, FAKE, 1 << 30, None)

    def io(**kw):
        d = dict(B=1, Tq=1, q_pos=FAKE, T=1, x=FAKE, pos0=FAKE, merge_w=FAKE, w_idx=FAKE, q_idx=FAKE, head_w=None,
                 q=FAKE, swa=FAKE, S=1, swa_len=FAKE, swa_pos0=FAKE, scale=1.0, out=FAKE, lse=None)
        d.update(kw)
        return csa._LayerIO(**d)

    assert lib.csa2_layer(C.byref(cfg), csa.MODE_FULL, C.byref(st), C.byref(io(q_idx=FAKE + 8)), None) == 1
    assert lib.csa2_layer(C.byref(cfg), csa.MODE_FULL, C.byref(st), C.byref(io(q_idx=None)), None) == 1
    assert lib.csa2_layer(C.byref(cfg), csa.MODE_FULL, C.byref(st), C.byref(io(out=FAKE + 4)), None) == 1
    assert lib.csa2_layer(C.byref(cfg), csa.MODE_FULL, C.byref(st), C.byref(io(scale=float("nan"))), None) == 1
    small = csa._GroupState(m, i, FAKE, 256, 0, FAKE, FAKE, FAKE, 16, None)
    assert lib.csa2_layer(C.byref(cfg), csa.MODE_FULL, C.byref(small), C.byref(io()), None) == 4
    # Reindex checks its indexer and attention arguments the same way
    assert lib.csa2_layer(C.byref(cfg), csa.MODE_REINDEX, C.byref(st), C.byref(io(q_idx=FAKE + 8)), None) == 1


def test_static_entry_point_reports_configuration_errors_first():
    """csa2_index_topk_static applies csa2_index_topk's checks in the same
    order: an unsupported configuration is reported as such even when the
    request would also be too large for the static array."""
    lib = csa.load()
    lib.csa2_index_topk_static.restype = C.c_int32
    i = csa._CacheDesc(FAKE, FAKE, FAKE, 1 << 20, 8, 128, 0)
    big = (64 << 20) // 4
    bad = csa.Cfg(ratio=3)
    assert lib.csa2_index_topk_static(C.byref(bad), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, big, None, FAKE, None,
                                      None, None) == 2
    bad = csa.Cfg(topk=0)
    assert lib.csa2_index_topk_static(C.byref(bad), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, big, None, FAKE, None,
                                      None, None) == 2
    cfg = csa.Cfg(ratio=1)
    assert lib.csa2_index_topk_static(C.byref(cfg), 1, 1, FAKE + 8, None, FAKE, C.byref(i), FAKE, big, None, FAKE,
                                      None, None, None) == 1
    assert lib.csa2_index_topk_static(C.byref(cfg), 1, 1, FAKE, None, FAKE, C.byref(i), FAKE, big, None, FAKE, None,
                                      None, None) == 4
