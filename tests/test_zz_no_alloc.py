"""csa2_index_topk_static: the indexer entry point for callers that cannot
allocate device memory (engines or plugin hosts that own every device byte,
decode loops that must not pay for cudaMalloc's synchronisation).  Its
scratch is a static array inside the library; the results must equal those
of csa2_index_topk with a caller-provided workspace, call after call.

Kept in a file that is collected last, so that a run stopping at the first
failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import compressed_sparse_attention_07_gb300 as csa
import synth
from tests import _paged
from tests.test_gpu_stages import _idx_caches

pytestmark = pytest.mark.gpu

H, CI = 32, 128


def _static(cfg, q_idx, q_pos, pc, n_ent, N, topk, pool_out, status):
    lib = csa.load()
    d = pc.desc()
    B, Tq = q_idx.shape[:2]
    return lib.csa2_index_topk_static(
        C.byref(cfg), B, Tq, C.c_void_p(q_idx.data_ptr()), None, C.c_void_p(q_pos.data_ptr()), C.byref(d),
        C.c_void_p(n_ent.data_ptr()), N, None, C.c_void_p(topk.data_ptr()),
        C.c_void_p(pool_out.data_ptr()) if pool_out is not None else None, C.c_void_p(status.data_ptr()),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(seed, B, N, integer):
    oc, pc = _idx_caches(B, N, "fp4", seed=seed, integer=integer, dup=integer)
    g = synth.rng(seed, "q")
    q_idx = synth.integer_bf16(g, (B, 2, H, CI), -1, 1) if integer else synth.normal_bf16(g, (B, 2, H, CI))
    q_pos = np.stack([np.full(B, N - 1), np.arange(B) * 97 + 40], 1).astype(np.int64)
    n_ent = np.full(B, N, np.int32)
    return pc, _paged.dev(q_idx), _paged.dev(q_pos), _paged.dev(n_ent)


def test_static_scratch_matches_workspace_entry_point_twice():
    lib = csa.load()
    lib.csa2_index_topk_static.restype = C.c_int32
    lib.csa2_index_static_scratch_bytes.restype = C.c_size_t
    assert lib.csa2_index_static_scratch_bytes() == 8 << 20
    cfg = csa.Cfg(ratio=1, topk=512, hsi_blocks=64)
    # two calls in a row with different data and sizes: the second must not
    # see anything the first left in the shared array
    for call, (seed, B, N, integer) in enumerate([(41, 3, 3000, True), (42, 5, 1900, False)]):
        pc, q_idx, q_pos, n_ent = _case(seed, B, N, integer)
        k = cfg.topk
        want_top = torch.full((B, 2, k), -9, dtype=torch.int32, device="cuda")
        want_pool = torch.full((B, 2, cfg.hsi_blocks), -9, dtype=torch.int32, device="cuda")
        ws = torch.empty(csa.index_workspace_bytes(cfg, B, 2, N), dtype=torch.uint8, device="cuda")
        csa.index_topk(cfg, q_idx, q_pos, pc, n_ent, N, want_top, ws, pool_out=want_pool)
        got_top = torch.full_like(want_top, -5)
        got_pool = torch.full_like(want_pool, -5)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _static(cfg, q_idx, q_pos, pc, n_ent, N, got_top, got_pool, st)
        torch.cuda.synchronize()
        assert rc == 0, csa.status_string(rc)
        assert int(st.item()) == 0
        assert torch.equal(got_top, want_top), "call %d: top-k differs" % call
        assert torch.equal(got_pool, want_pool), "call %d: HSI pool differs" % call


def test_static_scratch_rejects_oversized_requests():
    lib = csa.load()
    lib.csa2_index_topk_static.restype = C.c_int32
    cfg = csa.Cfg(ratio=1, topk=512, hsi_blocks=64)
    fake = C.c_void_p(0x10000)  # never dereferenced: the size check fails first
    d = csa._CacheDesc(0x10000, 0x10000, 0x10000, 1 << 16, 1 << 16, 128, 0)
    too_many = (8 << 20) // 4  # entries whose scores alone fill the array
    rc = lib.csa2_index_topk_static(C.byref(cfg), 1, 1, fake, None, fake, C.byref(d), fake, too_many, None, fake,
                                    fake, None, None)
    assert rc == 4  # CSA2_ERR_CAPACITY


def test_static_scratch_at_its_largest_accepted_size():
    """The largest sequence length whose per-query scratch (scores, HSI block
    maxima, key-range slots) fits the static array exactly: two queries run
    one after the other through the array and give the workspace entry
    point's results; one entry more is refused before any launch."""
    lib = csa.load()
    lib.csa2_index_topk_static.restype = C.c_int32
    cap = lib.csa2_index_static_scratch_bytes()
    cfg = csa.Cfg(ratio=1, topk=512, hsi_blocks=2048)
    lo, hi = 1, 4 << 20  # largest N with a per-query scratch of at most the array's size
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if csa.index_workspace_bytes(cfg, 1, 1, mid) <= cap:
            lo = mid
        else:
            hi = mid - 1
    N = lo
    assert csa.index_workspace_bytes(cfg, 1, 1, N) <= cap < csa.index_workspace_bytes(cfg, 1, 1, N + 1)
    B = 2
    pc, q_idx, q_pos, n_ent = _case(44, B, N, integer=False)
    q_idx, q_pos = q_idx[:, :1].contiguous(), q_pos[:, :1].contiguous()
    want_top = torch.full((B, 1, cfg.topk), -9, dtype=torch.int32, device="cuda")
    want_pool = torch.full((B, 1, cfg.hsi_blocks), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    csa.index_topk(cfg, q_idx, q_pos, pc, n_ent, N, want_top, ws, pool_out=want_pool)
    got_top = torch.full_like(want_top, -5)
    got_pool = torch.full_like(want_pool, -5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _static(cfg, q_idx, q_pos, pc, n_ent, N, got_top, got_pool, st)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    assert torch.equal(got_top, want_top) and torch.equal(got_pool, want_pool)
    fake = C.c_void_p(0x10000)  # never dereferenced: the size check fails first
    d = csa._CacheDesc(0x10000, 0x10000, 0x10000, 1 << 16, 1 << 16, 128, 0)
    rc = lib.csa2_index_topk_static(C.byref(cfg), B, 1, fake, None, fake, C.byref(d), fake, N + 1, None, fake, fake,
                                    None, None)
    assert rc == 4  # CSA2_ERR_CAPACITY


def test_static_scratch_with_single_queries_laid_end_to_end():
    """24 single queries of 20000 entries: the scorer lays their tiles end to
    end over one wave (CTA ranges crossing from one query into the next) in
    both entry points; the static one, whose array holds all 24 queries'
    scratch, gives the workspace entry point's results."""
    lib = csa.load()
    lib.csa2_index_topk_static.restype = C.c_int32
    cfg = csa.Cfg(ratio=1, topk=512, hsi_blocks=1024)
    B, N = 24, 20000
    assert csa.index_workspace_bytes(cfg, B, 1, N) <= lib.csa2_index_static_scratch_bytes()
    pc, q_idx, q_pos, n_ent = _case(45, B, N, integer=True)
    q_idx, q_pos = q_idx[:, :1].contiguous(), q_pos[:, :1].contiguous()
    want_top = torch.full((B, 1, cfg.topk), -9, dtype=torch.int32, device="cuda")
    want_pool = torch.full((B, 1, cfg.hsi_blocks), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    csa.index_topk(cfg, q_idx, q_pos, pc, n_ent, N, want_top, ws, pool_out=want_pool)
    got_top = torch.full_like(want_top, -5)
    got_pool = torch.full_like(want_pool, -5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _static(cfg, q_idx, q_pos, pc, n_ent, N, got_top, got_pool, st)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    assert torch.equal(got_top, want_top) and torch.equal(got_pool, want_pool)
