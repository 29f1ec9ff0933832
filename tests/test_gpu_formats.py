"""GPU-vs-oracle parity of the pages' own storage formats: the 68-byte
indexer entry (FP4 with one E4M3 scale per 32 channels; hn.213312.xyz
sec. 3.1) through the compressor, the indexer in every mode and the entry
decoder, and the FP8 window rows (sec. 2.4.4, read as OCP MXFP8) through
their encoder and the attention."""
import math

import numpy as np
import pytest
import torch

import compressed_sparse_attention_07_gb300 as csa
import oracle
import synth
from tests import _paged
from tests import _parity as P
from tests.test_gpu_stages import _check_compress, _main_caches

pytestmark = pytest.mark.gpu

D, CI, H, HM = 512, 128, 32, 64


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ----------------------------------------------------- MXFP8 window rows ----

def _window_rows(seed, B, T):
    """bf16 rows with blocks of very different magnitudes: ordinary, tiny
    (subnormal bf16), huge, all-zero, exact E4M3 ties, and negative values
    that round to zero next to a large block maximum."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((B, T, D))
    mags = np.exp(g.uniform(-30, 30, size=(B, T, D // 32)))
    x *= np.repeat(mags, 32, axis=-1)
    x[0, 0, 0:32] = 0.0
    x[0, 1, 32:64] = g.standard_normal(32) * 1e-39  # bf16 subnormals
    e4 = [oracle.e4m3_value(c) for c in range(0x7F)]
    x[0, 2, 64] = 300.0  # block scale 2^0: ties between E4M3 neighbours below
    for i in range(1, 32):
        x[0, 2, 64 + i] = (e4[40 + i] + e4[41 + i]) / 2 * (-1) ** i
    x[0, 3, 96] = 1000.0
    x[0, 3, 97:128] = -1e-6  # rounds to zero: +0
    bits = np.vectorize(oracle.bf16_round, otypes=[np.uint16])(x)
    return bits


def test_swa_encode_bit_exact_and_placed_by_row0():
    B, T, S = 3, 20, 40
    bits = _window_rows(41, B, T)
    row0 = np.array([0, 20, 5], np.int64)
    rows = torch.full((B, S, csa.SWA_FP8_ROW), 0xAB, dtype=torch.uint8, device="cuda")
    st = _status()
    csa.swa_encode(_paged.dev(bits), _paged.dev(row0), rows, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = rows.cpu().numpy()
    want = oracle.swa_encode(bits)
    for b in range(B):
        np.testing.assert_array_equal(got[b, row0[b]:row0[b] + T], want[b], err_msg="sequence %d" % b)
        keep = np.ones(S, bool)
        keep[row0[b]:row0[b] + T] = False
        assert (got[b, keep] == 0xAB).all()
    # a placement past the end is skipped and reported
    rows2 = torch.full((B, S, csa.SWA_FP8_ROW), 0xAB, dtype=torch.uint8, device="cuda")
    st = _status()
    csa.swa_encode(_paged.dev(bits), _paged.dev(np.array([0, 21, 5], np.int64)), rows2, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 17  # CSA2_ERR_BAD_INDEX
    g2 = rows2.cpu().numpy()
    assert (g2[1] == 0xAB).all()
    np.testing.assert_array_equal(g2[2, 5:25], want[2])


@pytest.mark.parametrize("dtype", ["fp4", "bf16"])
def test_attend_over_mxfp8_window_rows(dtype):
    """The attention test's shapes with the window rows in MXFP8 (encoded on
    the GPU, bit-checked, then read by the attention), including rows whose
    block scales lie below the f16 range (decoded through fp32) and large
    rows (values within f16 range, the limit of the f16 MMA operands)."""
    B, N, Tq, k, W = 3, 700, 3, 512, 128
    oc, pc = _main_caches(B, N, dtype, seed=42)
    g = synth.rng(42, "ids")
    topk = np.full((B, Tq, k), -1, np.int32)
    for b in range(B):
        for t in range(Tq):
            n = [512, 300, 0][(b + t) % 3]
            topk[b, t, :n] = np.sort(g.choice(N, size=n, replace=False))
    q = synth.normal_bf16(synth.rng(42, "q"), (B, Tq, HM, D))
    S = 200
    bits = synth.normal_bf16(synth.rng(42, "swa"), (B, S, D))
    f = oracle.bf16_bits_to_f64(bits)
    f[1, 40:60] *= 2.0 ** -40  # block scales below f16's range
    f[2, 10:30] *= 2.0 ** 12   # large values, still finite in f16
    bits = np.vectorize(oracle.bf16_round, otypes=[np.uint16])(f)
    rows = torch.zeros((B, S, csa.SWA_FP8_ROW), dtype=torch.uint8, device="cuda")
    st = _status()
    csa.swa_encode(_paged.dev(bits), _paged.dev(np.zeros(B, np.int64)), rows, status=st)
    orows = oracle.swa_encode(bits)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rows.cpu().numpy(), orows)
    swa_pos0 = np.array([0, 1000, 5000], np.int64)
    swa_len = np.array([150, 200, 60], np.int32)
    q_pos = np.array([[3, 100, 149], [1199, 1130, 1050], [5059, 5100, 4990]], np.int64)
    n_ent = np.array([N, N, N], np.int32)
    cfg = csa.Cfg(ratio=2, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, topk=k, window=W,
                  formats=csa.FMT_SWA_FP8)
    out = torch.empty((B, Tq, HM, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Tq, HM), dtype=torch.float32, device="cuda")
    csa.attend(cfg, _paged.dev(q), pc, _paged.dev(n_ent), _paged.dev(topk), rows, _paged.dev(swa_len),
               _paged.dev(swa_pos0), _paged.dev(q_pos), out, lse=lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_out, o_lse = oracle.attend(oc, n_ent, q, topk, orows, swa_len, swa_pos0, q_pos, W, 1 / math.sqrt(D),
                                 want_lse=True)
    err = P.attention_rel_err(out.cpu().numpy(), o_out)
    assert err <= P.ATT_TOL, err
    lg = lse.cpu().numpy()
    fin = np.isfinite(o_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    # the large rows put logits near 1e4: the fp32 LSE then carries a few ulps of that size
    np.testing.assert_allclose(lg[fin], o_lse[fin], rtol=2e-6, atol=1e-3)
    print("attend %s over MXFP8 window rows: max row rel err %.3g" % (dtype, err))


# ---------------------------------------------- 68-byte indexer entries ----

def test_compress_into_68_byte_indexer_entries():
    B, T, r = 3, 64, 2
    pos0 = np.array([0, 130, 4094], np.int64)
    x = synth.normal_bf16(synth.rng(43, "x"), (B, T, D))
    w = synth.merge_weights(synth.rng(43, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(43, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    M = T // r
    cap = int(pos0.max() // r + M)
    om, oi = oracle.Cache(B, cap, D, "fp4"), oracle.Cache(B, cap, CI, "fp4g32")
    diag = oracle.compress(x, pos0, w, w_idx, om, oi, r, 1e4, diagnostics=True)
    cfg = csa.Cfg(ratio=r, formats=csa.FMT_IDX_68B)
    pm, pi = _paged.cache_pair(B, cap, D, "fp4", 43), _paged.cache_pair(B, cap, CI, "fp4g32", 44)
    n_ent = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = _status()
    csa.compress(cfg, _paged.dev(x), _paged.dev(pos0), _paged.dev(w), _paged.dev(w_idx), pm, pi, n_ent, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exc = _check_compress(om, oi, pm, pi, diag, pos0, r, M, "fp4")
    print("compress into 68-byte indexer entries: %d near-boundary codes excused" % exc)


def _g32_caches(B, N, seed):
    """68-byte entries whose scores are exact: integer E2M1 codes and scales
    that are powers of two (0.25 .. 2), different in each 32-channel block."""
    oc = oracle.Cache(B, N, CI, "fp4g32")
    g = synth.rng(seed, "idx32")
    pick = synth.rng(seed, "dup").integers(0, 60, size=(B, N))  # repeated entries: ties straddle the k-th place
    for b in range(B):
        codes, _ = synth.integer_fp4_bytes(g, 60, CI)
        scales = np.array([0x28, 0x30, 0x38, 0x40], np.uint8)[g.integers(0, 4, size=(60, CI // 32))]
        oc.codes[b], oc.scales[b] = codes[pick[b]], scales[pick[b]]
    pc = _paged.cache_pair(B, N, CI, "fp4g32", seed)
    _paged.upload(pc, oc)
    return oc, pc


def _index(cfg, pc, q_idx, q_pos, n_ent, N, head_w=None, pool=None, want_pool=False):
    B, Tq = q_idx.shape[:2]
    topk = torch.full((B, Tq, cfg.topk), -7, dtype=torch.int32, device="cuda")
    pool_out = torch.full((B, Tq, cfg.hsi_blocks), -7, dtype=torch.int32, device="cuda") if want_pool else None
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, Tq, N, reindex=pool is not None), dtype=torch.uint8,
                     device="cuda")
    st = _status()
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pc, _paged.dev(n_ent), N, topk, ws,
                   head_w=None if head_w is None else _paged.dev(head_w),
                   pool=None if pool is None else _paged.dev(pool), pool_out=pool_out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return topk.cpu().numpy(), (pool_out.cpu().numpy() if want_pool else None)


@pytest.mark.parametrize("Tq", [1, 2, 5])
def test_index_on_68_byte_entries_full_and_reindex_bit_exact(Tq):
    """Full with the HSI pool (one query per group, or a multi-query block of
    2 or 5 positions sharing each tile), then Reindex over that pool (gather
    mode): bit-exact top-k and pools."""
    B, N, k, nb = 3, 5000, 512, 96
    oc, pc = _g32_caches(B, N, 45 + Tq)
    q_idx = synth.integer_bf16(synth.rng(45, "q%d" % Tq), (B, Tq, H, CI), -1, 1)
    n_ent = np.array([N, 3333, 900], np.int32)
    q_pos = np.stack([n - Tq + np.arange(Tq) for n in n_ent]).astype(np.int64)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb, formats=csa.FMT_IDX_68B)
    g_top, g_pool = _index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, 1, k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)
    q2 = synth.integer_bf16(synth.rng(46, "q%d" % Tq), (B, Tq, H, CI), -1, 1)
    r_top, _ = _index(cfg, pc, q2, q_pos, n_ent, N, pool=o_pool)
    o_rtop, _, _ = oracle.index_topk(oc, n_ent, q2, q_pos, 1, k, hsi_blocks=nb, pool=o_pool)
    np.testing.assert_array_equal(r_top, o_rtop)


def test_gather_dequant_of_68_byte_entries_bit_exact():
    B, N = 2, 300
    oc = oracle.Cache(B, N, CI, "fp4g32")
    g = synth.rng(47, "g32")
    for b in range(B):
        oc.codes[b], oc.scales[b] = synth.fp4_bytes(g, N, CI, 0x01, 0x7E, group=32)
    pc = _paged.cache_pair(B, N, CI, "fp4g32", 47)
    _paged.upload(pc, oc)
    ids = np.stack([np.arange(N), (np.arange(N) * 7) % N]).astype(np.int32)
    ids[1, 5] = -1
    out = torch.empty((B, N, CI), dtype=torch.float32, device="cuda")
    st = _status()
    csa.gather_dequant(pc, _paged.dev(ids), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    vals = oc.values()
    want = np.stack([vals[b][np.maximum(ids[b], 0)] for b in range(B)])
    want[1, 5] = 0.0
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), want)


# -------------------------------------------------- FP4 indexer queries ----

@pytest.mark.parametrize("dtype,Tq,mode", [("fp4", 2, "full"), ("fp4", 8, "full"), ("fp4", 5, "full"),
                                           ("fp4", 2, "reindex"), ("fp4g32", 5, "full"), ("bf16", 3, "full")])
def test_index_with_fp4_queries_bit_exact(dtype, Tq, mode):
    """FP4-encoded indexer queries (E2M1, E4M3 per 16 channels) on every
    scoring path: one query per group (Tq 2), runs of 4 (Tq 8), a multi-query
    block (Tq 5), Reindex gathers, 68-byte entries, a bf16 cache.  Queries
    are integers in [-5, 5], whose FP4 encodings are multiples of 1/16 (the
    group scales 0.8125, 0.6875, ...), and the cache values are multiples of
    1/4, so every score is exact and top-k and pools must match bit for bit."""
    B, N, k, nb = 2, 4000, 512, 80
    if dtype == "fp4g32":
        oc, pc = _g32_caches(B, N, 60 + Tq)
    else:
        oc = oracle.Cache(B, N, CI, dtype)
        g = synth.rng(60 + Tq, "int")
        pick = synth.rng(60 + Tq, "dup").integers(0, 50, size=(B, N))
        for b in range(B):
            if dtype == "fp4":
                c, s = synth.integer_fp4_bytes(g, 50, CI)
                oc.codes[b], oc.scales[b] = c[pick[b]], s[pick[b]]
            else:
                oc.bf16[b] = synth.integer_bf16(g, (50, CI), -6, 6)[pick[b]]
        pc = _paged.cache_pair(B, N, CI, dtype, 60 + Tq)
        _paged.upload(pc, oc)
    q_idx = synth.integer_bf16(synth.rng(61, "q%d" % Tq), (B, Tq, H, CI), -5, 5)
    n_ent = np.array([N, 2900], np.int32)
    q_pos = np.stack([n - Tq + np.arange(Tq) for n in n_ent]).astype(np.int64)
    fmt = csa.FMT_IDX_QFP4 | (csa.FMT_IDX_68B if dtype == "fp4g32" else 0)
    cfg = csa.Cfg(ratio=1, cache_dtype=csa.CACHE_BF16 if dtype == "bf16" else csa.CACHE_FP4, topk=k,
                  hsi_blocks=nb, formats=fmt)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, 1, k, hsi_blocks=nb, want_pool=True, q_fp4=True)
    if mode == "full":
        g_top, g_pool = _index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
        np.testing.assert_array_equal(g_pool, o_pool)
        np.testing.assert_array_equal(g_top, o_top)
    else:
        q2 = synth.integer_bf16(synth.rng(62, "q%d" % Tq), (B, Tq, H, CI), -5, 5)
        r_top, _ = _index(cfg, pc, q2, q_pos, n_ent, N, pool=o_pool)
        o_rtop, _, _ = oracle.index_topk(oc, n_ent, q2, q_pos, 1, k, hsi_blocks=nb, pool=o_pool, q_fp4=True)
        np.testing.assert_array_equal(r_top, o_rtop)
    # the FP4 queries change the selection against the bf16 queries
    b_top, _, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, 1, k)
    assert not np.array_equal(b_top, o_top)
