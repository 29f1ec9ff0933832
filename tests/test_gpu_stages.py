"""GPU-vs-oracle parity of each stage of the CSA2 path through the C ABI, at
sizes the oracle finishes in seconds that still span several tiles, pages
and ragged tails."""
import math

import numpy as np
import pytest
import torch

import compressed_sparse_attention_07_gb300 as csa
import oracle
import synth
from tests import _paged
from tests import _parity as P

pytestmark = pytest.mark.gpu

D, CI, H, HM = 512, 128, 32, 64


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------- dequant ----

@pytest.mark.parametrize("channels", [512, 128])
def test_dequant_bit_exact_every_code_and_scale(channels):
    """Every E2M1 code under every finite E4M3 scale decodes exactly."""
    B, n = 2, 254
    oc = oracle.Cache(B, n, channels, "fp4")
    codes = np.arange(channels // 2 * n * B, dtype=np.int64) % 256
    oc.codes[:] = codes.reshape(oc.codes.shape).astype(np.uint8)
    sc = np.arange(channels // 16 * n * B) % 254
    sc = np.where(sc >= 127, sc + 1, sc)  # skip 0x7F (NaN), keep 0x80..0xFE
    oc.scales[:] = sc.reshape(oc.scales.shape).astype(np.uint8)
    pc = _paged.cache_pair(B, n, channels, "fp4", seed=3)
    _paged.upload(pc, oc)
    ids = torch.from_numpy(np.stack([np.arange(n), np.arange(n)[::-1]]).astype(np.int32)).cuda()
    out = torch.empty((B, n, channels), dtype=torch.float32, device="cuda")
    st = _status()
    csa.gather_dequant(pc, ids, out, status=st)
    want = oc.values()
    want[1] = want[1][::-1]
    got = out.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    assert int(st.item()) == 0


def test_dequant_bf16_and_bad_page_status():
    oc = oracle.Cache(1, 100, 512, "bf16")
    oc.bf16[:] = synth.normal_bf16(synth.rng(5, "c"), oc.bf16.shape)
    pc = _paged.cache_pair(1, 100, 512, "bf16", seed=5)
    _paged.upload(pc, oc)
    ids = torch.arange(100, dtype=torch.int32, device="cuda").reshape(1, 100)
    out = torch.empty((1, 100, 512), dtype=torch.float32, device="cuda")
    csa.gather_dequant(pc, ids, out)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), oc.values()[0:1])
    # a block-table entry outside the pool is reported and the row reads as zeros
    pc.block_table[0, 1] = pc.num_pages + 5
    st = _status()
    csa.gather_dequant(pc, ids, out, status=st)
    assert int(st.item()) == 16  # CSA2_ERR_BAD_PAGE
    assert (out[0, 64:100] == 0).all()


# ------------------------------------------------------------ compress ----

def _compress_case(B, T, r, dtype, pos0, seed, theta=1e4, capacity=None):
    x = synth.normal_bf16(synth.rng(seed, "x"), (B, T, D))
    w = synth.merge_weights(synth.rng(seed, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(seed, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    pos0 = np.asarray(pos0, np.int64)
    M = T // r
    cap = capacity or int(pos0.max() // r + M)
    om, oi = oracle.Cache(B, cap, D, dtype), oracle.Cache(B, cap, CI, dtype)
    diag = oracle.compress(x, pos0, w, w_idx, om, oi, r, theta, diagnostics=True)
    cfg = csa.Cfg(ratio=r, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, rope_theta=theta)
    pm, pi = _paged.cache_pair(B, cap, D, dtype, seed), _paged.cache_pair(B, cap, CI, dtype, seed + 1)
    n_ent = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = _status()
    csa.compress(cfg, _paged.dev(x), _paged.dev(pos0), _paged.dev(w), _paged.dev(w_idx), pm, pi, n_ent, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert n_ent.cpu().tolist() == [int(p // r + M) for p in pos0]
    return om, oi, pm, pi, diag, cap


def _check_compress(om, oi, pm, pi, diag, pos0, r, M, dtype):
    B = len(pos0)
    gm, gms = _paged.download(pm, pm.capacity)
    gi, gis = _paged.download(pi, pi.capacity)
    rows = [np.arange(p // r, p // r + M) for p in pos0]
    tot_exc = 0
    for b in range(B):
        j = rows[b]
        if dtype == "fp4":
            u, e, bad = P.fp4_code_mismatches(gm[b, j], gms[b, j], om.codes[b, j], om.scales[b, j],
                                              diag["pre_main"][b], diag["mag_main"][b], P.MAIN_MARGIN)
            assert u == 0, "main codes differ away from decision boundaries"
            ok = ~bad
            u2, e2, _ = P.fp4_code_mismatches(gi[b, j][ok], gis[b, j][ok], oi.codes[b, j][ok], oi.scales[b, j][ok],
                                              diag["pre_idx"][b][ok], diag["mag_idx"][b][ok], P.IDX_MARGIN)
        else:
            u, e, bad = P.bf16_mismatches(gm[b, j], om.bf16[b, j], diag["pre_main"][b], diag["mag_main"][b],
                                          P.MAIN_MARGIN)
            assert u == 0
            ok = ~bad
            u2, e2, _ = P.bf16_mismatches(gi[b, j][ok], oi.bf16[b, j][ok], diag["pre_idx"][b][ok],
                                          diag["mag_idx"][b][ok], P.IDX_MARGIN)
        assert u2 == 0, "indexer K codes differ away from decision boundaries"
        tot_exc += e + e2
    return tot_exc


@pytest.mark.parametrize("dtype,r,T,pos0,theta", [
    ("fp4", 2, 2, [0, 130, 4094], 1e4),            # decode: one pair per sequence
    ("fp4", 2, 256, [0, 1048576], 1e4),            # prefill chunk, far positions
    ("fp4", 1, 1, [5, 262143, 64], 1.6e5),         # decoder decode step
    ("fp4", 1, 200, [0, 777], 1.6e5),              # ragged page tails
    ("bf16", 2, 64, [0, 2048], 1e4),
    ("bf16", 1, 3, [10, 100], 1.6e5),
])
def test_compress_matches_oracle(dtype, r, T, pos0, theta):
    B = len(pos0)
    om, oi, pm, pi, diag, cap = _compress_case(B, T, r, dtype, pos0, seed=11 + T, theta=theta)
    exc = _check_compress(om, oi, pm, pi, diag, pos0, r, T // r, dtype)
    print("compress %s r=%d T=%d: %d near-boundary codes excused" % (dtype, r, T, exc))


# --------------------------------------------------------------- index ----

def _idx_caches(B, N, dtype, seed, integer=False, dup=False):
    oc = oracle.Cache(B, N, CI, dtype)
    g = synth.rng(seed, "idx")
    for b in range(B):
        if dtype == "fp4":
            oc.codes[b], oc.scales[b] = synth.integer_fp4_bytes(g, N, CI) if integer else synth.fp4_bytes(g, N, CI)
        else:
            oc.bf16[b] = synth.integer_bf16(g, (N, CI)) if integer else synth.normal_bf16(g, (N, CI))
    if dup:  # repeat a few entries so that ties straddle the k-th place
        pick = synth.rng(seed, "dup").integers(0, 40, size=(B, N))
        for b in range(B):
            if dtype == "fp4":
                oc.codes[b], oc.scales[b] = oc.codes[b][pick[b]], oc.scales[b][pick[b]]
            else:
                oc.bf16[b] = oc.bf16[b][pick[b]]
    pc = _paged.cache_pair(B, N, CI, dtype, seed)
    _paged.upload(pc, oc)
    return oc, pc


def _run_index(cfg, pc, q_idx, q_pos, n_ent, N, head_w=None, pool=None, want_pool=False, ws_queries=None):
    B, Tq = q_idx.shape[:2]
    k = cfg.topk
    topk = torch.full((B, Tq, k), -7, dtype=torch.int32, device="cuda")
    pool_out = torch.full((B, Tq, cfg.hsi_blocks), -7, dtype=torch.int32, device="cuda") if want_pool else None
    per_q = csa.index_workspace_bytes(cfg, 1, 1, N, reindex=pool is not None)
    nq = B * Tq if ws_queries is None else ws_queries
    ws = torch.empty(per_q * nq, dtype=torch.uint8, device="cuda")
    st = _status()
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pc, _paged.dev(n_ent), N, topk, ws,
                   head_w=None if head_w is None else _paged.dev(head_w),
                   pool=None if pool is None else _paged.dev(pool), pool_out=pool_out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return topk.cpu().numpy(), (pool_out.cpu().numpy() if want_pool else None)


@pytest.mark.parametrize("dtype", ["fp4", "bf16"])
def test_index_topk_integer_mode_bit_exact(dtype):
    """Integer q and integer-valued K make every score exact: the top-k
    (lowest id on ties) and the HSI pool must match bit for bit, including
    chunked workspaces, ragged n_entries and short contexts."""
    B, N, k, nb = 3, 3000, 512, 64
    oc, pc = _idx_caches(B, N, dtype, seed=21, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(21, "q"), (B, 2, H, CI), -1, 1)
    q_pos = np.array([[2999, 1500], [2999, 2999], [300, 2999]], np.int64)
    n_ent = np.array([3000, 2457, 200], np.int32)
    cfg = csa.Cfg(ratio=1, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True, ws_queries=2)
    o_top, o_pool, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True,
                                         want_scores=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)
    ties = 0
    for b in range(B):
        for t in range(2):
            v = np.sort(s[b, t][np.isfinite(s[b, t])])[::-1]
            ties += len(v) > k and v[k - 1] == v[k]
    assert ties > 0


def test_index_topk_random_fp4_with_head_weights_and_ratio2():
    B, N, k = 2, 2500, 512
    oc, pc = _idx_caches(B, N, "fp4", seed=22)
    q_idx = synth.normal_bf16(synth.rng(22, "q"), (B, 3, H, CI))
    hw = synth.rng(22, "hw").uniform(0.0, 2.0, size=(B, 3, H)).astype(np.float32)
    q_pos = np.array([[4999, 2000, 1], [4999, 1100, 700]], np.int64)
    n_ent = np.array([2500, 2500], np.int32)
    cfg = csa.Cfg(ratio=2, topk=k)
    g_top, _ = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, head_w=hw)
    o_top, _, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=2, k=k, head_w=hw, want_scores=True)
    assert P.topk_mismatch(g_top.reshape(-1, k), o_top.reshape(-1, k), s.reshape(B * 3, -1), k, exact=False) == 0
    assert (g_top[0, 2] >= 0).sum() == 1 and g_top[0, 2, 0] == 0  # t = 1 sees entry 0 only


@pytest.mark.parametrize("N", [40000, 20000, 16000])
def test_select_threshold_bin_beyond_shared_list_and_single_slots(N):
    """N - 500 copies of one indexer row among 500 random rows: fewer than k
    keys lie above the copies' key, so the k-th place falls inside a bin of
    more than 8192 equal keys (refined over the scores themselves, the first
    ids win); N = 40000 selects over a cluster of CTAs, N = 20000 within one
    CTA at 32 keys a thread, N = 16000 at 16.  hsi_blocks = 1 keeps only the
    forced latest block and topk = 1 the single best entry."""
    B = 1
    oc = oracle.Cache(B, N, CI, "fp4")
    oc.codes[0], oc.scales[0] = synth.integer_fp4_bytes(synth.rng(26, "idx"), N, CI)
    oc.codes[0, 500:], oc.scales[0, 500:] = oc.codes[0, 7], oc.scales[0, 7]
    pc = _paged.cache_pair(B, N, CI, "fp4", 26)
    _paged.upload(pc, oc)
    q_idx = synth.integer_bf16(synth.rng(26, "q"), (B, 2, H, CI), -1, 1)
    q_pos = np.array([[N - 1, 12345]], np.int64)
    n_ent = np.array([N], np.int32)
    for k, nb in ((512, 1), (1, 3)):
        cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
        g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
        o_top, o_pool, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True,
                                             want_scores=True)
        np.testing.assert_array_equal(g_top, o_top)
        np.testing.assert_array_equal(g_pool, o_pool)
    v = s[0, 0][np.isfinite(s[0, 0])]
    assert (v > v[600]).sum() < 512 and v.max() - v.min() >= 1.0  # the case the test is for


@pytest.mark.parametrize("nb", [65, 128])
@pytest.mark.parametrize("N", [6000, 6003])
def test_full_topk_through_the_hsi_pool_is_exact(nb, N):
    """With HSI and at least k + 1 pool blocks the selection takes the pool
    first and the top-k among the pool's positions; on integer scores with
    many ties (duplicated rows) both must equal the oracle's top-k over all
    visible entries and its pool, bit for bit, including a pool of exactly
    k + 1 blocks.  With 6003 entries per row most queries' score and
    block-maximum rows start off a 16-byte boundary (read without vector
    loads)."""
    B, k = 3, 64
    oc, pc = _idx_caches(B, N, "fp4", seed=27, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(27, "q"), (B, 2, H, CI), -1, 1)
    q_pos = np.array([[5999, 3001], [5999, 5999], [777, 5999]], np.int64)
    n_ent = np.array([6000, 5555, 2000], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)


@pytest.mark.parametrize("dup", [True, False])
def test_full_topk_through_a_pool_over_more_blocks_than_one_round(dup):
    """The HSI pool chosen among 16385..32768 blocks (more than 16 keys a
    thread hold): the pool selection holds 32 keys a thread in registers,
    then the top-k among the pool's positions; integer scores (with 40
    distinct entries repeated, or not), bit for bit against the oracle's
    pool and top-k."""
    B, N, k, nb = 2, 262000, 64, 128
    oc, pc = _idx_caches(B, N, "fp4", seed=29, integer=True, dup=dup)
    q_idx = synth.integer_bf16(synth.rng(29, "q"), (B, 1, H, CI), -1, 1)
    q_pos = np.array([[261999], [140000]], np.int64)  # 32750 and 17501 blocks visible
    n_ent = np.array([262000, 200000], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_pool, o_pool)
    np.testing.assert_array_equal(g_top, o_top)


def test_reindex_over_pool_matches_oracle():
    B, N, k, nb = 2, 4000, 64, 40
    oc, pc = _idx_caches(B, N, "fp4", seed=23, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(23, "q"), (B, 1, H, CI), -1, 1)
    q_pos = np.array([[3999], [3500]], np.int64)
    n_ent = np.array([4000, 4000], np.int32)
    g = synth.rng(23, "pool")
    pool = np.full((B, 1, nb), -1, np.int32)
    for b in range(B):
        blocks = np.sort(g.choice(500, size=nb - 3, replace=False))
        pool[b, 0, :nb - 3] = blocks
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
    g_top, _ = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, pool=pool)
    o_top, _, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, pool=pool)
    np.testing.assert_array_equal(g_top, o_top)


# -------------------------------------------------------------- attend ----

def _main_caches(B, N, dtype, seed):
    oc = oracle.Cache(B, N, D, dtype)
    g = synth.rng(seed, "main")
    for b in range(B):
        if dtype == "fp4":
            oc.codes[b], oc.scales[b] = synth.fp4_bytes(g, N, D)
        else:
            oc.bf16[b] = synth.normal_bf16(g, (N, D))
    pc = _paged.cache_pair(B, N, D, dtype, seed)
    _paged.upload(pc, oc)
    return oc, pc


@pytest.mark.parametrize("dtype", ["fp4", "bf16"])
def test_attend_matches_oracle(dtype):
    """Decode and banded-window prefill queries, -1 padded top-k, a window
    clipped at the sequence start and a short window buffer."""
    B, N, Tq, k, W = 3, 700, 3, 512, 128
    oc, pc = _main_caches(B, N, dtype, seed=31)
    g = synth.rng(31, "ids")
    topk = np.full((B, Tq, k), -1, np.int32)
    for b in range(B):
        for t in range(Tq):
            n = [512, 300, 0][(b + t) % 3]
            topk[b, t, :n] = np.sort(g.choice(N, size=n, replace=False))
    q = synth.normal_bf16(synth.rng(31, "q"), (B, Tq, HM, D))
    S = 200
    swa = synth.normal_bf16(synth.rng(31, "swa"), (B, S, D))
    swa_pos0 = np.array([0, 1000, 5000], np.int64)
    swa_len = np.array([150, 200, 60], np.int32)
    q_pos = np.array([[3, 100, 149], [1199, 1130, 1050], [5059, 5100, 4990]], np.int64)
    n_ent = np.array([N, N, N], np.int32)
    scale = 1 / math.sqrt(D)
    cfg = csa.Cfg(ratio=2, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, topk=k, window=W)
    out = torch.empty((B, Tq, HM, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Tq, HM), dtype=torch.float32, device="cuda")
    st = _status()
    csa.attend(cfg, _paged.dev(q), pc, _paged.dev(n_ent), _paged.dev(topk), _paged.dev(swa), _paged.dev(swa_len),
               _paged.dev(swa_pos0), _paged.dev(q_pos), out, lse=lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_out, o_lse = oracle.attend(oc, n_ent, q, topk, swa, swa_len, swa_pos0, q_pos, W, scale, want_lse=True)
    err = P.attention_rel_err(out.cpu().numpy(), o_out)
    assert err <= P.ATT_TOL, err
    lg = lse.cpu().numpy()
    fin = np.isfinite(o_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], o_lse[fin], rtol=0, atol=1e-3)
    print("attend %s: max row rel err %.3g" % (dtype, err))


def test_attend_reports_out_of_range_ids():
    B, N = 1, 100
    oc, pc = _main_caches(B, N, "fp4", seed=32)
    topk = np.array([[[3, 50, 99, 100, -1]]], np.int32)  # 100 is past the last entry
    q = synth.normal_bf16(synth.rng(32, "q"), (1, 1, HM, D))
    swa = synth.normal_bf16(synth.rng(32, "swa"), (1, 4, D))
    cfg = csa.Cfg(ratio=1, topk=5, window=4)
    out = torch.empty((1, 1, HM, D), dtype=torch.float32, device="cuda")
    st = _status()
    csa.attend(cfg, _paged.dev(q), pc, _paged.dev(np.array([N], np.int32)), _paged.dev(topk), _paged.dev(swa),
               _paged.dev(np.array([4], np.int32)), _paged.dev(np.array([96], np.int64)),
               _paged.dev(np.array([[99]], np.int64)), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 17  # CSA2_ERR_BAD_INDEX
    want = oracle.attend(oc, np.array([N]), q, np.array([[[3, 50, 99, -1, -1]]], np.int32), swa,
                         np.array([4], np.int32), np.array([96]), np.array([[99]]), 4, 1 / math.sqrt(D))
    assert P.attention_rel_err(out.cpu().numpy(), want) <= P.ATT_TOL


@pytest.mark.parametrize("integer", [True, False])
def test_index_prefill_queries_share_tiles(integer):
    """Prefill-shaped indexing: 8 consecutive causal queries of one sequence
    (four per CTA on the tensor-core path) over a cache of many tiles, r = 2,
    with HSI blocks; exact on integer inputs, near-tie tolerant otherwise."""
    B, N, k, nb = 1, 9000, 512, 256
    oc, pc = _idx_caches(B, N, "fp4", seed=24, integer=integer, dup=integer)
    g = synth.rng(24, "q")
    Tq = 8
    q_idx = synth.integer_bf16(g, (B, Tq, H, CI), -1, 1) if integer else synth.normal_bf16(g, (B, Tq, H, CI))
    q_pos = (2 * N - Tq + np.arange(Tq)).reshape(1, Tq).astype(np.int64)  # last 8 positions: ragged visibility
    q_pos[0, :3] = [1, 200, 5001]
    n_ent = np.array([N], np.int32)
    cfg = csa.Cfg(ratio=2, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=2, k=k, hsi_blocks=nb, hsi_block=8,
                                         want_pool=True, want_scores=True)
    if integer:
        np.testing.assert_array_equal(g_top, o_top)
        np.testing.assert_array_equal(g_pool, o_pool)
    else:
        assert P.topk_mismatch(g_top.reshape(Tq, k), o_top.reshape(Tq, k), s.reshape(Tq, -1), k, exact=False) == 0
        for t in range(Tq):  # pools may differ only by near-tied block maxima
            gp, op = set(g_pool[0, t][g_pool[0, t] >= 0]), set(o_pool[0, t][o_pool[0, t] >= 0])
            if gp != op:
                nv = (q_pos[0, t] - 1) // 2 + 1
                bm = [s[0, t, 8 * b_:min(8 * b_ + 8, nv)].max() for b_ in range((nv + 7) // 8)]
                kth = sorted(bm, reverse=True)[nb - 1]
                assert all(abs(bm[b_] - kth) <= P.NEAR_TIE * abs(kth) for b_ in gp ^ op)


@pytest.mark.parametrize("dtype,Tq,chunk", [("fp4", 5, None), ("fp4", 2, None), ("bf16", 6, None),
                                            ("fp4", 7, None), ("fp4", 5, 5), ("bf16", 5, 6)])
def test_index_multi_query_blocks_share_tiles(dtype, Tq, chunk):
    """Multi-query decode: Tq consecutive positions of each of 3 sequences.
    A chunk of whole sequences puts up to 6 queries of a sequence in one
    group (Tq = 7: a group of 4 and a masked group of 3); a chunk that cuts a
    sequence (6 queries of 5-query blocks) falls back to one query per group.
    Integer inputs: top-k and HSI pool bit-exact, with head weights and
    ragged n_entries."""
    B, N, k, nb = 3, 4000, 512, 64
    oc, pc = _idx_caches(B, N, dtype, seed=26 + Tq, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(26, "q%d" % Tq), (B, Tq, H, CI), -1, 1)
    hw = synth.rng(26, "hw").integers(0, 3, size=(B, Tq, H)).astype(np.float32)
    n_ent = np.array([N, 3100, 700], np.int32)
    q_pos = np.stack([2 * n - Tq + np.arange(Tq) for n in n_ent]).astype(np.int64)  # the block ends the context
    cfg = csa.Cfg(ratio=2, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, head_w=hw, want_pool=True, ws_queries=chunk)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=2, k=k, head_w=hw, hsi_blocks=nb,
                                         want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)


def test_index_long_cache_many_tiles_per_cta():
    """One decode query per sequence over 40000 entries: each CTA walks many
    tiles through the shared-memory ring (wrap-around of every stage)."""
    B, N, k = 2, 40000, 512
    oc, pc = _idx_caches(B, N, "fp4", seed=25, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(25, "q"), (B, 1, H, CI), -1, 1)
    q_pos = np.array([[N - 1], [31000]], np.int64)
    n_ent = np.array([N, 35000], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=2048)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=2048, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)


# -------------------------------------------------------------- capture ----

def test_captured_index_and_attend_replay_on_new_data():
    """csa.capture records the library's calls (clusters, programmatic
    launches) as a graph; replayed after new query data is written into the
    same buffers, it gives exactly what the calls give when issued again."""
    B, N, k, W = 4, 5000, 512, 128
    _, pi = _idx_caches(B, N, "fp4", seed=28)
    _, pm = _main_caches(B, N, "fp4", 28)
    cfg = csa.Cfg(ratio=1, topk=k, window=W)
    g = synth.rng(28, "q")
    q_idx = _paged.dev(synth.normal_bf16(g, (B, 1, H, CI)))
    q = _paged.dev(synth.normal_bf16(g, (B, 1, 64, D)))
    swa = _paged.dev(synth.normal_bf16(g, (B, W, D)))
    q_pos = _paged.dev(np.full((B, 1), N - 1, np.int64))
    n_ent = _paged.dev(np.full(B, N, np.int32))
    swa_len = _paged.dev(np.full(B, W, np.int32))
    swa_pos0 = _paged.dev(np.full(B, N - W, np.int64))
    topk = torch.empty((B, 1, k), dtype=torch.int32, device="cuda")
    out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    st = _status()

    def calls():
        csa.index_topk(cfg, q_idx, q_pos, pi, n_ent, N, topk, ws, status=st)
        csa.attend(cfg, q, pm, n_ent, topk, swa, swa_len, swa_pos0, q_pos, out, status=st)

    graph = csa.capture(calls)
    g2 = synth.rng(29, "q")
    q_idx.copy_(_paged.dev(synth.normal_bf16(g2, (B, 1, H, CI))))
    q.copy_(_paged.dev(synth.normal_bf16(g2, (B, 1, 64, D))))
    graph()
    torch.cuda.synchronize()
    got_top, got_out = topk.clone(), out.clone()
    calls()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got_top, topk)
    assert torch.equal(got_out, out)


# ------------------------------------------------- larger configurations ----

@pytest.mark.parametrize("dtype,k,W,B,Tq", [
    ("fp4", 1024, 512, 2, 1),    # 12 row tiles: the head-split cluster kernel
    ("bf16", 1024, 512, 2, 2),
    ("fp4", 1024, 512, 40, 1),   # too many clusters for one wave: the per-query kernel
    ("fp4", 768, 0, 3, 2),       # six tiles of top-k rows and no window
    ("fp4", 640, 256, 3, 2),     # windows clipped at the sequence start
    ("fp4", 512, 128, 24, 1),    # the model's five row tiles: clusters of five beside the selection
    ("fp4", 512, 128, 28, 1),    # ... clusters of four (five would not fit beside the selection)
])
def test_attend_larger_selections_and_windows(dtype, k, W, B, Tq):
    """The attention kernels for configurations beyond six row tiles (maximum
    top-k 1024 and window 512) and without a window, and the query-cluster
    kernel in both of its cluster shapes, against the oracle."""
    N = 3000
    oc, pc = _main_caches(B, N, dtype, seed=70 + k + W)
    g = synth.rng(70, "ids%d" % k)
    topk = np.full((B, Tq, k), -1, np.int32)
    for b in range(B):
        for t in range(Tq):
            n = [k, k // 2, 7][(b + t) % 3]
            topk[b, t, :n] = np.sort(g.choice(N, size=n, replace=False))
    q = synth.normal_bf16(synth.rng(70, "q%d" % k), (B, Tq, HM, D))
    S = max(W, 1) + Tq
    swa = synth.normal_bf16(synth.rng(70, "swa%d" % k), (B, S, D))
    swa_pos0 = np.zeros(B, np.int64)
    swa_len = np.full(B, S, np.int32)
    # positions: the window runs past the buffer start for some queries
    q_pos = np.array([[min(S - 1, 3 + 200 * b + t * 50) for t in range(Tq)] for b in range(B)], np.int64)
    n_ent = np.full(B, N, np.int32)
    cfg = csa.Cfg(ratio=1, cache_dtype=csa.CACHE_FP4 if dtype == "fp4" else csa.CACHE_BF16, topk=k, window=W)
    out = torch.empty((B, Tq, HM, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Tq, HM), dtype=torch.float32, device="cuda")
    st = _status()
    csa.attend(cfg, _paged.dev(q), pc, _paged.dev(n_ent), _paged.dev(topk), _paged.dev(swa) if W else None,
               _paged.dev(swa_len), _paged.dev(swa_pos0), _paged.dev(q_pos), out, lse=lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_out, o_lse = oracle.attend(oc, n_ent, q, topk, swa, swa_len if W else np.zeros(B, np.int32), swa_pos0, q_pos,
                                 W, 1 / math.sqrt(D), want_lse=True)
    err = P.attention_rel_err(out.cpu().numpy(), o_out)
    assert err <= P.ATT_TOL, err
    lg = lse.cpu().numpy()
    fin = np.isfinite(o_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], o_lse[fin], rtol=0, atol=1e-3)
    print("attend %s k=%d W=%d B=%d Tq=%d: max row rel err %.3g" % (dtype, k, W, B, Tq, err))


def test_index_maximum_topk_and_hsi_blocks_bit_exact():
    """top-k 1024 with 4096 HSI blocks (the largest accepted), integer mode,
    one sequence shorter than the pool, and Reindex over the largest pool."""
    B, N, k, nb = 2, 40000, 1024, 4096
    oc, pc = _idx_caches(B, N, "fp4", seed=71, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(71, "q"), (B, 1, H, CI), -1, 1)
    q_pos = np.array([[N - 1], [20000]], np.int64)
    n_ent = np.array([N, 30000], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)
    q2 = synth.integer_bf16(synth.rng(72, "q"), (B, 1, H, CI), -1, 1)
    r_top, _ = _run_index(cfg, pc, q2, q_pos, n_ent, N, pool=o_pool)
    o_rtop, _, _ = oracle.index_topk(oc, n_ent, q2, q_pos, r=1, k=k, hsi_blocks=nb, pool=o_pool)
    np.testing.assert_array_equal(r_top, o_rtop)


@pytest.mark.parametrize("integer,k", [(True, 512), (False, 512), (True, 1024), (False, 97)])
def test_select_many_queries_over_long_caches(integer, k):
    """96 causal queries over 20000 entries: one CTA per selection holding
    twice the positions of the 16-keys-a-thread selection, 32 keys in each
    thread's registers; integer inputs with repeated entries make ties
    straddle the threshold for some queries."""
    B, N, Tq = 1, 20000, 96
    oc, pc = _idx_caches(B, N, "fp4", seed=73 + k, integer=integer, dup=integer)
    g = synth.rng(73, "q%d" % k)
    q_idx = synth.integer_bf16(g, (B, Tq, H, CI), -1, 1) if integer else synth.normal_bf16(g, (B, Tq, H, CI))
    q_pos = (N - 2 * Tq + 2 * np.arange(Tq)).reshape(1, Tq).astype(np.int64)  # ragged visibility, all > 16384
    n_ent = np.array([N], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k)
    g_top, _ = _run_index(cfg, pc, q_idx, q_pos, n_ent, N)
    o_top, _, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, want_scores=True)
    if integer:
        np.testing.assert_array_equal(g_top, o_top)
        ties = 0
        for t in range(Tq):
            v = np.sort(s[0, t][np.isfinite(s[0, t])])[::-1]
            ties += v[k - 1] == v[k]
        assert ties > 0
    else:
        assert P.topk_mismatch(g_top.reshape(Tq, k), o_top.reshape(Tq, k), s.reshape(Tq, -1), k, exact=False) == 0


@pytest.mark.parametrize("integer", [True, False])
def test_select_sampled_pass_over_very_long_caches(integer):
    """80 causal queries over 140000 entries: one CTA per selection over more
    than eight rounds of positions, where a 1/16 sample of the keys picks the
    bin above which the selection is listed in one pass.  Integer inputs with
    repeated entries make ties straddle the threshold for some queries (the
    general passes then take over) and must still match bit for bit."""
    B, N, Tq, k = 1, 140000, 80, 512
    oc, pc = _idx_caches(B, N, "fp4", seed=77, integer=integer, dup=integer)
    g = synth.rng(77, "q")
    q_idx = synth.integer_bf16(g, (B, Tq, H, CI), -1, 1) if integer else synth.normal_bf16(g, (B, Tq, H, CI))
    q_pos = (N - 3 * Tq + 3 * np.arange(Tq)).reshape(1, Tq).astype(np.int64)
    n_ent = np.array([N], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k)
    g_top, _ = _run_index(cfg, pc, q_idx, q_pos, n_ent, N)
    o_top, _, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, want_scores=True)
    if integer:
        np.testing.assert_array_equal(g_top, o_top)
    else:
        assert P.topk_mismatch(g_top.reshape(Tq, k), o_top.reshape(Tq, k), s.reshape(Tq, -1), k, exact=False) == 0


def test_degenerate_queries_nothing_visible_and_no_rows():
    """Queries before the first complete group (nothing visible: the top-k
    is all -1 and the pool empty), a context shorter than k and than the
    pool, and attention with neither selected entries nor window rows
    (output zero, LSE -inf), against the oracle."""
    B, N, k, nb = 2, 40, 64, 16
    oc, pc = _idx_caches(B, N, "fp4", seed=79, integer=True, dup=True)
    q_idx = synth.integer_bf16(synth.rng(79, "q"), (B, 3, H, CI), -1, 1)
    q_pos = np.array([[0, 1, 2 * N - 1], [0, 5, 30]], np.int64)  # r = 2: position 0 sees nothing
    n_ent = np.array([N, 17], np.int32)
    cfg = csa.Cfg(ratio=2, topk=k, hsi_blocks=nb)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=2, k=k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)
    assert (g_top[:, 0] == -1).all() and (g_pool[:, 0] == -1).all()
    # attention: query 0 of each sequence has no entry and (swa_len 0) no window row
    om, pm = _main_caches(B, N, "fp4", seed=79)
    q = synth.normal_bf16(synth.rng(79, "qa"), (B, 3, HM, D))
    swa = synth.normal_bf16(synth.rng(79, "swa"), (B, 8, D))
    swa_len = np.array([0, 8], np.int32)
    swa_pos0 = np.array([0, 23], np.int64)
    W = 8
    acfg = csa.Cfg(ratio=2, topk=k, window=W)
    out = torch.empty((B, 3, HM, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 3, HM), dtype=torch.float32, device="cuda")
    st = _status()
    csa.attend(acfg, _paged.dev(q), pm, _paged.dev(n_ent), _paged.dev(o_top), _paged.dev(swa), _paged.dev(swa_len),
               _paged.dev(swa_pos0), _paged.dev(q_pos), out, lse=lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_out, o_lse = oracle.attend(om, n_ent, q, o_top, swa, swa_len, swa_pos0, q_pos, W, 1 / math.sqrt(D),
                                 want_lse=True)
    g_out, g_lse = out.cpu().numpy(), lse.cpu().numpy()
    assert (g_out[0, 0] == 0).all() and np.isneginf(g_lse[0, 0]).all()  # nothing to attend to
    assert np.array_equal(np.isfinite(g_lse), np.isfinite(o_lse))
    fin = np.isfinite(o_lse)
    np.testing.assert_allclose(g_lse[fin], o_lse[fin], rtol=0, atol=1e-3)
    assert P.attention_rel_err(g_out[:, 1:], o_out[:, 1:]) <= P.ATT_TOL


@pytest.mark.parametrize("mode", ["full_hsi", "full", "reindex", "multi_query"])
def test_index_in_two_calls_equals_index_topk(mode):
    """csa2_index_score followed by csa2_index_select gives what
    csa2_index_topk gives, bit for bit, on integer inputs (exact scores, ties
    broken by id): Full with and without the HSI pool, Reindex over a pool,
    and a multi-query block of 5 positions per sequence."""
    B, N, k, nb = 3, 9000, 128, 200
    oc, pc = _idx_caches(B, N, "fp4", seed=31, integer=True, dup=True)
    Tq = 5 if mode == "multi_query" else 1
    q_idx = synth.integer_bf16(synth.rng(31, "q"), (B, Tq, H, CI), -1, 1)
    q_pos = np.array([[8995 + t for t in range(Tq)], [7000 + t for t in range(Tq)], [4000 + t for t in range(Tq)]],
                     np.int64)
    n_ent = np.array([9000, 8000, 9000], np.int32)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb if mode != "full" else 0)
    pool = None
    if mode == "reindex":
        _, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True)
        pool = _paged.dev(o_pool)
    want_pool = mode == "full_hsi"
    ref_top, ref_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, pool=None if pool is None else o_pool,
                                   want_pool=want_pool)
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, Tq, N, reindex=pool is not None), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xAB)  # no state carried in from elsewhere
    topk = torch.full((B, Tq, k), -7, dtype=torch.int32, device="cuda")
    pool_out = torch.full((B, Tq, nb), -7, dtype=torch.int32, device="cuda") if want_pool else None
    st = _status()
    qp, ne = _paged.dev(q_pos), _paged.dev(n_ent)
    csa.index_score(cfg, _paged.dev(q_idx), qp, pc, ne, N, ws, pool=pool, hsi=want_pool, status=st)
    csa.index_select(cfg, qp, pc, ne, N, topk, ws, pool=pool, pool_out=pool_out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(topk.cpu().numpy(), ref_top)
    if want_pool:
        np.testing.assert_array_equal(pool_out.cpu().numpy(), ref_pool)
    # a workspace short of one query's worth for all of them is refused
    small = torch.empty(ws.numel() - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(csa.CsaError):
        csa.index_score(cfg, _paged.dev(q_idx), qp, pc, ne, N, small, pool=pool, hsi=want_pool, status=st)


@pytest.mark.parametrize("nb", [2048, 4096])
def test_large_pools_over_many_blocks_are_ascending_and_exact(nb):
    """A Full layer with HSI over more than 32768 blocks (the decoder group's
    262144 entries hold 32768): the pool selection runs over rows longer
    than one CTA's registers, through the sampled one-pass selection (pool
    of 2048) or the staged passes (pool of 4096), and its ids must come out
    ascending.  Random inputs (few ties: the sampled path) compared up to
    near-ties; integer inputs with ties compared bit for bit."""
    B, N, k = 1, 280000, 512
    for integer in (False, True):
        oc, pc = _idx_caches(B, N, "fp4", seed=32 + integer, integer=integer, dup=integer)
        q_idx = (synth.integer_bf16(synth.rng(32, "q"), (B, 1, H, CI), -1, 1) if integer else
                 synth.normal_bf16(synth.rng(32, "q"), (B, 1, H, CI)))
        q_pos = np.array([[N - 1]], np.int64)
        n_ent = np.array([N], np.int32)
        cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb)
        g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
        o_top, o_pool, s = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True,
                                             want_scores=True)
        gp = g_pool.reshape(B, nb)
        assert np.all(np.diff(gp[0][gp[0] >= 0]) > 0), "pool ids not ascending"
        assert np.all(np.diff(g_top[0, 0][g_top[0, 0] >= 0]) > 0), "top-k ids not ascending"
        if integer:
            np.testing.assert_array_equal(g_top, o_top)
            np.testing.assert_array_equal(g_pool, o_pool)
        else:
            assert P.pool_mismatch(gp, o_pool.reshape(B, nb), s.reshape(B, -1)) == 0
            assert P.topk_mismatch(g_top.reshape(B, k), o_top.reshape(B, k), s.reshape(B, -1), k, exact=False) == 0


def _single_query_scan(fmt, seed, N, n_ent, q_pos, nb=1024, k=512):
    """Integer-valued single-query scans of B sequences (repeated rows make
    ties at the k-th place): top-k and HSI pool against the oracle, bit for
    bit."""
    B = len(n_ent)
    oc = oracle.Cache(B, N, CI, fmt)
    g = synth.rng(seed, "idx")
    for b in range(B):
        codes, scales = synth.integer_fp4_bytes(g, N, CI)  # every scale 1.0
        oc.codes[b], oc.scales[b] = codes, scales[:, :oc.scales.shape[-1]]
    pick = synth.rng(seed, "dup").integers(0, min(3000, N), size=(B, N))
    for b in range(B):
        oc.codes[b], oc.scales[b] = oc.codes[b][pick[b]], oc.scales[b][pick[b]]
    pc = _paged.cache_pair(B, N, CI, "fp4" if fmt == "fp4" else "fp4g32", seed)
    _paged.upload(pc, oc)
    q_idx = synth.integer_bf16(synth.rng(seed, "q"), (B, 1, H, CI), -1, 1)
    n_ent = np.asarray(n_ent, np.int32)
    q_pos = np.asarray(q_pos, np.int64).reshape(B, 1)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb, formats=csa.FMT_IDX_68B if fmt == "fp4g32" else 0)
    g_top, g_pool = _run_index(cfg, pc, q_idx, q_pos, n_ent, N, want_pool=True)
    o_top, o_pool, _ = oracle.index_topk(oc, n_ent, q_idx, q_pos, r=1, k=k, hsi_blocks=nb, want_pool=True)
    np.testing.assert_array_equal(g_top, o_top)
    np.testing.assert_array_equal(g_pool, o_pool)


@pytest.mark.parametrize("fmt", ["fp4", "fp4g32"])
def test_single_query_scan_many_tiles_per_cta_exact(fmt):
    """The single-query scan over many pages: 8 sequences of up to 50000
    entries share one wave of CTAs, so every CTA streams about 20 tiles (its
    shared-memory ring of 16 slots wraps around); ragged entry counts and
    query positions leave inactive tiles at the ends of some ranges.  The
    68-byte entries run the same path."""
    _single_query_scan(fmt, 33, 50000, [50000, 49999, 31000, 50000, 12345, 50000, 40000, 50000],
                       [49999, 49999, 30999, 20000, 12344, 49999, 39999, 777])


@pytest.mark.parametrize("fmt", ["fp4", "fp4g32"])
def test_single_query_scan_flattened_over_one_wave_exact(fmt):
    """24 single queries, too many for one wave of per-query CTA ranges: the
    scorer lays the queries' tiles end to end over one CTA per SM, so most
    CTAs' ranges cross from one query into the next (two query tiles, two
    key-range slots) and the selection reads each query's slots by the
    partition.  Ragged lengths: a sequence of one entry, short sequences whose
    CTAs have no visible tile, a query that sees a few entries only."""
    n_ent = [20000, 1, 19999, 300, 20000, 12345, 20000, 129, 20000, 20000, 7000, 20000,
             20000, 18000, 20000, 128, 20000, 20000, 20000, 5000, 20000, 19000, 20000, 20000]
    q_pos = [19999, 0, 19998, 299, 100, 12344, 19999, 128, 19999, 3, 6999, 19999,
             19999, 17999, 10000, 127, 19999, 19999, 19999, 4999, 19999, 18999, 19999, 640]
    _single_query_scan(fmt, 34, 20000, n_ent, q_pos)


@pytest.mark.parametrize("fmt", ["fp4", "fp4g32"])
def test_single_query_scan_flattened_across_nearly_every_cta_exact(fmt):
    """151 single queries of up to 700 entries (6 tiles each) over one wave
    of 152 CTAs of about 6 tiles: nearly every CTA's range crosses from one
    query into the next, and each query's key range is spread over two
    slots.  A pool of 40 blocks with k = 32 takes the fused selection (the
    pool, then the top-k among its positions, bounded below by the pool's
    threshold key).  Short sequences and queries that see a few entries
    only."""
    B, N = 151, 700
    n_ent = [N if b % 5 else 1 + (37 * b) % N for b in range(B)]
    q_pos = [(n - 1) if b % 3 else (53 * b) % N for b, n in enumerate(n_ent)]
    _single_query_scan(fmt, 35, N, n_ent, q_pos, nb=40, k=32)
