"""GPU-vs-oracle parity at the full sizes of the synthetic workloads, in
the launch configurations bench.py times.  The GPU runs the whole workload;
the oracle checks every output where it finishes in seconds (decode b1 and
b8, the multi-query decode block) and sampled sequences / query rows
otherwise (decode b32: 3 of 32 sequences; decoder group: 2 of 16 sequences
through all 20 layers; prefill: 6 of 4096 query rows).  Each side works from its own cache: the compressor runs on
both, the seeded random prefix is shared input."""
import math

import numpy as np
import pytest
import torch

import compressed_sparse_attention_07_gb300 as csa
import oracle
import synth
from tests import _paged
from tests import _parity as P
from tests.test_gpu_stages import _check_compress

pytestmark = pytest.mark.gpu

D, CI = 512, 128
SCALE = 1 / math.sqrt(D)


def _cfg(wl):
    fmt = ((csa.FMT_IDX_68B if wl.idx68 else 0) | (csa.FMT_SWA_FP8 if wl.swa_fp8 else 0) |
           (csa.FMT_IDX_QFP4 if wl.q_fp4 else 0))
    return csa.Cfg(ratio=wl.ratio, cache_dtype=csa.CACHE_FP4 if wl.cache == "fp4" else csa.CACHE_BF16,
                   topk=wl.topk, window=wl.window, hsi_blocks=wl.hsi_blocks if wl.hsi else 0, rope_theta=wl.theta,
                   formats=fmt)


def _idx_dtype(wl):
    return "fp4g32" if wl.idx68 else wl.cache


def _prefix(wl, b, n):
    """Seeded random cache prefix of sequence b (n entries), canonical form."""
    g = synth.rng(wl.seed, "prefix%d" % b)
    m, i = oracle.Cache(1, n, D, wl.cache), oracle.Cache(1, n, CI, wl.cache)
    for c in (m, i):
        if wl.cache == "fp4":
            c.codes[0], c.scales[0] = synth.fp4_bytes(g, n, c.channels)
        else:
            c.bf16[0] = synth.normal_bf16(g, (n, c.channels))
    return m, i


def _step_inputs(wl, B, tag=""):
    s = wl.seed
    w = synth.merge_weights(synth.rng(s, "w"), wl.ratio, D)
    w_idx = synth.normal_bf16(synth.rng(s, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    q = synth.normal_bf16(synth.rng(s, "q" + tag), (B, 1, 64, D))
    q_idx = synth.normal_bf16(synth.rng(s, "q_idx" + tag), (B, 1, 32, CI))
    swa = synth.normal_bf16(synth.rng(s, "swa" + tag), (B, wl.window, D))
    return w, w_idx, q, q_idx, swa


def _compress_full_context(wl):
    """Configs 1-2: the whole context goes through the compressor on both sides."""
    B, r, ctx = wl.batch, wl.ratio, wl.ctx
    N = ctx // r
    x = synth.normal_bf16(synth.rng(wl.seed, "ctx_tokens"), (B, ctx, D))
    w, w_idx, q, q_idx, swa = _step_inputs(wl, B)
    om, oi = oracle.Cache(B, N, D, wl.cache), oracle.Cache(B, N, CI, _idx_dtype(wl))
    diag = oracle.compress(x, np.zeros(B, np.int64), w, w_idx, om, oi, r, wl.theta, diagnostics=True)
    cfg = _cfg(wl)
    pm, pi = _paged.cache_pair(B, N, D, wl.cache, wl.seed), _paged.cache_pair(B, N, CI, _idx_dtype(wl), wl.seed + 1)
    n_ent = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.compress(cfg, _paged.dev(x), _paged.dev(np.zeros(B, np.int64)), _paged.dev(w), _paged.dev(w_idx), pm, pi,
                 n_ent, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exc = _check_compress(om, oi, pm, pi, diag, np.zeros(B, np.int64), r, N, wl.cache)
    print("%s: %d near-boundary codes excused of %d entries" % (wl.name, exc, B * N))
    return cfg, om, oi, pm, pi, n_ent, q, q_idx, swa


@pytest.mark.parametrize("name", ["decode_b1_ctx4096_r2_bf16", "decode_b8_ctx32768_r2_fp4",
                                  "decode_b8_ctx32768_r2_fp4_idx68_fp8swa", "decode_b8_ctx32768_r2_fp4_qfp4"])
def test_decode_full_context_through_the_compressor(name):
    """The whole context through the compressor on both sides, then indexing
    and attention of the last position.  The pages' own formats (68-byte
    indexer entries, MXFP8 window rows) run the same check; their window rows
    are encoded on each side and compared bit for bit first."""
    wl = synth.WORKLOADS[name]
    B, N = wl.batch, wl.ctx // wl.ratio
    cfg, om, oi, pm, pi, n_ent, q, q_idx, swa = _compress_full_context(wl)
    swa_dev = _paged.dev(swa)
    if wl.swa_fp8:
        rows = torch.zeros((B, wl.window, csa.SWA_FP8_ROW), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        csa.swa_encode(swa_dev, torch.zeros(B, dtype=torch.int64, device="cuda"), rows, status=st)
        swa = oracle.swa_encode(swa)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        np.testing.assert_array_equal(rows.cpu().numpy(), swa)
        swa_dev = rows
    q_pos = np.full((B, 1), wl.ctx - 1, np.int64)
    swa_len, swa_pos0 = np.full(B, wl.window, np.int32), np.full(B, wl.ctx - wl.window, np.int64)
    topk = torch.empty((B, 1, wl.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pi, n_ent, N, topk, ws, status=st)
    csa.attend(cfg, _paged.dev(q), pm, n_ent, topk, swa_dev, _paged.dev(swa_len), _paged.dev(swa_pos0),
               _paged.dev(q_pos), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n_arr = np.full(B, N, np.int32)
    o_top, _, s = oracle.index_topk(oi, n_arr, q_idx, q_pos, wl.ratio, wl.topk, want_scores=True, q_fp4=wl.q_fp4)
    assert P.topk_mismatch(topk.cpu().numpy().reshape(B, -1), o_top.reshape(B, -1), s.reshape(B, -1), wl.topk,
                           exact=False) == 0
    o_out = oracle.attend(om, n_arr, q, o_top, swa, swa_len, swa_pos0, q_pos, wl.window, SCALE)
    err = P.attention_rel_err(out.cpu().numpy(), o_out)
    print("%s: attention max row rel err %.3g" % (name, err))
    assert err <= P.ATT_TOL


def _random_prefix_caches(wl, B, N, samples):
    """GPU caches holding every sequence's seeded prefix; oracle caches for the
    sampled sequences only."""
    pm, pi = _paged.cache_pair(B, N, D, wl.cache, wl.seed), _paged.cache_pair(B, N, CI, wl.cache, wl.seed + 1)
    om, oi = oracle.Cache(len(samples), N, D, wl.cache), oracle.Cache(len(samples), N, CI, wl.cache)
    for b in range(B):
        m, i = _prefix(wl, b, N)
        _paged.upload_seq(pm, b, m)
        _paged.upload_seq(pi, b, i)
        if b in samples:
            j = samples.index(b)
            om.codes[j], om.scales[j] = m.codes[0], m.scales[0]
            oi.codes[j], oi.scales[j] = i.codes[0], i.scales[0]
    return pm, pi, om, oi


def test_decode_b32_hsi_sampled_sequences():
    wl = synth.WORKLOADS["decode_b32_ctx131072_r1_fp4_hsi"]
    B, N, r = wl.batch, wl.ctx // wl.ratio, wl.ratio
    samples = [0, 13, 31]
    pm, pi, om, oi = _random_prefix_caches(wl, B, N, samples)
    cfg = _cfg(wl)
    w, w_idx, q, q_idx, swa = _step_inputs(wl, B)
    x = synth.normal_bf16(synth.rng(wl.seed, "x_step"), (B, r, D))
    pos0 = np.full(B, wl.ctx - r, np.int64)
    q_pos = np.full((B, 1), wl.ctx - 1, np.int64)
    swa_len, swa_pos0 = np.full(B, wl.window, np.int32), np.full(B, wl.ctx - wl.window, np.int64)
    n_ent = torch.full((B,), N - 1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, 1, wl.topk), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, 1, wl.hsi_blocks), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
    csa.compress(cfg, _paged.dev(x), _paged.dev(pos0), _paged.dev(w), _paged.dev(w_idx), pm, pi, n_ent, status=st)
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pi, n_ent, N, topk, ws, pool_out=pool, status=st)
    csa.attend(cfg, _paged.dev(q), pm, n_ent, topk, _paged.dev(swa), _paged.dev(swa_len), _paged.dev(swa_pos0),
               _paged.dev(q_pos), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sm = np.array(samples)
    oracle.compress(x[sm], pos0[sm], w, w_idx, om, oi, r, wl.theta)
    n_arr = np.full(len(samples), N, np.int32)
    o_top, o_pool, s = oracle.index_topk(oi, n_arr, q_idx[sm], q_pos[sm], r, wl.topk, hsi_blocks=wl.hsi_blocks,
                                         want_pool=True, want_scores=True)
    g_top = topk.cpu().numpy()[sm]
    g_pool = pool.cpu().numpy()[sm]
    assert P.topk_mismatch(g_top.reshape(len(sm), -1), o_top.reshape(len(sm), -1), s.reshape(len(sm), -1), wl.topk,
                           exact=False) == 0
    for j in range(len(sm)):
        gp, op = set(g_pool[j, 0].tolist()), set(o_pool[j, 0].tolist())
        if gp != op:  # only near-tied block maxima may differ
            bm = s[j, 0].reshape(-1, 8).max(-1)
            kth = np.sort(bm)[::-1][wl.hsi_blocks - 1]
            assert all(abs(bm[b_] - kth) <= P.NEAR_TIE * abs(kth) for b_ in (gp ^ op) if b_ >= 0)
        assert (N - 1) // 8 in gp
    o_out = oracle.attend(om, n_arr, q[sm], o_top, swa[sm], swa_len[sm], swa_pos0[sm], q_pos[sm], wl.window, SCALE)
    err = P.attention_rel_err(out.cpu().numpy()[sm], o_out)
    print("decode b32 HSI: attention max row rel err %.3g" % err)
    assert err <= P.ATT_TOL


def test_decoder_group_sampled_sequences():
    wl = synth.WORKLOADS["decoder_group20_b16_ctx262144_fp4"]
    B, N, r = wl.batch, wl.ctx // wl.ratio, wl.ratio
    samples = [0, 15]
    sm = np.array(samples)
    pm, pi, om, oi = _random_prefix_caches(wl, B, N, samples)
    cfg = _cfg(wl)
    w, w_idx, _, _, _ = _step_inputs(wl, B)
    x = synth.normal_bf16(synth.rng(wl.seed, "x_step"), (B, r, D))
    pos0 = np.full(B, wl.ctx - r, np.int64)
    q_pos = np.full((B, 1), wl.ctx - 1, np.int64)
    swa_len, swa_pos0 = np.full(B, wl.window, np.int32), np.full(B, wl.ctx - wl.window, np.int64)
    n_dev = torch.full((B,), N - 1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, 1, wl.topk), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, 1, wl.hsi_blocks), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    state = csa.GroupState(pm, pi, n_dev, N, topk, pool, ws, st)
    oracle.compress(x[sm], pos0[sm], w, w_idx, om, oi, r, wl.theta)
    n_arr = np.full(len(samples), N, np.int32)
    o_top = o_pool = None
    modes = {"full": csa.MODE_FULL, "reindex": csa.MODE_REINDEX, "reuse": csa.MODE_REUSE}
    worst = 0.0
    for layer, mode in wl.layers:
        _, _, q, q_idx, swa = _step_inputs(wl, B, tag="L%d" % layer)
        out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
        kw = {}
        if mode == "full":
            kw = dict(x=_paged.dev(x), pos0=_paged.dev(pos0), merge_w=_paged.dev(w), w_idx=_paged.dev(w_idx))
        topk_before, pool_before = topk.clone(), pool.clone()
        csa.layer(cfg, modes[mode], state, _paged.dev(q_pos), _paged.dev(q), _paged.dev(swa), _paged.dev(swa_len),
                  _paged.dev(swa_pos0), out, q_idx=_paged.dev(q_idx) if mode != "reuse" else None, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, (layer, csa.status_string(int(st.item())))
        if mode != "full":  # the pool stays the Full layer's; a Reuse layer republishes the source top-k unchanged
            assert torch.equal(pool, pool_before), (layer, mode)
        if mode == "reuse":
            assert torch.equal(topk, topk_before), (layer, mode)
        if mode == "full":
            o_top, o_pool, s = oracle.index_topk(oi, n_arr, q_idx[sm], q_pos[sm], r, wl.topk,
                                                 hsi_blocks=wl.hsi_blocks, want_pool=True, want_scores=True)
            g_pool = pool.cpu().numpy()[sm]
            assert P.pool_mismatch(g_pool.reshape(len(sm), -1), o_pool.reshape(len(sm), -1),
                                   s.reshape(len(sm), -1)) == 0, layer
        elif mode == "reindex":
            o_top, _, s = oracle.index_topk(oi, n_arr, q_idx[sm], q_pos[sm], r, wl.topk, hsi_blocks=wl.hsi_blocks,
                                            pool=o_pool, want_scores=True)
        if mode != "reuse":
            g_top = topk.cpu().numpy()[sm]
            assert P.topk_mismatch(g_top.reshape(len(sm), -1), o_top.reshape(len(sm), -1),
                                   s.reshape(len(sm), -1), wl.topk, exact=False) == 0, (layer, mode)
        o_out = oracle.attend(om, n_arr, q[sm], o_top, swa[sm], swa_len[sm], swa_pos0[sm], q_pos[sm], wl.window,
                              SCALE)
        err = P.attention_rel_err(out.cpu().numpy()[sm], o_out)
        worst = max(worst, err)
        assert err <= P.ATT_TOL, (layer, mode, err)
    print("decoder group: worst attention max row rel err %.3g over 20 layers" % worst)


def test_prefill_chunk_sampled_rows():
    wl = synth.WORKLOADS["prefill_4096_on_1m_r2_fp4"]
    B, r, Tq, ctx, W = wl.batch, wl.ratio, wl.tq, wl.ctx, wl.window
    N = (ctx + Tq) // r
    P0 = ctx // r
    pm, pi = _paged.cache_pair(B, N, D, wl.cache, wl.seed), _paged.cache_pair(B, N, CI, wl.cache, wl.seed + 1)
    m, i = _prefix(wl, 0, P0)
    om, oi = oracle.Cache(1, N, D, wl.cache), oracle.Cache(1, N, CI, wl.cache)
    om.codes[0, :P0], om.scales[0, :P0] = m.codes[0], m.scales[0]
    oi.codes[0, :P0], oi.scales[0, :P0] = i.codes[0], i.scales[0]
    _paged.upload(pm, om)
    _paged.upload(pi, oi)
    cfg = _cfg(wl)
    s = wl.seed
    x = synth.normal_bf16(synth.rng(s, "x_chunk"), (B, Tq, D))
    w = synth.merge_weights(synth.rng(s, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(s, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    q = synth.normal_bf16(synth.rng(s, "q"), (B, Tq, 64, D))
    q_idx = synth.normal_bf16(synth.rng(s, "q_idx"), (B, Tq, 32, CI))
    S = W - 1 + Tq
    swa = synth.normal_bf16(synth.rng(s, "swa"), (B, S, D))
    swa_len, swa_pos0 = np.array([S], np.int32), np.array([ctx - W + 1], np.int64)
    q_pos = (ctx + np.arange(Tq, dtype=np.int64)).reshape(1, Tq)
    pos0 = np.array([ctx], np.int64)
    n_ent = torch.full((B,), P0, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, Tq, wl.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, 1, Tq, N), dtype=torch.uint8, device="cuda")  # one pass, as timed
    out = torch.empty((B, Tq, 64, D), dtype=torch.float32, device="cuda")
    csa.compress(cfg, _paged.dev(x), _paged.dev(pos0), _paged.dev(w), _paged.dev(w_idx), pm, pi, n_ent, status=st)
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pi, n_ent, N, topk, ws, status=st)
    csa.attend(cfg, _paged.dev(q), pm, n_ent, topk, _paged.dev(swa), _paged.dev(swa_len), _paged.dev(swa_pos0),
               _paged.dev(q_pos), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(n_ent.item()) == N
    diag = oracle.compress(x, pos0, w, w_idx, om, oi, r, wl.theta, diagnostics=True)
    exc = _check_compress(om, oi, pm, pi, diag, pos0, r, Tq // r, wl.cache)
    print("prefill compressor: %d near-boundary codes excused" % exc)
    rows = np.array([0, 1, 1000, 2047, 2048, Tq - 1])
    n_arr = np.array([N], np.int32)
    o_top, _, sc = oracle.index_topk(oi, n_arr, q_idx[:, rows], q_pos[:, rows], r, wl.topk, want_scores=True)
    g_top = topk.cpu().numpy()[:, rows]
    assert P.topk_mismatch(g_top.reshape(len(rows), -1), o_top.reshape(len(rows), -1), sc.reshape(len(rows), -1),
                           wl.topk, exact=False) == 0
    o_out = oracle.attend(om, n_arr, q[:, rows], o_top, swa, swa_len, swa_pos0, q_pos[:, rows], W, SCALE)
    err = P.attention_rel_err(out.cpu().numpy()[:, rows], o_out)
    print("prefill: attention max row rel err %.3g on %d sampled rows" % (err, len(rows)))
    assert err <= P.ATT_TOL


def test_multi_query_decode_block_every_row():
    """Multi-query decode: a block of 5 draft positions per sequence appended
    to 8 sequences of 32768 tokens, r = 2.  The compressor takes the block's
    two complete groups (the fifth token stays in the window rows); each
    sequence's 5 queries share one indexer group; every query row of every
    sequence is checked against the oracle."""
    wl = synth.WORKLOADS["mqdecode_b8_q5_ctx32768_r2_fp4"]
    B, r, Tq, ctx, W = wl.batch, wl.ratio, wl.tq, wl.ctx, wl.window
    Tc = Tq - Tq % r
    N, P0 = (ctx + Tq) // r, ctx // r
    pm, pi = _paged.cache_pair(B, N, D, wl.cache, wl.seed), _paged.cache_pair(B, N, CI, wl.cache, wl.seed + 1)
    om, oi = oracle.Cache(B, N, D, wl.cache), oracle.Cache(B, N, CI, wl.cache)
    for b in range(B):
        m, i = _prefix(wl, b, P0)
        om.codes[b, :P0], om.scales[b, :P0] = m.codes[0], m.scales[0]
        oi.codes[b, :P0], oi.scales[b, :P0] = i.codes[0], i.scales[0]
    _paged.upload(pm, om)
    _paged.upload(pi, oi)
    cfg = _cfg(wl)
    s = wl.seed
    x = synth.normal_bf16(synth.rng(s, "x_chunk"), (B, Tc, D))
    w = synth.merge_weights(synth.rng(s, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(s, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    q = synth.normal_bf16(synth.rng(s, "q"), (B, Tq, 64, D))
    q_idx = synth.normal_bf16(synth.rng(s, "q_idx"), (B, Tq, 32, CI))
    S = W - 1 + Tq
    swa = synth.normal_bf16(synth.rng(s, "swa"), (B, S, D))
    swa_len, swa_pos0 = np.full(B, S, np.int32), np.full(B, ctx - W + 1, np.int64)
    q_pos = np.tile(ctx + np.arange(Tq, dtype=np.int64), (B, 1))
    pos0 = np.full(B, ctx, np.int64)
    n_ent = torch.full((B,), P0, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, Tq, wl.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, Tq, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Tq, 64, D), dtype=torch.float32, device="cuda")
    csa.compress(cfg, _paged.dev(x), _paged.dev(pos0), _paged.dev(w), _paged.dev(w_idx), pm, pi, n_ent, status=st)
    csa.index_topk(cfg, _paged.dev(q_idx), _paged.dev(q_pos), pi, n_ent, N, topk, ws, status=st)
    csa.attend(cfg, _paged.dev(q), pm, n_ent, topk, _paged.dev(swa), _paged.dev(swa_len), _paged.dev(swa_pos0),
               _paged.dev(q_pos), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert (n_ent.cpu().numpy() == N).all()
    diag = oracle.compress(x, pos0, w, w_idx, om, oi, r, wl.theta, diagnostics=True)
    exc = _check_compress(om, oi, pm, pi, diag, pos0, r, Tc // r, wl.cache)
    print("multi-query block compressor: %d near-boundary codes excused" % exc)
    n_arr = np.full(B, N, np.int32)
    o_top, _, sc = oracle.index_topk(oi, n_arr, q_idx, q_pos, r, wl.topk, want_scores=True)
    g_top = topk.cpu().numpy()
    assert P.topk_mismatch(g_top.reshape(B * Tq, -1), o_top.reshape(B * Tq, -1), sc.reshape(B * Tq, -1), wl.topk,
                           exact=False) == 0
    assert (g_top >= 0).all()  # every query sees far more than k entries: no padding
    # the block's own entries are visible only from the positions that complete them
    assert not np.isin(g_top[:, 0], [P0, P0 + 1]).any() and not np.isin(g_top[:, 2], [P0 + 1]).any()
    o_out = oracle.attend(om, n_arr, q, o_top, swa, swa_len, swa_pos0, q_pos, W, SCALE)
    err = P.attention_rel_err(out.cpu().numpy(), o_out)
    print("multi-query block: attention max row rel err %.3g over %d rows" % (err, B * Tq))
    assert err <= P.ATT_TOL


def test_encoder_group_prefill_sampled_rows():
    """The encoder macro block on a prefill chunk: 4096 tokens appended to a
    1 M-token context, layer 2 Full (compress the chunk, index all 4096
    positions causally) and layers 3-7 Reuse, each layer with its own query
    and banded window; 5 query rows checked through all six layers."""
    wl = synth.WORKLOADS["encoder_group6_prefill_4096_on_1m_r2_fp4"]
    B, r, Tq, ctx, W = wl.batch, wl.ratio, wl.tq, wl.ctx, wl.window
    N, P0 = (ctx + Tq) // r, ctx // r
    pm, pi = _paged.cache_pair(B, N, D, wl.cache, wl.seed), _paged.cache_pair(B, N, CI, wl.cache, wl.seed + 1)
    m, i = _prefix(wl, 0, P0)
    om, oi = oracle.Cache(1, N, D, wl.cache), oracle.Cache(1, N, CI, wl.cache)
    om.codes[0, :P0], om.scales[0, :P0] = m.codes[0], m.scales[0]
    oi.codes[0, :P0], oi.scales[0, :P0] = i.codes[0], i.scales[0]
    _paged.upload(pm, om)
    _paged.upload(pi, oi)
    cfg = _cfg(wl)
    s = wl.seed
    x = synth.normal_bf16(synth.rng(s, "x_chunk"), (B, Tq, D))
    w = synth.merge_weights(synth.rng(s, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(s, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    S = W - 1 + Tq
    swa_len, swa_pos0 = np.array([S], np.int32), np.array([ctx - W + 1], np.int64)
    q_pos = (ctx + np.arange(Tq, dtype=np.int64)).reshape(1, Tq)
    pos0 = np.array([ctx], np.int64)
    n_ent = torch.full((B,), P0, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, Tq, wl.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, 1, Tq, N), dtype=torch.uint8, device="cuda")  # one pass, as timed
    state = csa.GroupState(pm, pi, n_ent, N, topk, None, ws, st)
    rows = np.array([0, 1, 2047, 2048, Tq - 1])
    n_arr = np.array([N], np.int32)
    o_top = None
    for layer, mode in wl.layers:
        ls = s * 1000 + layer
        q = synth.normal_bf16(synth.rng(ls, "q"), (B, Tq, 64, D))
        swa = synth.normal_bf16(synth.rng(ls, "swa"), (B, S, D))
        q_idx = synth.normal_bf16(synth.rng(ls, "q_idx"), (B, Tq, 32, CI)) if mode != "reuse" else None
        out = torch.empty((B, Tq, 64, D), dtype=torch.float32, device="cuda")
        kw = {}
        if mode == "full":
            kw = dict(x=_paged.dev(x), pos0=_paged.dev(pos0), merge_w=_paged.dev(w), w_idx=_paged.dev(w_idx))
        csa.layer(cfg, {"full": csa.MODE_FULL, "reuse": csa.MODE_REUSE}[mode], state, _paged.dev(q_pos),
                  _paged.dev(q), _paged.dev(swa), _paged.dev(swa_len), _paged.dev(swa_pos0), out,
                  q_idx=None if q_idx is None else _paged.dev(q_idx), **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        if mode == "full":
            assert int(n_ent.item()) == N
            diag = oracle.compress(x, pos0, w, w_idx, om, oi, r, wl.theta, diagnostics=True)
            exc = _check_compress(om, oi, pm, pi, diag, pos0, r, Tq // r, wl.cache)
            print("encoder group prefill compressor: %d near-boundary codes excused" % exc)
            o_top, _, sc = oracle.index_topk(oi, n_arr, q_idx[:, rows], q_pos[:, rows], r, wl.topk, want_scores=True)
            g_top = topk.cpu().numpy()[:, rows]
            assert P.topk_mismatch(g_top.reshape(len(rows), -1), o_top.reshape(len(rows), -1),
                                   sc.reshape(len(rows), -1), wl.topk, exact=False) == 0
        o_out = oracle.attend(om, n_arr, q[:, rows], o_top, swa, swa_len, swa_pos0, q_pos[:, rows], W, SCALE)
        err = P.attention_rel_err(out.cpu().numpy()[:, rows], o_out)
        print("encoder group prefill L%d %s: attention max row rel err %.3g" % (layer, mode, err))
        assert err <= P.ATT_TOL, (layer, err)
