"""Pins of the oracle's sparse attention (one softmax over top-k entries and
the window rows, key = value): the dense limit, convex-hull readout, closed
forms for one and two rows, uniform weights at q = 0, window bounds, and the
Reuse-mode identities of the cross-layer schedule."""
import math
import os

import numpy as np
import pytest

import oracle
import synth

D, HM = 512, 64
SCALE = 1 / math.sqrt(D)


def _main_cache(seed, B, N, dtype="fp4"):
    c = oracle.Cache(B, N, D, dtype)
    g = synth.rng(seed, "main_cache")
    if dtype == "fp4":
        for b in range(B):
            c.codes[b], c.scales[b] = synth.fp4_bytes(g, N, D)
    else:
        c.bf16[:] = synth.normal_bf16(g, (B, N, D))
    return c


def _swa(seed, B, S):
    return synth.normal_bf16(synth.rng(seed, "swa"), (B, S, D))


def test_dense_limit_k_at_least_n():
    """k >= N: selecting every visible entry equals dense attention over all
    entries plus the window (separately coded)."""
    for dtype, r in (("fp4", 2), ("bf16", 1)):
        B, N, W = 2, 37, 8
        main = _main_cache(1, B, N, dtype)
        q = synth.normal_bf16(synth.rng(1, "q"), (B, 2, HM, D))
        q_pos = np.array([[2 * N - 1, 40], [2 * N - 1, 13]], np.int64) if r == 2 else \
            np.array([[N - 1, 20], [N - 1, 3]], np.int64)
        n_ent = np.array([N, N - 5], np.int32)
        swa = _swa(1, B, 100)
        swa_pos0 = np.array([0, 0], np.int64)
        swa_len = np.array([100, 100], np.int32)
        k = 64
        topk = np.full((B, 2, k), -1, np.int32)
        for b in range(B):
            for t in range(2):
                nv = min((q_pos[b, t] - (r - 1)) // r + 1, n_ent[b])
                topk[b, t, :nv] = np.arange(nv)
        o1 = oracle.attend(main, n_ent, q, topk, swa, swa_len, swa_pos0, q_pos, W, SCALE)
        o2 = oracle.attend_dense(main, n_ent, q, swa, swa_len, swa_pos0, q_pos, r, W, SCALE)
        np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)


def test_convex_hull_and_probability_mass():
    """Key = value makes every output a convex combination of the read rows:
    each output channel lies within the rows' range, and identical rows give
    back that row whatever the query."""
    B, N, W = 1, 50, 16
    main = _main_cache(2, B, N)
    q = synth.normal_bf16(synth.rng(2, "q"), (B, 1, HM, D), std=4.0)
    topk = synth.rng(2, "ids").permutation(N)[:20].astype(np.int32).reshape(1, 1, 20)
    swa = _swa(2, B, W)
    q_pos = np.array([[200]], np.int64)
    args = (np.array([N], np.int32), q, topk, swa, np.array([W], np.int32), np.array([200 - W + 1]),
            q_pos, W, SCALE)
    out = oracle.attend(main, *args)
    rows = np.concatenate([main.values()[0, topk[0, 0]], synth.bf16_bits_to_f64(swa[0])])
    lo, hi = rows.min(axis=0), rows.max(axis=0)
    assert (out[0, 0] >= lo - 1e-12).all() and (out[0, 0] <= hi + 1e-12).all()
    same = oracle.Cache(1, N, D, "bf16")
    row = synth.normal_bf16(synth.rng(3, "row"), (D,))
    same.bf16[0, :] = row
    swa_same = np.broadcast_to(row, (1, W, D)).copy()
    out2 = oracle.attend(same, np.array([N], np.int32), q, topk, swa_same, np.array([W], np.int32),
                         np.array([200 - W + 1]), q_pos, W, SCALE)
    np.testing.assert_allclose(out2[0, 0], np.broadcast_to(synth.bf16_bits_to_f64(row), (HM, D)),
                               rtol=1e-14, atol=1e-15)


def test_zero_query_gives_mean_of_union():
    B, N, W = 1, 30, 5
    main = _main_cache(4, B, N)
    q = np.zeros((1, 1, HM, D), np.uint16)
    ids = np.array([[[3, 7, 8, 21, -1, -1]]], np.int32)
    swa = _swa(4, B, W)
    q_pos = np.array([[90]], np.int64)
    out = oracle.attend(main, np.array([N], np.int32), q, ids, swa, np.array([W], np.int32),
                        np.array([86]), q_pos, W, SCALE)
    rows = np.concatenate([main.values()[0, [3, 7, 8, 21]], synth.bf16_bits_to_f64(swa[0])])
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(rows.mean(axis=0), (HM, D)), rtol=1e-13,
                               atol=1e-15)


def test_one_and_two_row_closed_forms():
    """One row: output = that row, lse = scale * q.c.  Two rows: weights are the
    logistic function of the logit difference."""
    N = 4
    main = _main_cache(5, 1, N)
    vals = main.values()[0]
    q = synth.normal_bf16(synth.rng(5, "q"), (1, 1, HM, D))
    qf = synth.bf16_bits_to_f64(q)[0, 0]
    empty_swa = np.zeros((1, 1, D), np.uint16)
    out, lse = oracle.attend(main, np.array([N], np.int32), q, np.array([[[2, -1]]], np.int32), empty_swa,
                             np.array([0], np.int32), np.array([0]), np.array([[10]]), 128, SCALE,
                             want_lse=True)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(vals[2], (HM, D)), rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], SCALE * (qf @ vals[2]), rtol=1e-12)
    out2 = oracle.attend(main, np.array([N], np.int32), q, np.array([[[1, 3]]], np.int32), empty_swa,
                         np.array([0], np.int32), np.array([0]), np.array([[10]]), 128, SCALE)
    dl = SCALE * (qf @ vals[3] - qf @ vals[1])
    p3 = 1 / (1 + np.exp(-dl))
    want = (1 - p3)[:, None] * vals[1] + p3[:, None] * vals[3]
    np.testing.assert_allclose(out2[0, 0], want, rtol=1e-12, atol=1e-14)


def test_window_bounds_and_empty_slots():
    """Rows outside t-W+1..t and -1 top-k slots never contribute: planting a
    huge row just outside the window, or at an id only reachable through a -1
    slot, leaves the output unchanged."""
    N, W, S = 10, 4, 12
    main = _main_cache(6, 1, N)
    q = synth.normal_bf16(synth.rng(6, "q"), (1, 1, HM, D))
    swa = _swa(6, 1, S)
    t = 107  # rows at positions 100..111; window = 104..107
    args = dict(swa_len=np.array([S], np.int32), swa_pos0=np.array([100]), q_pos=np.array([[t]]),
                window=W, scale=SCALE)
    ids = np.array([[[1, -1, 4, -1]]], np.int32)
    base = oracle.attend(main, np.array([N], np.int32), q, ids, swa, **args)
    swa2 = swa.copy()
    big = oracle.bf16_round(1000.0)
    swa2[0, 3, :] = big   # position 103: just before the window
    swa2[0, 8, :] = big   # position 108: after the query
    out = oracle.attend(main, np.array([N], np.int32), q, ids, swa2, **args)
    np.testing.assert_array_equal(out, base)
    # the window at the start of a sequence is clipped at position 0
    out0 = oracle.attend(main, np.array([N], np.int32), q, ids, swa, swa_len=np.array([S], np.int32),
                         swa_pos0=np.array([0]), q_pos=np.array([[1]]), window=W, scale=SCALE)
    rows = np.concatenate([main.values()[0, [1, 4]], synth.bf16_bits_to_f64(swa[0, :2])])
    out_dense = oracle.attend(main, np.array([N], np.int32), np.zeros_like(q), ids, swa,
                              swa_len=np.array([S], np.int32), swa_pos0=np.array([0]),
                              q_pos=np.array([[1]]), window=W, scale=SCALE)
    np.testing.assert_allclose(out_dense[0, 0, 0], rows.mean(axis=0), rtol=1e-13)
    assert np.isfinite(out0).all()


def test_out_of_range_topk_is_rejected():
    main = _main_cache(7, 1, 5)
    q = synth.normal_bf16(synth.rng(7, "q"), (1, 1, HM, D))
    with pytest.raises(ValueError):
        oracle.attend(main, np.array([5], np.int32), q, np.array([[[5]]], np.int32),
                      np.zeros((1, 1, D), np.uint16), np.array([0], np.int32), np.array([0]),
                      np.array([[10]]), 4, SCALE)


def _gold(name):
    out = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", name)):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            out[k] = v
    return out


def test_decoder_schedule_reuse_sources():
    """Layer 20 Full, Reindex at 24/28/32/36, Reuse follows the latest
    indexing layer: 21-23 <- 20, 25-27 <- 24, ..., 37-39 <- 36."""
    modes = oracle.layer_modes(synth.DECODER_GROUP)
    gold = _gold("hsi_config.txt")
    idx_src = [int(v) for v in gold["index_source_layers"][0:]]
    assert sorted(l for l, (m, _) in modes.items() if m in ("full", "reindex")) == [
        l for l in idx_src if l >= 20]
    for l, (m, src) in modes.items():
        if m == "reuse":
            assert src == max(s for s in idx_src if s < l)
        else:
            assert src == l
    assert int(gold["candidate_topk_blocks"][0]) * int(gold["candidate_block_size"][0]) == int(
        gold["pool_positions"][0])
    with pytest.raises(ValueError):
        oracle.layer_modes([(5, "reuse")])


def _reuse_group(seed, N=300, W=128, k=64, nb=16):
    """A decoder-style group state: a seeded FP4 main and indexer cache of N
    entries (r = 1), a Full layer with HSI run on it."""
    main = _main_cache(seed, 1, N)
    idx = oracle.Cache(1, N, 128, "fp4")
    idx.codes[0], idx.scales[0] = synth.fp4_bytes(synth.rng(seed, "idx"), N, 128)
    st = oracle.GroupState(main, idx, [N], r=1, k=k, hsi_blocks=nb)
    q_pos = np.array([[N - 1]])
    a = dict(swa_len=np.array([W], np.int32), swa_pos0=np.array([N - W]), window=W, scale=SCALE)
    q_src = synth.normal_bf16(synth.rng(seed, "q_src"), (1, 1, HM, D))
    swa_src = _swa(seed, 1, W)
    q_idx = synth.normal_bf16(synth.rng(seed, "q_idx"), (1, 1, 32, 128))
    src = oracle.layer("full", st, q_pos, q_src, swa_src, q_idx=q_idx, **a)
    return st, q_pos, a, q_src, swa_src, src


def test_reuse_layer_reads_only_the_source_top_k():
    """Reuse (hn.213312.xyz sec. 2.3.2, access table of sec. 3.2): the layer
    reads the latest published top-k and writes nothing.  Checked by
    behaviour, not by restating the attention: (1) the published top-k and
    pool and both caches are bit-identical after a Reuse layer; (2) a huge
    row planted at an id outside the source top-k leaves the Reuse output
    bit-identical; (3) changing a row inside the source top-k changes it;
    (4) given the source layer's own query and window rows, a Reuse layer
    reproduces the source layer's output exactly."""
    st, q_pos, a, q_src, swa_src, src = _reuse_group(8)
    topk0, pool0 = st.topk.copy(), st.pool.copy()
    codes0, scales0, icodes0 = st.main.codes.copy(), st.main.scales.copy(), st.idx.codes.copy()
    q_own = synth.normal_bf16(synth.rng(8, "q_own"), (1, 1, HM, D))
    swa_own = _swa(9, 1, a["window"])
    base = oracle.layer("reuse", st, q_pos, q_own, swa_own, **a)
    # (1) nothing published or cached changed
    np.testing.assert_array_equal(st.topk, topk0)
    np.testing.assert_array_equal(st.pool, pool0)
    np.testing.assert_array_equal(st.main.codes, codes0)
    np.testing.assert_array_equal(st.main.scales, scales0)
    np.testing.assert_array_equal(st.idx.codes, icodes0)
    # (2) an entry outside the source top-k, made huge, is never read
    sel = set(topk0[0, 0][topk0[0, 0] >= 0].tolist())
    outside = next(j for j in range(st.main.n_cap) if j not in sel)
    st.main.codes[0, outside, :] = 0x77    # every element +6
    st.main.scales[0, outside, :] = 0x7E   # scale 448
    np.testing.assert_array_equal(oracle.layer("reuse", st, q_pos, q_own, swa_own, **a), base)
    st.main.codes[0, outside], st.main.scales[0, outside] = codes0[0, outside], scales0[0, outside]
    # (3) an entry inside the source top-k is read
    inside = sorted(sel)[len(sel) // 2]
    st.main.codes[0, inside, :] = 0x77
    st.main.scales[0, inside, :] = 0x7E
    changed = oracle.layer("reuse", st, q_pos, q_own, swa_own, **a)
    assert np.abs(changed - base).max() > 1e-3
    st.main.codes[0, inside], st.main.scales[0, inside] = codes0[0, inside], scales0[0, inside]
    # (4) the source layer's query and window rows give the source output
    np.testing.assert_array_equal(oracle.layer("reuse", st, q_pos, q_src, swa_src, **a), src)


def test_reindex_publishes_from_the_pool_and_writes_no_cache():
    """Reindex (hn.213312.xyz sec. 2.3.2, sec. 2.3.4): its published top-k
    lies inside the Full layer's pool, the pool and caches are unchanged,
    and a Reuse layer after it reads the Reindex layer's top-k."""
    st, q_pos, a, _, _, _ = _reuse_group(10)
    pool0 = st.pool.copy()
    codes0, icodes0 = st.main.codes.copy(), st.idx.codes.copy()
    q = synth.normal_bf16(synth.rng(10, "q_r"), (1, 1, HM, D))
    swa = _swa(11, 1, a["window"])
    q_idx = synth.normal_bf16(synth.rng(10, "q_idx_r"), (1, 1, 32, 128))
    out_r = oracle.layer("reindex", st, q_pos, q, swa, q_idx=q_idx, **a)
    np.testing.assert_array_equal(st.pool, pool0)
    np.testing.assert_array_equal(st.main.codes, codes0)
    np.testing.assert_array_equal(st.idx.codes, icodes0)
    blocks = set(pool0[0, 0][pool0[0, 0] >= 0].tolist())
    ids = st.topk[0, 0][st.topk[0, 0] >= 0]
    assert len(ids) > 0 and all(int(j) // 8 in blocks for j in ids)
    np.testing.assert_array_equal(oracle.layer("reuse", st, q_pos, q, swa, **a), out_r)
    with pytest.raises(ValueError):
        oracle.layer("reindex", oracle.GroupState(st.main, st.idx, [300], 1, 64, 16), q_pos, q, swa,
                     q_idx=q_idx, **a)
