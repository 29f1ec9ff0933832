"""Pins of the oracle's variants for the pages' own formats: FP4 indexer
queries (sec. 2.4.4: V4 already trained its indexer Q/K in FP4), and two
storage variants:
the 68-byte indexer entry (FP4 with one E4M3 scale per 32 channels;
hn.213312.xyz sec. 3.1 prints 68 B per 128-channel indexer entry) and the
FP8 window rows (sec. 2.4.4: the SWA KV stays FP8), read as OCP MXFP8 --
E4M3 elements with one power-of-two E8M0 scale per 32 channels.  Checked by
brute-force searches in exact rationals, binade properties of the block
scale, round trips, byte counts, and reductions to the pinned bf16 paths."""
import math
import os
from fractions import Fraction

import numpy as np

import oracle
import synth
from tests.test_oracle_codec import _brute_encode_group, _nearest, _table


# ------------------------------------------------- FP4, 32-channel scales ----

def test_fp4_group32_brute_force():
    rng = np.random.default_rng(31)
    groups = [rng.standard_normal(32) for _ in range(30)]
    groups += [rng.standard_normal(32) * 1e-4, rng.standard_normal(32) * 3000, np.zeros(32)]
    g = rng.standard_normal(32)
    g[17] = 6 * (oracle.e4m3_value(0x30) + oracle.e4m3_value(0x31)) / 2  # scale tie in the second half
    groups.append(g)
    x = np.concatenate(groups)
    codes, scales = oracle.fp4_encode(x[None, :], group=32)
    assert scales.shape == (1, len(groups))
    for gi in range(len(groups)):
        want_codes, want_sc = _brute_encode_group(x[32 * gi:32 * gi + 32])
        assert scales[0, gi] == want_sc, gi
        got = [(codes[0, (32 * gi + i) // 2] >> (4 * (i % 2))) & 15 for i in range(32)]
        assert got == want_codes, gi


def test_fp4_group32_entry_is_the_pages_68_bytes():
    gold = {r[0]: r[1:] for r in _table("kv_bytes_per_token.txt")}
    c, s = oracle.fp4_encode(np.zeros((1, 128)), group=32)
    assert c.nbytes + s.nbytes == int(gold["indexer_entry_bytes"][0]) == 68
    c, s = oracle.fp4_encode(np.zeros((1, 512)))
    assert c.nbytes + s.nbytes == int(gold["main_entry_bytes"][0])


def test_fp4_group32_equals_group16_when_both_halves_share_amax():
    """With equal half maxima the one 32-channel scale is the 16-channel scale
    of either half, so the codes agree with the pinned per-16 encoder."""
    rng = np.random.default_rng(32)
    x = rng.standard_normal((20, 128))
    for blk in range(4):
        a = x[:, 32 * blk:32 * blk + 16]
        b = x[:, 32 * blk + 16:32 * blk + 32]
        m = np.maximum(np.abs(a).max(1), np.abs(b).max(1))
        a[np.arange(20), np.abs(a).argmax(1)] = m * np.sign(a[np.arange(20), np.abs(a).argmax(1)])
        b[np.arange(20), np.abs(b).argmax(1)] = m * np.sign(b[np.arange(20), np.abs(b).argmax(1)])
    c32, s32 = oracle.fp4_encode(x, group=32)
    c16, s16 = oracle.fp4_encode(x)
    np.testing.assert_array_equal(c32, c16)
    np.testing.assert_array_equal(np.repeat(s32, 2, axis=1), s16)
    np.testing.assert_array_equal(oracle.fp4_decode(c32, s32), oracle.fp4_decode(c16, s16))


def _g32_cache(seed, B, N):
    g = np.random.default_rng(seed)
    c = oracle.Cache(B, N, 128, "fp4g32")
    c.codes[:] = g.integers(0, 256, size=c.codes.shape, dtype=np.uint8)
    c.scales[:] = g.integers(0x20, 0x3D, size=c.scales.shape, dtype=np.uint8)
    return c


def _as_bf16_cache(c):
    """A bf16 cache holding the decoded values (exact: an E2M1 magnitude times
    an E4M3 scale has at most 6 significant bits)."""
    v = c.values()
    bc = oracle.Cache(c.B, c.n_cap, c.channels, "bf16")
    bc.bf16[:] = np.vectorize(oracle.bf16_round, otypes=[np.uint16])(v)
    np.testing.assert_array_equal(bc.values(), v)
    return bc


def test_index_topk_on_68_byte_entries_equals_the_decoded_bf16_cache():
    B, N, k = 2, 300, 64
    c = _g32_cache(33, B, N)
    bc = _as_bf16_cache(c)
    q_idx = synth.normal_bf16(synth.rng(33, "q"), (B, 2, 32, 128))
    q_pos = np.array([[N - 1, 150], [N - 1, 40]], np.int64)
    n_ent = np.array([N, N - 7], np.int32)
    t1, p1, s1 = oracle.index_topk(c, n_ent, q_idx, q_pos, 1, k, hsi_blocks=8, want_pool=True, want_scores=True)
    t2, p2, s2 = oracle.index_topk(bc, n_ent, q_idx, q_pos, 1, k, hsi_blocks=8, want_pool=True, want_scores=True)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(p1, p2)
    np.testing.assert_array_equal(s1, s2)


def test_compress_into_68_byte_indexer_entries():
    """Same main cache and the same pre-quantisation indexer K as the per-16
    layout; the stored indexer entries are the 32-channel encoding of K."""
    B, T, r, D, Ci = 2, 8, 2, 512, 128
    x = synth.normal_bf16(synth.rng(34, "x"), (B, T, D))
    w = synth.merge_weights(synth.rng(34, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(34, "w_idx"), (D, Ci), std=1 / math.sqrt(D))
    pos0 = np.array([0, 6], np.int64)
    n = 16
    m1, i1 = oracle.Cache(B, n, D, "fp4"), oracle.Cache(B, n, Ci, "fp4")
    m2, i2 = oracle.Cache(B, n, D, "fp4"), oracle.Cache(B, n, Ci, "fp4g32")
    d1 = oracle.compress(x, pos0, w, w_idx, m1, i1, r, 1e4, diagnostics=True)
    d2 = oracle.compress(x, pos0, w, w_idx, m2, i2, r, 1e4, diagnostics=True)
    np.testing.assert_array_equal(m1.codes, m2.codes)
    np.testing.assert_array_equal(m1.scales, m2.scales)
    np.testing.assert_array_equal(d1["pre_idx"], d2["pre_idx"])
    for b in range(B):
        j = np.arange(pos0[b] // r, pos0[b] // r + T // r)
        want_c, want_s = oracle.fp4_encode(d2["pre_idx"][b], group=32)
        np.testing.assert_array_equal(i2.codes[b, j], want_c)
        np.testing.assert_array_equal(i2.scales[b, j], want_s)


# ------------------------------------------------------- MXFP8 window rows ----

def test_e8m0_is_a_biased_power_of_two():
    assert oracle.e8m0_value(127) == 1.0
    for b in range(254):
        assert oracle.e8m0_value(b + 1) == 2 * oracle.e8m0_value(b)
    assert oracle.e8m0_value(0) == math.ldexp(1.0, -127)
    assert math.isnan(oracle.e8m0_value(255))


def _blocks(rng):
    out = [rng.standard_normal(32) * s for s in (1.0, 1e-3, 37.0, 1e5, 3e-30)]
    out.append(np.zeros(32))
    z = rng.standard_normal(32)
    z[5] = 8.0  # amax a power of two: the block maximum codes to 256 (E4M3 2^8)
    out.append(z)
    return out


def test_mxfp8_block_scale_puts_the_maximum_in_the_top_binade():
    rng = np.random.default_rng(35)
    blocks = _blocks(rng)
    for _ in range(60):
        blocks.append(rng.standard_normal(32) * math.exp(rng.uniform(-20, 20)))
    x = np.concatenate(blocks)
    row = oracle.mxfp8_encode(x[None, :])[0]
    nb = len(blocks)
    assert row.shape == (32 * nb + nb,)
    for gi, blk in enumerate(blocks):
        sb = int(row[32 * nb + gi])
        amax = Fraction(float(np.abs(blk).max()))
        if amax == 0:
            assert sb == 0 and not row[32 * gi:32 * gi + 32].any()
            continue
        X = Fraction(2) ** (sb - 127)
        assert 256 <= amax / X < 512, (gi, sb)


def test_mxfp8_elements_brute_force():
    rng = np.random.default_rng(36)
    blocks = _blocks(rng)
    # exact E4M3 midpoints (ties to the even code) and values past 448 X
    g = np.zeros(32)
    g[0] = 300.0  # X = 2^0 for amax in [256, 512)
    e4 = [oracle.e4m3_value(b) for b in range(0x7F)]
    for i, c in enumerate(range(40, 70)):
        g[1 + i] = (e4[c] + e4[c + 1]) / 2 * (-1) ** i
    g[31] = 470.0  # above 448: saturates
    blocks.append(g)
    x = np.concatenate(blocks)
    nb = len(blocks)
    row = oracle.mxfp8_encode(x[None, :])[0]
    for gi, blk in enumerate(blocks):
        X = Fraction(2) ** (int(row[32 * nb + gi]) - 127)
        for i, v in enumerate(blk):
            y = abs(Fraction(float(v))) / X
            mag = min(_nearest(e4, y), 126) if y <= 448 else 126
            want = (mag | 0x80) if (v < 0 and mag != 0) else mag
            assert row[32 * gi + i] == want, (gi, i, float(v))
    assert row[32 * (nb - 1) + 31] == 0x7E


def test_mxfp8_round_trip_on_representable_blocks():
    rng = np.random.default_rng(37)
    n = 40
    codes = rng.integers(0, 0x7F, size=(n, 512)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(n, 512)) << 7).astype(np.uint8)
    codes[:, ::32] = rng.integers(0x78, 0x7F, size=(n, 16)).astype(np.uint8)  # top binade: 256..448
    codes[(codes & 0x7F) == 0] = 0  # +0 for zero
    scales = rng.integers(100, 150, size=(n, 16)).astype(np.uint8)
    rows = np.concatenate([codes, scales], axis=1)
    vals = oracle.mxfp8_decode(rows)
    np.testing.assert_array_equal(oracle.mxfp8_encode(vals), rows)


def test_mxfp8_window_row_is_528_bytes_and_swa_encode_reads_bf16():
    bits = synth.normal_bf16(synth.rng(38, "swa"), (2, 3, 512))
    rows = oracle.swa_encode(bits)
    assert rows.shape == (2, 3, 528) and rows.dtype == np.uint8
    np.testing.assert_array_equal(rows, oracle.mxfp8_encode(oracle.bf16_bits_to_f64(bits)))


def test_attend_on_mxfp8_rows_equals_bf16_rows_of_the_decoded_values():
    """Decoded MXFP8 values (4 significant bits times a power of two) are
    exact in bf16, so attention over the FP8 rows equals attention over bf16
    rows holding those values (the bf16 path is pinned separately)."""
    D, N, W, S = 512, 40, 16, 20
    main = oracle.Cache(1, N, D, "fp4")
    main.codes[0], main.scales[0] = synth.fp4_bytes(synth.rng(39, "main"), N, D)
    q = synth.normal_bf16(synth.rng(39, "q"), (1, 2, 64, D))
    topk = np.array([[[1, 5, 9, -1, 30], [0, 2, 4, 6, -1]]], np.int32)
    swa_bits = synth.normal_bf16(synth.rng(39, "swa"), (1, S, D))
    rows = oracle.swa_encode(swa_bits)
    dec = oracle.mxfp8_decode(rows)
    dec_bits = np.vectorize(oracle.bf16_round, otypes=[np.uint16])(dec)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(dec_bits), dec)
    args = (np.array([S], np.int32), np.array([100], np.int64), np.array([[110, 119]], np.int64), W, 1 / math.sqrt(D))
    o8, l8 = oracle.attend(main, np.array([N], np.int32), q, topk, rows, *args, want_lse=True)
    ob, lb = oracle.attend(main, np.array([N], np.int32), q, topk, dec_bits, *args, want_lse=True)
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)
    d8 = oracle.attend_dense(main, np.array([N], np.int32), q, rows, *args[:3], 1, W, 1 / math.sqrt(D))
    db = oracle.attend_dense(main, np.array([N], np.int32), q, dec_bits, *args[:3], 1, W, 1 / math.sqrt(D))
    np.testing.assert_array_equal(d8, db)


# ------------------------------------------------- FP4 indexer queries ----

def test_fp4_queries_equal_bf16_queries_holding_their_fp4_values():
    """Scoring with FP4 queries equals scoring with bf16 queries that hold the
    queries' FP4 encodings read back (exact in bf16: at most 6 significant
    bits), on both cache formats; the FP4 queries are the pinned encoder's."""
    B, Tq, N, k = 2, 2, 400, 64
    for dtype in ("fp4", "fp4g32"):
        c = oracle.Cache(B, N, 128, dtype)
        g = synth.rng(50, dtype)
        for b in range(B):
            c.codes[b], c.scales[b] = synth.fp4_bytes(g, N, 128, group=16 if dtype == "fp4" else 32)
        q_idx = synth.normal_bf16(synth.rng(50, "q"), (B, Tq, 32, 128))
        qc, qs = oracle.fp4_encode(oracle.bf16_bits_to_f64(q_idx))
        qv = oracle.fp4_decode(qc, qs)
        q_bits = np.vectorize(oracle.bf16_round, otypes=[np.uint16])(qv)
        np.testing.assert_array_equal(oracle.bf16_bits_to_f64(q_bits), qv)
        q_pos = np.array([[N - 1, 200], [N - 1, 17]], np.int64)
        n_ent = np.array([N, N - 3], np.int32)
        hw = synth.rng(50, "hw").uniform(0, 2, size=(B, Tq, 32)).astype(np.float32)
        t1, p1, s1 = oracle.index_topk(c, n_ent, q_idx, q_pos, 1, k, head_w=hw, hsi_blocks=8, want_pool=True,
                                       want_scores=True, q_fp4=True)
        t2, p2, s2 = oracle.index_topk(c, n_ent, q_bits, q_pos, 1, k, head_w=hw, hsi_blocks=8, want_pool=True,
                                       want_scores=True)
        np.testing.assert_array_equal(t1, t2)
        np.testing.assert_array_equal(p1, p2)
        np.testing.assert_array_equal(s1, s2)
        # and the FP4 queries do change the scores
        _, _, s3 = oracle.index_topk(c, n_ent, q_idx, q_pos, 1, k, head_w=hw, want_scores=True)
        assert not np.array_equal(s1, s3)
