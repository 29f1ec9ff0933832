"""Pins of the oracle's compressor (merge 2:1 / 1:1, RoPE after the merge,
encode, indexer-K projection from the stored entry) by special cases that
reduce it to something else: selection, identity, complex rotation, norms."""
import numpy as np

import oracle
import synth

D, CI = 512, 128


def _run(x, pos0, w, w_idx, r, theta, dtype, rope_dims=64, n_cap=None):
    B, T, _ = x.shape
    n_cap = n_cap or int(max(pos0) // r + T // r + 3)
    main = oracle.Cache(B, n_cap, D, dtype)
    idx = oracle.Cache(B, n_cap, CI, dtype)
    diag = oracle.compress(x, pos0, w, w_idx, main, idx, r, theta, rope_dims, diagnostics=True)
    return main, idx, diag


def _inputs(seed, B, T, r):
    x = synth.normal_bf16(synth.rng(seed, "x"), (B, T, D))
    w = synth.merge_weights(synth.rng(seed, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(seed, "w_idx"), (D, CI), std=1 / np.sqrt(D))
    return x, w, w_idx


def test_ratio2_halves_entry_count_and_touches_nothing_else():
    x, w, w_idx = _inputs(0, 2, 8, 2)
    pos0 = np.array([0, 6], np.int64)
    main, idx, diag = _run(x, pos0, w, w_idx, 2, 1e4, "fp4", n_cap=12)
    assert diag["pre_main"].shape == (2, 4, D)
    written = (main.scales != 0).any(axis=2) | (main.codes != 0).any(axis=2)
    assert written[0].tolist() == [True] * 4 + [False] * 8
    assert written[1].tolist() == [False] * 3 + [True] * 4 + [False] * 5


def test_merge_reduces_to_selection_and_is_linear():
    """w1 = 0 selects the even token, w0 = 0 the odd one; swapping the two
    tokens together with the two weight rows changes nothing; doubling x
    doubles the merged entry (no RoPE: rope_dims = 0)."""
    x, w, w_idx = _inputs(1, 1, 4, 2)
    xf = synth.bf16_bits_to_f64(x)
    w_even = w.copy()
    w_even[1] = 0
    _, _, d = _run(x, np.array([0]), w_even, w_idx, 2, 1e4, "fp4", rope_dims=0)
    np.testing.assert_array_equal(d["pre_main"][0], w_even[0].astype(np.float64) * xf[0, 0::2])
    w_odd = w.copy()
    w_odd[0] = 0
    _, _, d = _run(x, np.array([0]), w_odd, w_idx, 2, 1e4, "fp4", rope_dims=0)
    np.testing.assert_array_equal(d["pre_main"][0], w_odd[1].astype(np.float64) * xf[0, 1::2])
    _, _, d1 = _run(x, np.array([0]), w, w_idx, 2, 1e4, "fp4", rope_dims=0)
    xs = x.copy()
    xs[:, 0::2], xs[:, 1::2] = x[:, 1::2], x[:, 0::2]
    _, _, d2 = _run(xs, np.array([0]), w[::-1].copy(), w_idx, 2, 1e4, "fp4", rope_dims=0)
    np.testing.assert_allclose(d1["pre_main"], d2["pre_main"], rtol=0, atol=1e-15)
    x2 = synth.normal_bf16(synth.rng(9, "x"), (1, 4, D), std=1.0)
    x2f = synth.bf16_bits_to_f64(x2)
    x2d = (np.asarray(x2f * 2, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    _, _, da = _run(x2, np.array([0]), w, w_idx, 2, 1e4, "fp4", rope_dims=0)
    _, _, db = _run(x2d, np.array([0]), w, w_idx, 2, 1e4, "fp4", rope_dims=0)
    np.testing.assert_array_equal(db["pre_main"], 2 * da["pre_main"])


def test_rope_is_complex_rotation_at_last_covered_position():
    """With r = 1 and unit weights the compressor is RoPE + encode.  Each pair
    (2i, 2i+1) of the first 64 channels must equal (x_2i + i x_2i+1) times
    exp(i p theta^(-2i/64)) with p the entry's position; the other channels
    pass through; r = 2 rotates entry j at position 2j + 1."""
    for r in (1, 2):
        x, w, w_idx = _inputs(2, 1, 6, r)
        w = np.ones((r, D), np.float32) if r == 1 else w
        pos0 = np.array([10 * r], np.int64)
        _, _, d = _run(x, pos0, w, w_idx, r, 1e4, "fp4")
        xf = synth.bf16_bits_to_f64(x)[0]
        merged = sum(w[i].astype(np.float64) * xf[i::r] for i in range(r))
        for m in range(merged.shape[0]):
            p = r * (pos0[0] // r + m) + r - 1
            z = merged[m, 0:64:2] + 1j * merged[m, 1:64:2]
            ang = p * np.power(1e4, -np.arange(32) * 2.0 / 64)
            zr = z * np.exp(1j * ang)
            got = d["pre_main"][0, m]
            np.testing.assert_allclose(got[0:64:2], zr.real, rtol=0, atol=1e-12)
            np.testing.assert_allclose(got[1:64:2], zr.imag, rtol=0, atol=1e-12)
            np.testing.assert_allclose(got[64:], merged[m, 64:], rtol=0, atol=1e-15)


def test_rope_preserves_pair_norms_and_is_identity_at_position_zero():
    x, w, w_idx = _inputs(3, 1, 1, 1)
    w = np.ones((1, D), np.float32)
    _, _, d = _run(x, np.array([0]), w, w_idx, 1, 1.6e5, "bf16")
    xf = synth.bf16_bits_to_f64(x)[0, 0]
    np.testing.assert_array_equal(d["pre_main"][0, 0], xf)  # p = 0: angle 0
    x, _, _ = _inputs(4, 1, 8, 1)
    _, _, d = _run(x, np.array([1000]), w, w_idx, 1, 1.6e5, "bf16")
    xf = synth.bf16_bits_to_f64(x)[0]
    n_in = xf[:, 0:64:2] ** 2 + xf[:, 1:64:2] ** 2
    n_out = d["pre_main"][0][:, 0:64:2] ** 2 + d["pre_main"][0][:, 1:64:2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13)


def test_stored_entries_are_the_encoded_pre_values():
    x, w, w_idx = _inputs(5, 2, 4, 2)
    for dtype in ("fp4", "bf16"):
        main, idx, d = _run(x, np.array([0, 2]), w, w_idx, 2, 1e4, dtype)
        pre = d["pre_main"]
        for b, base in ((0, 0), (1, 1)):
            if dtype == "fp4":
                c, s = oracle.fp4_encode(pre[b])
                np.testing.assert_array_equal(main.codes[b, base:base + 2], c)
                np.testing.assert_array_equal(main.scales[b, base:base + 2], s)
            else:
                want = [[oracle.bf16_round(v) for v in row] for row in pre[b]]
                np.testing.assert_array_equal(main.bf16[b, base:base + 2], want)
        assert (d["mag_main"] >= np.abs(d["pre_main"])).all()
        assert (d["mag_idx"] >= np.abs(d["pre_idx"])).all()


def test_indexer_k_is_projected_from_the_stored_entry():
    """W_idx selecting channels 0..127 (ones on a diagonal) makes the
    pre-encode indexer K equal the stored, decoded main entry's first 128
    channels exactly -- the projection reads the quantised entry, not the
    pre-quantisation values."""
    x, w, _ = _inputs(6, 1, 4, 2)
    sel = np.zeros((D, CI), np.uint16)
    sel[np.arange(CI), np.arange(CI)] = 0x3F80  # bf16 1.0
    for dtype in ("fp4", "bf16"):
        main, idx, d = _run(x, np.array([0]), w, sel, 2, 1e4, dtype)
        stored = main.values()[0, :2, :CI]
        np.testing.assert_array_equal(d["pre_idx"][0], stored)
        assert not np.array_equal(d["pre_idx"][0], d["pre_main"][0, :, :CI])


def test_argument_checks():
    x, w, w_idx = _inputs(7, 1, 3, 2)
    import pytest
    with pytest.raises(ValueError):
        _run(x, np.array([0]), w, w_idx, 2, 1e4, "fp4")  # T not a multiple of r
    x, w, w_idx = _inputs(7, 1, 4, 2)
    with pytest.raises(ValueError):
        _run(x, np.array([1]), w, w_idx, 2, 1e4, "fp4")  # pos0 not a multiple of r
