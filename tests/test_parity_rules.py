"""The comparison rules of the GPU parity tests, checked on planted
mistakes (CPU only): a rule that excused these would let a wrong kernel
pass."""
import numpy as np

from tests import _parity as P


def _bits(x):
    return (np.float32(x).view(np.uint32) >> 16).astype(np.uint16)


def test_bf16_rule_excuses_only_a_rounding_flip_within_the_bound():
    one, below = _bits(1.0), np.uint16(0x3F7F)        # 1.0 and the bf16 just below it
    mid = (1.0 + 0.99609375) / 2
    M, margin = np.array([1.0]), 2.0 ** -30
    g, o = np.array([one]), np.array([below])
    # the oracle's value sits just below the midpoint: a GPU 1.0 is a legal rounding flip
    assert P.bf16_mismatches(g, o, np.array([mid - margin / 2]), M, margin)[:2] == (0, 1)
    # further below than the evaluation bound: not excused
    assert P.bf16_mismatches(g, o, np.array([mid - 4 * margin]), M, margin)[:2] == (1, 0)
    # two codes away, even at the midpoint: not excused
    assert P.bf16_mismatches(np.array([np.uint16(0x3F81)]), o, np.array([mid]), M, margin)[:2] == (1, 0)
    # at a binade edge the half-gap below 1.0 is the smaller binade's
    assert P.bf16_mismatches(g, o, np.array([1.0 - 0.00390625 / 2 - 0.0001]), M, margin)[:2] == (1, 0)
    # a sign flip near zero is excused only within the bound
    tiny = np.array([_bits(1e-30)])
    assert P.bf16_mismatches(np.array([_bits(-1e-30)]), tiny, np.array([0.0]), np.array([1e-29]), 1.0)[:2] == (0, 1)
    assert P.bf16_mismatches(np.array([_bits(-1e-30)]), tiny, np.array([1e-30]), np.array([1e-31]), 1.0)[:2] == (1, 0)


def test_pool_rule_flags_a_wrong_block_and_a_missing_forced_block():
    n, nb, block = 200, 4, 8
    s = np.arange(n, dtype=np.float64)[None, :].copy()       # block b scores 8b + 7
    s[0, 10] = 1000.0                                        # block 1 is the best
    forced = (n - 1) // block                                # block 24
    ora = np.array([[1, 22, 23, forced]], np.int32)
    assert P.pool_mismatch(ora.copy(), ora, s) == 0
    assert P.pool_mismatch(np.array([[1, 21, 23, forced]], np.int32), ora, s) == 1   # block 21 is not a near-tie
    assert P.pool_mismatch(np.array([[1, 21, 22, 23]], np.int32), ora, s) == 1       # forced block missing
    assert P.pool_mismatch(np.array([[1, 22, forced, -1]], np.int32), ora, s) == 1   # a block short
    assert P.pool_mismatch(np.array([[22, 1, 23, forced]], np.int32), ora, s) == 1   # not ascending
    # a genuine near-tie at the lowest pooled block is accepted
    s2 = s.copy()
    s2[0, 21 * block + 7] = s2[0, 22 * block + 7] * (1 + 1e-7)
    assert P.pool_mismatch(np.array([[1, 21, 23, forced]], np.int32), ora, s2) == 0


def test_topk_rule_flags_a_non_tie_swap():
    s = np.arange(100, dtype=np.float64)[None, :]
    ora = np.array([[96, 97, 98, 99]], np.int32)
    assert P.topk_mismatch(ora.copy(), ora, s, 4, exact=False) == 0
    assert P.topk_mismatch(np.array([[90, 97, 98, 99]], np.int32), ora, s, 4, exact=False) == 1
    assert P.topk_mismatch(np.array([[96, 97, 99, 98]], np.int32), ora, s, 4, exact=True) == 1
