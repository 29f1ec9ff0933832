"""Pins of the oracle's indexer, top-k, HSI pool and Reindex: brute-force
selection on tiny inputs, reduced special cases of the score, visibility and
the HSI containment properties."""
import numpy as np
import pytest

import oracle
import synth

CI, H = 128, 32


def _cache(seed, B, n_cap, dtype="fp4", integer=False):
    c = oracle.Cache(B, n_cap, CI, dtype)
    g = synth.rng(seed, "idx_cache")
    if dtype == "fp4":
        for b in range(B):
            if integer:
                c.codes[b], c.scales[b] = synth.integer_fp4_bytes(g, n_cap, CI)
            else:
                c.codes[b], c.scales[b] = synth.fp4_bytes(g, n_cap, CI)
    else:
        c.bf16[:] = synth.normal_bf16(g, (B, n_cap, CI))
    return c


def _brute_topk(scores, cand, k):
    ids = [j for j in range(len(scores)) if cand[j]]
    ids.sort(key=lambda j: (-scores[j], j))
    sel = sorted(ids[:k])
    return sel + [-1] * (k - len(sel))


def test_topk_brute_force_integer_mode_with_ties():
    """Integer q (-3..3) and integer-valued FP4 K: scores are exact integers
    with many ties, so the lowest-index tie rule is exercised."""
    B, N, k = 2, 61, 16
    cache = _cache(1, B, N, integer=True)
    # repeat a few distinct entries so that equal scores straddle the k-th place
    pick = synth.rng(1, "dup").integers(0, 7, size=(B, N))
    for b in range(B):
        cache.codes[b] = cache.codes[b][pick[b]]
        cache.scales[b] = cache.scales[b][pick[b]]
    q = synth.integer_bf16(synth.rng(1, "q_idx"), (B, 3, H, CI))
    q_pos = np.array([[60, 30, 5], [60, 59, 0]], np.int64)
    n_ent = np.array([N, 50], np.int32)
    topk, _, s = oracle.index_topk(cache, n_ent, q, q_pos, r=1, k=k, want_scores=True)
    assert np.all(np.isfinite(s[s > -np.inf]))
    fin = s[np.isfinite(s)]
    assert np.array_equal(fin, np.round(fin)), "integer inputs give integer scores"
    n_ties = 0
    for b in range(B):
        for t in range(3):
            nv = min(q_pos[b, t] + 1, n_ent[b])
            cand = [j < nv for j in range(N)]
            assert topk[b, t].tolist() == _brute_topk(s[b, t], cand, k)
            vals = sorted(s[b, t, :nv], reverse=True)
            n_ties += len(vals) > k and vals[k - 1] == vals[k]
    assert n_ties > 0, "the case must contain ties across the k-th place"


def test_visibility_counts():
    """Entry j covers positions 2j, 2j+1 and is visible from t = 2j + 1 on."""
    N = 40
    cache = _cache(2, 1, N)
    q = synth.normal_bf16(synth.rng(2, "q_idx"), (1, 5, H, CI))
    q_pos = np.array([[0, 1, 6, 7, 79]], np.int64)
    topk, _, s = oracle.index_topk(cache, np.array([N], np.int32), q, q_pos, r=2, k=64, want_scores=True)
    want_nv = [0, 1, 3, 4, 40]
    for t, nv in enumerate(want_nv):
        assert (topk[0, t] >= 0).sum() == nv
        assert topk[0, t][:nv].tolist() == list(range(nv))
        assert np.isfinite(s[0, t, :nv]).all() and np.isneginf(s[0, t, nv:]).all()


def test_score_special_cases():
    """One-hot indexer entries reduce the score to sum_h w_h ReLU(q_h[c]) * v;
    a negated query zeroes every head whose dot was positive; weights scale
    linearly; a single non-zero head weight gives a single ReLU'd dot."""
    N = 8
    cache = oracle.Cache(1, N, CI, "bf16")
    chans = [0, 5, 64, 127, 3, 9, 100, 42]
    vals = [1.0, 2.0, 0.5, 4.0, 1.0, 1.0, 1.0, 1.0]
    for j, (c, v) in enumerate(zip(chans, vals)):
        cache.bf16[0, j, c] = oracle.bf16_round(v)
    q = synth.integer_bf16(synth.rng(3, "q"), (1, 1, H, CI), -3, 3)
    qf = synth.bf16_bits_to_f64(q)[0, 0]
    hw = synth.rng(3, "w").uniform(0.5, 2.0, size=(1, 1, H)).astype(np.float32)
    _, _, s = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                head_w=hw, want_scores=True)
    for j, (c, v) in enumerate(zip(chans, vals)):
        want = sum(float(hw[0, 0, h]) * max(qf[h, c], 0.0) * v for h in range(H))
        assert s[0, 0, j] == pytest.approx(want, rel=1e-15, abs=0)
    hw1 = np.zeros_like(hw)
    hw1[0, 0, 7] = 1.0
    _, _, s1 = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                 head_w=hw1, want_scores=True)
    for j, (c, v) in enumerate(zip(chans, vals)):
        assert s1[0, 0, j] == max(qf[7, c] * v, 0.0)
    qn = (q ^ np.uint16(0x8000)).astype(np.uint16)  # negate every query element
    _, _, s0 = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                 want_scores=True)
    _, _, sn = oracle.index_topk(cache, np.array([N], np.int32), qn, np.array([[N - 1]]), r=1, k=4,
                                 want_scores=True)
    for j, (c, v) in enumerate(zip(chans, vals)):
        assert s0[0, 0, j] + sn[0, 0, j] == pytest.approx(sum(abs(qf[h, c]) * v for h in range(H)))
    _, _, s2 = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                 head_w=2 * hw, want_scores=True)
    _, _, sh = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                 head_w=hw, want_scores=True)
    np.testing.assert_array_equal(s2, 2 * sh)


def _hsi_case(seed, N, k, nb, bs, integer=False):
    cache = _cache(seed, 1, N, integer=integer)
    g = synth.rng(seed, "q_idx")
    q = synth.integer_bf16(g, (1, 2, H, CI)) if integer else synth.normal_bf16(g, (1, 2, H, CI))
    q_pos = np.array([[N - 1, N - 6]], np.int64)
    return cache, q, q_pos


@pytest.mark.parametrize("integer", [False, True])
def test_hsi_pool_brute_force_and_containment(integer):
    # containment of the Full top-k in the pool needs nb - 1 >= k (2047 >= 512)
    N, k, nb, bs = 203, 5, 6, 8
    cache, q, q_pos = _hsi_case(4, N, k, nb, bs, integer)
    n_ent = np.array([N], np.int32)
    topk, pool, s = oracle.index_topk(cache, n_ent, q, q_pos, r=1, k=k, hsi_blocks=nb, hsi_block=bs,
                                      want_pool=True, want_scores=True)
    for t in range(2):
        nv = q_pos[0, t] + 1
        nblk = (nv + bs - 1) // bs
        forced = (nv - 1) // bs
        bmax = [max(s[0, t, b * bs:min((b + 1) * bs, nv)]) for b in range(nblk)]
        others = sorted((b for b in range(nblk) if b != forced), key=lambda b: (-bmax[b], b))
        want = sorted([forced] + others[:nb - 1])
        assert pool[0, t].tolist() == want + [-1] * (nb - len(want))
        ent = {j for b in want for j in range(b * bs, (b + 1) * bs)}
        assert set(topk[0, t][topk[0, t] >= 0].tolist()) <= ent, "Full top-k lies inside the pool"
        assert forced in pool[0, t]


def test_hsi_forced_block_is_kept_when_it_scores_lowest():
    """Make the block holding the latest visible entry score lowest: it must
    still be in the pool, displacing the lowest-ranked other block."""
    N, nb, bs = 64, 3, 8
    cache = oracle.Cache(1, N, CI, "bf16")
    cache.bf16[0, :, 0] = oracle.bf16_round(1.0)
    for j in range(N):
        cache.bf16[0, j, 0] = oracle.bf16_round(float(N - j))  # earlier entries score higher
    q = np.zeros((1, 1, H, CI), np.uint16)
    q[..., 0] = oracle.bf16_round(1.0)
    _, pool, _ = oracle.index_topk(cache, np.array([N], np.int32), q, np.array([[N - 1]]), r=1, k=4,
                                   hsi_blocks=nb, hsi_block=bs, want_pool=True)
    assert pool[0, 0].tolist() == [0, 1, 7]


def test_reindex_over_all_blocks_equals_full_and_pool_restricts():
    N, k, bs = 150, 10, 8
    cache = _cache(5, 1, N)
    q = synth.normal_bf16(synth.rng(5, "q_idx"), (1, 1, H, CI))
    q_pos = np.array([[N - 1]], np.int64)
    n_ent = np.array([N], np.int32)
    full, _, s = oracle.index_topk(cache, n_ent, q, q_pos, r=1, k=k, want_scores=True)
    nblk = (N + bs - 1) // bs
    all_blocks = np.arange(nblk, dtype=np.int32).reshape(1, 1, -1)
    re_all, _, _ = oracle.index_topk(cache, n_ent, q, q_pos, r=1, k=k, hsi_blocks=nblk, hsi_block=bs,
                                     pool=all_blocks)
    np.testing.assert_array_equal(re_all, full)
    pool = np.array([[[2, 5, 11, 18, -1, -1]]], np.int32)
    q2 = synth.normal_bf16(synth.rng(6, "q_idx"), (1, 1, H, CI))
    re, _, s2 = oracle.index_topk(cache, n_ent, q2, q_pos, r=1, k=k, hsi_blocks=6, hsi_block=bs,
                                  pool=pool, want_scores=True)
    cand = [False] * N
    for b in (2, 5, 11, 18):
        for j in range(b * bs, min((b + 1) * bs, N)):
            cand[j] = True
    assert re[0, 0].tolist() == _brute_topk(s2[0, 0], cand, k)
    assert np.isneginf(s2[0, 0][~np.array(cand)]).all()


def test_short_context_pads_with_minus_one():
    cache = _cache(7, 1, 10)
    q = synth.normal_bf16(synth.rng(7, "q_idx"), (1, 1, H, CI))
    topk, pool, _ = oracle.index_topk(cache, np.array([3], np.int32), q, np.array([[100]]), r=1, k=5,
                                      hsi_blocks=4, hsi_block=8, want_pool=True)
    assert topk[0, 0].tolist() == [0, 1, 2, -1, -1]
    assert pool[0, 0].tolist() == [0, -1, -1, -1]
