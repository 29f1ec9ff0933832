"""Comparison rules shared by the GPU parity tests (test code only).

- FP4 / bf16 dequantisation: bit-exact.
- Encoded codes from the compressor: bit-exact, except where the oracle's
  pre-encoding value lies within the rounding-error bound of an fp32
  evaluation of a decision boundary.  The bound is margin * M, with M the sum
  of |terms| that formed the value (returned by the oracle): 2^-19 M for the
  merged / rotated entry (at most ~10 fp32 roundings of terms of size M),
  2^-14 M for indexer K (a 512-term fp32 sum).  Excused positions are counted
  and reported; an entry whose stored main codes differ excuses its indexer K.
- Top-k: bit-exact on integer-valued inputs (exact scores); otherwise set
  equality up to near-ties: every id in the symmetric difference must have an
  oracle score within 1e-5 relative of the oracle's k-th score.
- Attention: per (token, head) row, max|o - o*| / max|o*| <= 2e-2.
"""
import numpy as np

import oracle

MAIN_MARGIN = 2.0 ** -19
IDX_MARGIN = 2.0 ** -14
NEAR_TIE = 1e-5
ATT_TOL = 2e-2

_E4 = np.array([oracle.e4m3_value(c) for c in range(127)])
_E4_ALL = np.array([oracle.e4m3_value(c) for c in range(256)])  # byte -> value (NaN for 0x7F / 0xFF)
_SCALE_T = 3.0 * (_E4[:-1] + _E4[1:])  # 6 * midpoints, increasing
_E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def fp4_code_mismatches(gpu_codes, gpu_scales, ora_codes, ora_scales, pre, mag, margin):
    """Returns (n_unexcused, n_excused, bad_entry_mask [..., entries]); the scale
    group (16 or 32 channels) follows from the shape of the scales."""
    C = pre.shape[-1]
    G = ora_scales.shape[-1]
    gs = C // G
    lead = pre.shape[:-1]
    pre_g = pre.reshape(lead + (G, gs))
    mag_g = mag.reshape(lead + (G, gs))
    amax = np.abs(pre_g).max(-1)
    tol_a = margin * mag_g.max(-1)
    near_scale = (np.abs(amax[..., None] - _SCALE_T) <= tol_a[..., None]).any(-1)

    def nib(codes):
        lo, hi = codes & 15, codes >> 4
        return np.stack([lo, hi], -1).reshape(lead + (C,))

    gc, oc = nib(gpu_codes), nib(ora_codes)
    s = _E4_ALL[ora_scales.astype(np.int64)]
    s_el = np.repeat(s, gs, axis=-1)
    near_code = (np.abs(np.abs(pre)[..., None] - s_el[..., None] * _E2M1_MID) <= (margin * mag)[..., None]).any(-1)
    near_code |= np.repeat(near_scale, gs, axis=-1)
    scale_bad = gpu_scales != ora_scales
    code_bad = gc != oc
    unexcused = int((scale_bad & ~near_scale).sum() + (code_bad & ~near_code).sum())
    excused = int((scale_bad & near_scale).sum() + (code_bad & near_code).sum())
    bad_entry = scale_bad.any(-1) | code_bad.any(-1)
    return unexcused, excused, bad_entry


def _bf16_neighbour(bits, up: bool):
    """Value of the bf16 next to `bits` toward +inf (up) or -inf.  Between the
    two zeros the gap is 0: a value of one sign never rounds to the other
    sign's zero."""
    b = bits.astype(np.int64)
    key = np.where(b & 0x8000, 0x7FFF - (b & 0x7FFF), b + 0x8000)   # monotone in the value
    nk = key + 1 if up else key - 1
    nb = np.where(nk >= 0x8000, nk - 0x8000, 0x8000 | (0x7FFF - nk)).astype(np.uint32)
    return (nb << 16).view(np.float32).astype(np.float64)


def bf16_mismatches(gpu_vals, ora_vals, pre, mag, margin):
    """A bf16 code g that differs from the oracle's is excused only when g is
    the round-to-nearest of some value within the fp32 evaluation bound of
    the oracle's pre-rounding value: g's rounding interval (half the gap to
    its neighbour on the side of `pre`, so at a binade edge the smaller
    binade's half-gap below a power of two) must reach to within
    margin * M of pre.  Equivalently the rounding midpoint between g and
    the next bf16 toward pre lies within margin * M of pre."""
    g = (gpu_vals.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    diff = gpu_vals != ora_vals
    above = pre > g
    nb = np.where(above, _bf16_neighbour(gpu_vals, True), _bf16_neighbour(gpu_vals, False))
    half_gap = np.abs(nb - g) / 2.0
    near = np.abs(g - pre) <= margin * mag + half_gap
    unexcused = int((diff & ~near).sum())
    excused = int((diff & near).sum())
    return unexcused, excused, diff.any(-1)


def topk_mismatch(gpu_ids, ora_ids, ora_scores, k, exact: bool):
    """Number of query rows whose top-k differs beyond the rules above."""
    bad = 0
    for qi in range(gpu_ids.shape[0]):
        g, o = gpu_ids[qi], ora_ids[qi]
        if exact:
            bad += not np.array_equal(g, o)
            continue
        gs, os_ = set(g[g >= 0].tolist()), set(o[o >= 0].tolist())
        if len(gs) != len(os_) or (g >= 0).sum() != len(gs):
            bad += 1
            continue
        diff = gs ^ os_
        if not diff:
            continue
        s = ora_scores[qi]
        kth = np.sort(s[np.isfinite(s)])[::-1][min(k, np.isfinite(s).sum()) - 1]
        ok = all(abs(s[j] - kth) <= NEAR_TIE * abs(kth) for j in diff)
        bad += not ok
    return bad


def pool_mismatch(gpu_pool, ora_pool, ora_scores, block=8):
    """Number of query rows whose HSI pool differs beyond near-ties.  Pools
    are ascending block ids, -1 padded.  Block score = max of the oracle's
    scores over the block's visible positions (non-finite = not visible).
    Both pools must hold the same number of blocks and the oracle's forced
    block (its latest visible block); every block in the symmetric
    difference must score within 1e-5 relative of the lowest-scoring
    non-forced block of the oracle's pool."""
    bad = 0
    for qi in range(gpu_pool.shape[0]):
        g, o = gpu_pool[qi], ora_pool[qi]
        gs, os_ = set(g[g >= 0].tolist()), set(o[o >= 0].tolist())
        if len(gs) != len(os_) or (g >= 0).sum() != len(gs) or not np.all(np.diff(g[g >= 0]) > 0):
            bad += 1
            continue
        s = ora_scores[qi]
        vis = np.nonzero(np.isfinite(s))[0]
        if len(vis) == 0:
            bad += len(gs) != 0
            continue
        forced = int(vis.max()) // block
        if forced not in gs:
            bad += 1
            continue
        diff = gs ^ os_
        if not diff:
            continue
        nb = (len(s) + block - 1) // block
        sp = np.full(nb * block, -np.inf)
        sp[:len(s)] = np.where(np.isfinite(s), s, -np.inf)
        bs = sp.reshape(nb, block).max(-1)
        rest = [bs[j] for j in os_ if j != forced]
        kth = min(rest) if rest else -np.inf
        ok = all(j != forced and abs(bs[j] - kth) <= NEAR_TIE * abs(kth) for j in diff)
        bad += not ok
    return bad


def attention_rel_err(out, ref):
    """max over (token, head) rows of max|o - o*| / max|o*|."""
    o = out.reshape(-1, out.shape[-1]).astype(np.float64)
    r = ref.reshape(-1, ref.shape[-1])
    num = np.abs(o - r).max(-1)
    den = np.abs(r).max(-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())
