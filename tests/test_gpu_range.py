"""Inputs at and beyond the range of the tensor cores' f16 operands: the
largest finite bf16 magnitudes that f16 holds give the oracle's results,
and a magnitude beyond 65504 in the attention queries, the window rows or
the indexer queries over an FP4 cache is reported as CSA2_ERR_RANGE instead
of producing silent infinities."""
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
ERR_RANGE = 19
BIG_OK = oracle.bf16_round(65280.0)   # the largest bf16 below 65504 (it is exact in f16)
BIG = oracle.bf16_round(1.0e6)


def _attend_case(seed, B=2, N=900, k=512, W=128):
    oc = oracle.Cache(B, N, D, "fp4")
    g = synth.rng(seed, "main")
    for b in range(B):
        oc.codes[b], oc.scales[b] = synth.fp4_bytes(g, N, D)
    pc = _paged.cache_pair(B, N, D, "fp4", seed)
    _paged.upload(pc, oc)
    topk = np.stack([np.sort(synth.rng(seed, "ids%d" % b).choice(N, size=k, replace=False)) for b in range(B)])
    topk = topk.reshape(B, 1, k).astype(np.int32)
    q = synth.normal_bf16(synth.rng(seed, "q"), (B, 1, HM, D))
    swa = synth.normal_bf16(synth.rng(seed, "swa"), (B, W, D))
    q_pos = np.full((B, 1), 2 * N - 1, np.int64)
    swa_len = np.full(B, W, np.int32)
    swa_pos0 = np.full(B, 2 * N - W, np.int64)
    return oc, pc, topk, q, swa, q_pos, swa_len, swa_pos0


def _run_attend(pc, topk, q, swa, q_pos, swa_len, swa_pos0, k=512, W=128):
    B = q.shape[0]
    cfg = csa.Cfg(ratio=2, topk=k, window=W)
    out = torch.empty((B, 1, HM, D), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.attend(cfg, _paged.dev(q), pc, _paged.dev(np.full(B, 900, np.int32)), _paged.dev(topk),
               _paged.dev(swa), _paged.dev(swa_len), _paged.dev(swa_pos0), _paged.dev(q_pos), out, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def test_attention_at_the_largest_f16_magnitude_matches_the_oracle():
    oc, pc, topk, q, swa, q_pos, swa_len, swa_pos0 = _attend_case(41)
    q = q.copy()
    q[0, 0, 3, 7] = BIG_OK                        # a query channel at 65280
    q[1, 0, 60, 100] = BIG_OK | 0x8000
    swa = swa.copy()
    swa[1, 5, 9] = BIG_OK                         # a window value at 65280
    out, st = _run_attend(pc, topk, q, swa, q_pos, swa_len, swa_pos0)
    assert st == 0
    ref = oracle.attend(oc, np.full(2, 900, np.int32), q, topk, swa, swa_len, swa_pos0, q_pos, 128,
                        1 / math.sqrt(D))
    assert P.attention_rel_err(out, ref) <= P.ATT_TOL


@pytest.mark.parametrize("where", ["q", "swa"])
def test_attention_beyond_the_f16_range_is_reported(where):
    oc, pc, topk, q, swa, q_pos, swa_len, swa_pos0 = _attend_case(42)
    q, swa = q.copy(), swa.copy()
    if where == "q":
        q[1, 0, 10, 200] = BIG
    else:
        swa[0, 127, 33] = BIG | 0x8000
    _, st = _run_attend(pc, topk, q, swa, q_pos, swa_len, swa_pos0)
    assert st == ERR_RANGE


def test_indexer_query_beyond_the_f16_range_is_reported():
    B, N, k = 2, 3000, 64
    oc = oracle.Cache(B, N, CI, "fp4")
    g = synth.rng(43, "idx")
    for b in range(B):
        oc.codes[b], oc.scales[b] = synth.fp4_bytes(g, N, CI)
    pc = _paged.cache_pair(B, N, CI, "fp4", 43)
    _paged.upload(pc, oc)
    q_idx = synth.normal_bf16(synth.rng(43, "q"), (B, 1, H, CI))
    q_pos = np.full((B, 1), N - 1, np.int64)
    n_ent = np.full(B, N, np.int32)
    cfg = csa.Cfg(ratio=1, topk=k)
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, N), dtype=torch.uint8, device="cuda")
    for big, want in ((BIG_OK, 0), (BIG, ERR_RANGE)):
        qi = q_idx.copy()
        qi[1, 0, 5, 17] = big
        topk = torch.empty((B, 1, k), dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        csa.index_topk(cfg, _paged.dev(qi), _paged.dev(q_pos), pc, _paged.dev(n_ent), N, topk, ws, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == want
        if want == 0:
            o_top, _, s = oracle.index_topk(oc, n_ent, qi, q_pos, r=1, k=k, want_scores=True)
            assert P.topk_mismatch(topk.cpu().numpy().reshape(B, k), o_top.reshape(B, k), s.reshape(B, -1), k,
                                   exact=False) == 0
