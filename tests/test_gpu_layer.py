"""The Full / Reindex / Reuse dispatcher (csa2_layer) over a small decoder
group, GPU against the oracle layer by layer: published top-k, HSI pool and
attention output."""
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

D, CI = 512, 128


def test_decoder_group_schedule_matches_oracle():
    B, N0, W, k, nb = 2, 2999, 128, 32, 64
    N = N0 + 1
    cap = 3072
    seed = 51
    # seeded random FP4 prefix, identical on both sides
    om, oi = oracle.Cache(B, cap, D, "fp4"), oracle.Cache(B, cap, CI, "fp4")
    g = synth.rng(seed, "prefix")
    for b in range(B):
        om.codes[b, :N0], om.scales[b, :N0] = synth.fp4_bytes(g, N0, D)
        oi.codes[b, :N0], oi.scales[b, :N0] = synth.fp4_bytes(g, N0, CI)
    pm, pi = _paged.cache_pair(B, cap, D, "fp4", seed), _paged.cache_pair(B, cap, CI, "fp4", seed + 1)
    _paged.upload(pm, om)
    _paged.upload(pi, oi)
    # this step's token (r = 1) compressed by the Full layer
    x = synth.normal_bf16(synth.rng(seed, "x"), (B, 1, D))
    w = synth.merge_weights(synth.rng(seed, "w"), 1, D)
    w_idx = synth.normal_bf16(synth.rng(seed, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    pos0 = np.full(B, N0, np.int64)
    oracle.compress(x, pos0, w, w_idx, om, oi, 1, 1.6e5)
    n_ent = np.full(B, N, np.int32)
    q_pos = np.full((B, 1), N0, np.int64)
    swa_len = np.full(B, W, np.int32)
    swa_pos0 = np.full(B, N0 - W + 1, np.int64)
    cfg = csa.Cfg(ratio=1, topk=k, hsi_blocks=nb, rope_theta=1.6e5)
    schedule = [(20, "full"), (21, "reuse"), (22, "reindex"), (23, "reuse"), (24, "reindex"), (25, "reuse")]
    modes = oracle.layer_modes(schedule)

    n_dev = torch.full((B,), N0, dtype=torch.int32, device="cuda")
    topk_d = torch.full((B, 1, k), -3, dtype=torch.int32, device="cuda")
    pool_d = torch.full((B, 1, nb), -3, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(csa.index_workspace_bytes(cfg, B, 1, cap), csa.index_workspace_bytes(cfg, B, 1, cap, True)),
                     dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = csa.GroupState(pm, pi, n_dev, cap, topk_d, pool_d, ws, st)

    o_topk = o_pool = None
    for layer, mode in schedule:
        ls = seed * 100 + layer
        q = synth.normal_bf16(synth.rng(ls, "q"), (B, 1, 64, D))
        q_idx = synth.normal_bf16(synth.rng(ls, "q_idx"), (B, 1, 32, CI))
        swa = synth.normal_bf16(synth.rng(ls, "swa"), (B, W, D))
        out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
        kw = {}
        if mode == "full":
            kw = dict(x=_paged.dev(x), pos0=_paged.dev(pos0), merge_w=_paged.dev(w), w_idx=_paged.dev(w_idx))
        m = {"full": csa.MODE_FULL, "reindex": csa.MODE_REINDEX, "reuse": csa.MODE_REUSE}[mode]
        topk_before, pool_before = topk_d.clone(), pool_d.clone()
        csa.layer(cfg, m, state, _paged.dev(q_pos), _paged.dev(q), _paged.dev(swa), _paged.dev(swa_len),
                  _paged.dev(swa_pos0), out, q_idx=_paged.dev(q_idx) if mode != "reuse" else None, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, csa.status_string(int(st.item()))
        if mode != "full":  # Reindex and Reuse never touch the pool; Reuse publishes nothing
            assert torch.equal(pool_d, pool_before), (layer, mode)
        if mode == "reuse":
            assert torch.equal(topk_d, topk_before), (layer, mode)
        # oracle, same schedule
        if mode == "full":
            o_topk, o_pool, s = oracle.index_topk(oi, n_ent, q_idx, q_pos, 1, k, hsi_blocks=nb, want_pool=True,
                                                  want_scores=True)
            assert P.topk_mismatch(topk_d.cpu().numpy().reshape(B, k), o_topk.reshape(B, k), s.reshape(B, -1), k,
                                   exact=False) == 0
            gp = pool_d.cpu().numpy()
            assert P.pool_mismatch(gp.reshape(B, nb), o_pool.reshape(B, nb), s.reshape(B, -1)) == 0
            assert all(((N - 1) // 8) in gp[b, 0] for b in range(B)), "latest block kept"
        elif mode == "reindex":
            o_topk, _, s = oracle.index_topk(oi, n_ent, q_idx, q_pos, 1, k, hsi_blocks=nb, pool=o_pool,
                                             want_scores=True)
            assert P.topk_mismatch(topk_d.cpu().numpy().reshape(B, k), o_topk.reshape(B, k), s.reshape(B, -1), k,
                                   exact=False) == 0
        else:
            assert modes[layer][1] == layer - 1
        # the oracle attends over its own published top-k (never the GPU's)
        o_out = oracle.attend(om, n_ent, q, o_topk, swa, swa_len, swa_pos0, q_pos, W, 1 / math.sqrt(D))
        err = P.attention_rel_err(out.cpu().numpy(), o_out)
        assert err <= P.ATT_TOL, (layer, mode, err)
    assert int(n_dev.cpu()[0]) == N


def test_encoder_macro_block_schedule_matches_oracle():
    """The encoder's CSA2 macro block: layer 2 Full (r = 2: the step's two
    tokens merged into one entry, indexing without HSI), layers 3-7 Reuse of
    layer 2's top-k, each with its own query and window rows."""
    B, E0, W, k = 3, 1500, 128, 64
    r = 2
    cap = 1600
    seed = 52
    om, oi = oracle.Cache(B, cap, D, "fp4"), oracle.Cache(B, cap, CI, "fp4")
    g = synth.rng(seed, "prefix")
    for b in range(B):
        om.codes[b, :E0], om.scales[b, :E0] = synth.fp4_bytes(g, E0, D)
        oi.codes[b, :E0], oi.scales[b, :E0] = synth.fp4_bytes(g, E0, CI)
    pm, pi = _paged.cache_pair(B, cap, D, "fp4", seed), _paged.cache_pair(B, cap, CI, "fp4", seed + 1)
    _paged.upload(pm, om)
    _paged.upload(pi, oi)
    x = synth.normal_bf16(synth.rng(seed, "x"), (B, r, D))
    w = synth.merge_weights(synth.rng(seed, "w"), r, D)
    w_idx = synth.normal_bf16(synth.rng(seed, "w_idx"), (D, CI), std=1 / math.sqrt(D))
    pos0 = np.full(B, r * E0, np.int64)            # tokens 3000, 3001 -> entry 1500
    oracle.compress(x, pos0, w, w_idx, om, oi, r, 1e4)
    N = E0 + 1
    n_ent = np.full(B, N, np.int32)
    t = r * E0 + r - 1                              # the query is the step's last token
    q_pos = np.full((B, 1), t, np.int64)
    swa_len = np.full(B, W, np.int32)
    swa_pos0 = np.full(B, t - W + 1, np.int64)
    cfg = csa.Cfg(ratio=r, topk=k, hsi_blocks=0, rope_theta=1e4)
    schedule = list(synth.ENCODER_GROUP)
    modes = oracle.layer_modes(schedule)

    n_dev = torch.full((B,), E0, dtype=torch.int32, device="cuda")
    topk_d = torch.full((B, 1, k), -3, dtype=torch.int32, device="cuda")
    ws = torch.empty(csa.index_workspace_bytes(cfg, B, 1, cap), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = csa.GroupState(pm, pi, n_dev, cap, topk_d, None, ws, st)
    o_topk = None
    for layer, mode in schedule:
        ls = seed * 100 + layer
        q = synth.normal_bf16(synth.rng(ls, "q"), (B, 1, 64, D))
        q_idx = synth.normal_bf16(synth.rng(ls, "q_idx"), (B, 1, 32, CI))
        swa = synth.normal_bf16(synth.rng(ls, "swa"), (B, W, D))
        out = torch.empty((B, 1, 64, D), dtype=torch.float32, device="cuda")
        kw = {}
        if mode == "full":
            kw = dict(x=_paged.dev(x), pos0=_paged.dev(pos0), merge_w=_paged.dev(w), w_idx=_paged.dev(w_idx))
        m = {"full": csa.MODE_FULL, "reuse": csa.MODE_REUSE}[mode]
        topk_before = topk_d.clone()
        csa.layer(cfg, m, state, _paged.dev(q_pos), _paged.dev(q), _paged.dev(swa), _paged.dev(swa_len),
                  _paged.dev(swa_pos0), out, q_idx=_paged.dev(q_idx) if mode != "reuse" else None, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, csa.status_string(int(st.item()))
        if mode == "reuse":  # the source layer's top-k, bit for bit
            assert torch.equal(topk_d, topk_before), (layer, mode)
        if mode == "full":
            o_topk, _, s = oracle.index_topk(oi, n_ent, q_idx, q_pos, r, k, want_scores=True)
            assert P.topk_mismatch(topk_d.cpu().numpy().reshape(B, k), o_topk.reshape(B, k), s.reshape(B, -1), k,
                                   exact=False) == 0
        else:
            assert modes[layer][1] == 2
        o_out = oracle.attend(om, n_ent, q, o_topk, swa, swa_len, swa_pos0, q_pos, W, 1 / math.sqrt(D))
        err = P.attention_rel_err(out.cpu().numpy(), o_out)
        assert err <= P.ATT_TOL, (layer, mode, err)
    assert int(n_dev.cpu()[0]) == N
