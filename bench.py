"""CSA2 benchmark: query-tokens/s of one CSA2 step on synthetic inputs.

A step is one pass of the whole path over one batch: the compressor on the
step's new tokens, the indexer with top-k (and the HSI pool / Reindex on
decoder workloads), and sparse attention over top-k plus the window.  The
default workload is the decoder-layer decode step: batch 32, 131072 tokens of
context at ratio 1 in an FP4 cache, the hierarchical indexer (HSI, 2048
blocks of 8) and top-512 plus the 128-row window.

Timing: W warm-up steps launched eagerly; then the step is captured once as a
CUDA graph and K replays are timed, each bracketed by CUDA events on the
launching stream.  Before every step a 256 MiB buffer is written so that the
step starts with a cold L2 (the inputs are smaller than L2).  The per-stage
durations used for the roofline come from one graph per stage replayed back
to back after the same flush; the eager launch of the step through the Python
API is timed too (eager_ms_per_step), and the end-to-end leg runs eagerly
with the inputs copied from pinned host memory and the output copied back.
Under torchrun every rank runs its own batch (weak scaling, no data-path
collective); rank 0 prints one JSON line with the max over ranks.

On one GPU with the default workload the same run also measures the two
other workloads with a stated target -- the 20-layer decoder group (per
group time) and the 4096-token prefill chunk (indexer against the tensor
peak) -- and reports them under "targets".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--batch B] [--tq T] [--impl reference]
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "CSA2 sparse-attention query-tokens/s at 1 GB300; achieved HBM GB/s vs peak"
UNIT = "query-tokens/s"
DEFAULT_WORKLOAD = "decode_b32_ctx131072_r1_fp4_hsi"
# workloads with a stated target, measured beside the default one: the
# decoder group's time per group and the prefill indexer's tensor fraction
TARGETS = {"decoder_group20_b16_ctx262144_fp4": {"ms_per_step": 0.111},
           "prefill_4096_on_1m_r2_fp4": {"roofline_frac": 0.50}}
FLUSH_BYTES = 256 << 20
_FLUSH_READ = {}


def flush_l2(flush, k):
    """Evict L2 before a timed step: write `flush`, a buffer larger than L2,
    so nothing of the step stays resident, then read a second buffer of the
    same size, so that the lines just written go back to HBM here, outside
    the timed region, instead of during the step's first loads (the step
    starts with a cold L2 holding no dirty lines, as ncu's own cache control
    leaves it)."""
    import torch
    flush.fill_(k & 0xFF)
    rd = _FLUSH_READ.get(flush.device)
    if rd is None:
        rd = _FLUSH_READ[flush.device] = torch.zeros(flush.numel() // 8, dtype=torch.int64, device=flush.device)
    torch.amax(rd)


# algorithmic bytes per unit (hot-path scope table): indexer 72 B per visible
# FP4 entry per query (256 B per bf16 entry); attention 512 x 288 + 128 x 1024
# + Q 65536 + fp32 out 131072 + ids 2048 B per query token; compressor
# r x 1024 B in + 360 B out per entry.
IDX_ENTRY_BYTES = {"fp4": 72, "bf16": 256}
MAIN_ENTRY_BYTES = {"fp4": 288, "bf16": 1024}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# stage's kernels, from one ncu capture of this bench's default command; the
# summaries under profiles/ name the capture.  A stage with no capture of the
# current kernels reports null.
TRAFFIC = {
    "decode_b32_ctx131072_r1_fp4_hsi": {
        "index_score": (302600704 + 17805056, "profiles/score_tc_kernel_decode_b32_ctx131072_r1_fp4_hsi.md"),
        "index_select": (9095936, "profiles/select_kernel_decode_b32_ctx131072_r1_fp4_hsi.md"),
        "attend": (12979456, "profiles/attend_qc_kernel_decode_b32_ctx131072_r1_fp4_hsi.md"),
    },
}


def attend_kernel(topk, window):
    """The decode attention kernel the library launches for this many row
    tiles of 128 (a query cluster of 4-5 CTAs, else one CTA per tile)."""
    tiles = (topk + 127) // 128 + (window + 127) // 128
    return "attend_qc_kernel" if tiles in (4, 5) else "attend_rows_kernel" if tiles <= 6 else "attend_split_kernel"


def attend_query_bytes(cache, topk=512, window=128, row_bytes=1024):
    """Top-k entries + window rows (bf16 1024 B, MXFP8 528 B) + bf16 Q + fp32 out + ids."""
    return topk * MAIN_ENTRY_BYTES[cache] + window * row_bytes + 64 * 512 * 2 + 64 * 512 * 4 + topk * 4


def select_bytes(n_entries: int, wl) -> int:
    """Workspace bytes one query's selection reads and writes: its fp32
    scores (and HSI block maxima), the top-k (and pool) ids."""
    hsi = wl.hsi and not wl.layers
    return 4 * n_entries + (4 * (-(-n_entries // 8)) + 4 * wl.hsi_blocks if hsi else 0) + 4 * wl.topk


def index_chunk(per_query_bytes: int, queries: int, budget: int = 16 << 30) -> int:
    """Queries per indexer pass: all of them when their workspace fits the
    budget (one score and one selection launch), else as many as fit."""
    return max(1, min(queries, budget // max(per_query_bytes, 1)))


def idx_entry_bytes(wl):
    return 68 if wl.idx68 else IDX_ENTRY_BYTES[wl.cache]


def swa_row_bytes(wl):
    return 528 if wl.swa_fp8 else 1024


def peaks():
    """(HBM GB/s, sustained bf16 TFLOP/s, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            self.path = os.path.join("/tmp", "csa2_clocks_%d_%d.csv" % (os.getpid(), self.index))
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- workload ----

def _dev(a, device):
    import torch
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)


def _fill_cache(c, cd, g, device):
    """Seeded random cache contents: uniform FP4 codes with E4M3 scales in
    0x20..0x3C, or N(0,1) bf16 values (same distribution as the tests)."""
    import torch
    import compressed_sparse_attention_07_gb300 as csa
    if cd != csa.CACHE_BF16:
        c.data.random_(0, 256, generator=g)
        c.scales.random_(0x20, 0x3D, generator=g)
    else:
        v = torch.randn(c.data.numel() // 2, generator=g, device=device, dtype=torch.float32)
        c.data.view(torch.int16).copy_(v.to(torch.bfloat16).view(torch.int16).view(c.data.shape[0], -1))


class StepBase:
    """Common pieces: config, caches with a seeded random prefix, step inputs
    on the device and as host arrays (for the end-to-end leg)."""

    def __init__(self, wl: synth.Workload, device, seed_offset=0):
        import torch
        import compressed_sparse_attention_07_gb300 as csa
        self.torch, self.csa, self.wl, self.device = torch, csa, wl, device
        self.cd = csa.CACHE_FP4 if wl.cache == "fp4" else csa.CACHE_BF16
        fmt = ((csa.FMT_IDX_68B if wl.idx68 else 0) | (csa.FMT_SWA_FP8 if wl.swa_fp8 else 0) |
               (csa.FMT_IDX_QFP4 if wl.q_fp4 else 0))
        self.cfg = csa.Cfg(ratio=wl.ratio, cache_dtype=self.cd, topk=wl.topk, window=wl.window,
                           hsi_blocks=wl.hsi_blocks if wl.hsi else 0, rope_theta=wl.theta, formats=fmt)
        self.seed = wl.seed + seed_offset
        self.B = wl.batch
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def make_caches(self, capacity):
        g = self.torch.Generator(device=self.device)
        g.manual_seed(self.seed)
        self.main = self.csa.PagedCache(self.B, capacity, 512, self.cd, device=self.device)
        self.idx = self.csa.PagedCache(self.B, capacity, 128, self.cfg.idx_dtype, device=self.device)
        for c in (self.main, self.idx):
            _fill_cache(c, c.cache_dtype, g, self.device)

    def upload(self):
        self.d = {k: _dev(v, self.device) for k, v in self.h.items()}

    def inputs_host(self):
        return self.h

    def late_inputs(self):
        """(index of the first call that reads them, input names): inputs the
        first calls of a step do not read, so their upload can overlap them."""
        calls = len(self.stages)
        return calls - 1, {k for k in ("q", "swa", "swa_len", "swa_pos0") if k in self.h}

    def step(self, events=None, d=None):
        """Run the stages in order, recording events[i] before stage i and
        events[-1] after the last."""
        calls = self.calls(d or self.d)
        ev = events or [None] * (len(calls) + 1)
        if ev[0] is not None:
            ev[0].record()
        for i, c in enumerate(calls):
            c()
            if ev[i + 1] is not None:
                ev[i + 1].record()
        return self.out


class DecodeStep(StepBase):
    """One decode step of one CSA2 layer in Full mode: compress the step's r
    new tokens per sequence (one entry), index the whole visible cache (plus
    the HSI pool on the decoder Full layer), attend over top-k and window.
    With FP8 window rows the step also encodes its newest window row into
    the resident MXFP8 window (the older rows were encoded by earlier steps)."""

    def __init__(self, wl, device, seed_offset=0):
        super().__init__(wl, device, seed_offset)
        torch, csa, B, r, s = self.torch, self.csa, self.B, wl.ratio, self.seed
        self.N = wl.ctx // r
        self.make_caches(self.N)
        ctx = wl.ctx
        self.h = {
            "x": synth.normal_bf16(synth.rng(s, "x_step"), (B, r, 512)),
            "pos0": np.full(B, ctx - r, np.int64),
            "q": synth.normal_bf16(synth.rng(s, "q"), (B, 1, 64, 512)),
            "q_idx": synth.normal_bf16(synth.rng(s, "q_idx"), (B, 1, 32, 128)),
            "swa": synth.normal_bf16(synth.rng(s, "swa"), (B, wl.window, 512)),
            "swa_len": np.full(B, wl.window, np.int32),
            "swa_pos0": np.full(B, ctx - wl.window, np.int64),
            "q_pos": np.full((B, 1), ctx - 1, np.int64),
        }
        if wl.swa_fp8:
            # resident MXFP8 window: rows ctx-W .. ctx-2 encoded once here; the
            # step's input is the newest bf16 row, encoded into row W-1
            older = self.h.pop("swa")
            self.h["swa_new"] = np.ascontiguousarray(older[:, -1:])
            self.swa8 = torch.zeros((B, wl.window, csa.SWA_FP8_ROW), dtype=torch.uint8, device=device)
            csa.swa_encode(_dev(older[:, :-1], device), torch.zeros(B, dtype=torch.int64, device=device), self.swa8,
                           status=self.status)
            self.swa_row0 = torch.full((B,), wl.window - 1, dtype=torch.int64, device=device)
        self.upload()
        self.merge_w = _dev(synth.merge_weights(synth.rng(s, "w"), r, 512), device)
        self.w_idx = _dev(synth.normal_bf16(synth.rng(s, "w_idx"), (512, 128), 1 / math.sqrt(512)), device)
        self.n_entries = torch.full((B,), self.N - 1, dtype=torch.int32, device=device)
        self.topk = torch.empty((B, 1, wl.topk), dtype=torch.int32, device=device)
        self.pool = torch.empty((B, 1, wl.hsi_blocks), dtype=torch.int32, device=device) if wl.hsi else None
        self.ws = torch.empty(csa.index_workspace_bytes(self.cfg, B, 1, self.N), dtype=torch.uint8, device=device)
        self.out = torch.empty((B, 1, 64, 512), dtype=torch.float32, device=device)
        self.stages = ["compress", "index_score", "index_select", "attend"]
        self.launches_per_step = 4  # compress, score, select, attend
        eb = idx_entry_bytes(wl)
        self.stage_bytes = {"compress": B * (r * 1024 + (288 + eb if wl.cache == "fp4" else 1280)),
                            "index_score": B * self.N * eb,
                            "index_select": B * select_bytes(self.N, wl),
                            "attend": B * attend_query_bytes(wl.cache, wl.topk, wl.window, swa_row_bytes(wl))}
        self.stage_kernels = {"compress": "compress_kernel", "index_score": "score_tc_kernel",
                              "index_select": "select_kernel", "attend": attend_kernel(wl.topk, wl.window)}
        if wl.swa_fp8:
            self.stages.insert(1, "swa_encode")
            self.launches_per_step += 1
            self.stage_bytes["swa_encode"] = B * (1024 + 528)
            self.stage_kernels["swa_encode"] = "swa_encode_kernel"
        self.units = B
        self.cfg_extra = {"batch_per_gpu": B, "ctx": ctx, "entries": self.N}

    def calls(self, d):
        csa, st = self.csa, self.status
        c = [
            lambda: csa.compress(self.cfg, d["x"], d["pos0"], self.merge_w, self.w_idx, self.main, self.idx,
                                 self.n_entries, status=st),
            lambda: csa.index_score(self.cfg, d["q_idx"], d["q_pos"], self.idx, self.n_entries, self.N, self.ws,
                                    hsi=self.pool is not None, status=st),
            lambda: csa.index_select(self.cfg, d["q_pos"], self.idx, self.n_entries, self.N, self.topk, self.ws,
                                     pool_out=self.pool, status=st),
            lambda: csa.attend(self.cfg, d["q"], self.main, self.n_entries, self.topk,
                               self.swa8 if self.wl.swa_fp8 else d["swa"], d["swa_len"], d["swa_pos0"], d["q_pos"],
                               self.out, status=st),
        ]
        if self.wl.swa_fp8:
            c.insert(1, lambda: csa.swa_encode(d["swa_new"], self.swa_row0, self.swa8, status=st))
        return c


class PrefillStep(StepBase):
    """One chunk of Tq query tokens per sequence appended to a long context (a
    prefill chunk, or a multi-query decode block of draft positions): the
    compressor on the chunk's complete groups of r tokens (a trailing partial
    group stays in the window rows), causal indexing of every chunk token over
    the prefix plus the chunk's own entries, attention with the banded window
    (rows t-W+1..t of the chunk and the prefix tail)."""

    def __init__(self, wl, device, seed_offset=0):
        super().__init__(wl, device, seed_offset)
        torch, csa, B, r, s = self.torch, self.csa, self.B, wl.ratio, self.seed
        Tq, ctx, W = wl.tq, wl.ctx, wl.window
        Tc = Tq - Tq % r  # tokens that complete a compressor group
        self.N = (ctx + Tq) // r
        self.make_caches(self.N)
        S = W - 1 + Tq
        self.h = {
            "x": synth.normal_bf16(synth.rng(s, "x_chunk"), (B, Tc, 512)),
            "pos0": np.full(B, ctx, np.int64),
            "q": synth.normal_bf16(synth.rng(s, "q"), (B, Tq, 64, 512)),
            "q_idx": synth.normal_bf16(synth.rng(s, "q_idx"), (B, Tq, 32, 128)),
            "swa": synth.normal_bf16(synth.rng(s, "swa"), (B, S, 512)),
            "swa_len": np.full(B, S, np.int32),
            "swa_pos0": np.full(B, ctx - (W - 1), np.int64),
            "q_pos": np.tile(ctx + np.arange(Tq, dtype=np.int64), (B, 1)),
        }
        self.upload()
        self.merge_w = _dev(synth.merge_weights(synth.rng(s, "w"), r, 512), device)
        self.w_idx = _dev(synth.normal_bf16(synth.rng(s, "w_idx"), (512, 128), 1 / math.sqrt(512)), device)
        self.n_entries = torch.full((B,), ctx // r, dtype=torch.int32, device=device)
        self.topk = torch.empty((B, Tq, wl.topk), dtype=torch.int32, device=device)
        self.pool = None
        per_q = csa.index_workspace_bytes(self.cfg, 1, 1, self.N)
        self.chunk = index_chunk(per_q, B * Tq)
        self.ws = torch.empty(per_q * self.chunk, dtype=torch.uint8, device=device)
        self.out = torch.empty((B, Tq, 64, 512), dtype=torch.float32, device=device)
        if self.chunk < B * Tq:
            raise SystemExit("the indexer workspace of %s does not hold every query in one pass" % wl.name)
        self.stages = ["compress", "index_score", "index_select", "attend"]
        self.launches_per_step = 4
        pairs = sum(min((ctx + t - (r - 1)) // r + 1, self.N) for t in range(Tq)) * B
        self.stage_bytes = {"compress": B * (Tq // r) * (r * 1024 + 360),
                            "index_score": B * self.N * IDX_ENTRY_BYTES[wl.cache] + B * Tq * (8192 + 2048),
                            "index_select": B * Tq * select_bytes(self.N, wl),
                            "attend": B * Tq * attend_query_bytes(wl.cache, wl.topk, wl.window)}
        self.stage_flops = {"index_score": pairs * 8192, "attend": B * Tq * 4 * 64 * 512 * (wl.topk + wl.window)}
        self.stage_kernels = {"compress": "compress_kernel", "index_score": "score_tc_kernel",
                              "index_select": "select_kernel", "attend": attend_kernel(wl.topk, wl.window)}
        self.units = B * Tq
        self.cfg_extra = {"batch_per_gpu": B, "ctx": ctx, "query_tokens": Tq, "entries": self.N,
                          "index_pairs": pairs}

    calls = DecodeStep.calls


class GroupStep(StepBase):
    """One step through a cross-layer group: decoder layers 20-39 (layer 20
    Full: compress the new token, full indexing with the HSI pool; layers
    24/28/32/36 Reindex over the pool; the other fifteen Reuse) or the encoder
    macro block 2-7 (layer 2 Full without HSI, five Reuse), in decode (one
    query token per sequence) or on a prefill chunk of Tq tokens (the Full
    layer compresses the chunk and indexes every chunk token causally); every
    layer has its own query, indexer query and window rows."""

    def __init__(self, wl, device, seed_offset=0):
        super().__init__(wl, device, seed_offset)
        torch, csa, B, r, s = self.torch, self.csa, self.B, wl.ratio, self.seed
        ctx, Tq, W = wl.ctx, wl.tq, wl.window
        self.N = (ctx + Tq) // r if Tq > 1 else ctx // r
        self.make_caches(self.N)
        self.layers = list(wl.layers)
        S = W - 1 + Tq if Tq > 1 else W
        if Tq > 1:
            self.h = {"x": synth.normal_bf16(synth.rng(s, "x_chunk"), (B, Tq, 512)), "pos0": np.full(B, ctx, np.int64),
                      "swa_len": np.full(B, S, np.int32), "swa_pos0": np.full(B, ctx - (W - 1), np.int64),
                      "q_pos": np.tile(ctx + np.arange(Tq, dtype=np.int64), (B, 1))}
        else:
            self.h = {"x": synth.normal_bf16(synth.rng(s, "x_step"), (B, r, 512)), "pos0": np.full(B, ctx - r, np.int64),
                      "swa_len": np.full(B, W, np.int32), "swa_pos0": np.full(B, ctx - W, np.int64),
                      "q_pos": np.full((B, 1), ctx - 1, np.int64)}
        for layer, mode in self.layers:
            ls = s * 1000 + layer
            self.h["q%d" % layer] = synth.normal_bf16(synth.rng(ls, "q"), (B, Tq, 64, 512))
            self.h["swa%d" % layer] = synth.normal_bf16(synth.rng(ls, "swa"), (B, S, 512))
            if mode != "reuse":
                self.h["q_idx%d" % layer] = synth.normal_bf16(synth.rng(ls, "q_idx"), (B, Tq, 32, 128))
        self.upload()
        self.merge_w = _dev(synth.merge_weights(synth.rng(s, "w"), r, 512), device)
        self.w_idx = _dev(synth.normal_bf16(synth.rng(s, "w_idx"), (512, 128), 1 / math.sqrt(512)), device)
        self.n_entries = torch.full((B,), ctx // r if Tq > 1 else self.N - 1, dtype=torch.int32, device=device)
        topk = torch.empty((B, Tq, wl.topk), dtype=torch.int32, device=device)
        pool = torch.empty((B, Tq, wl.hsi_blocks), dtype=torch.int32, device=device) if wl.hsi else None
        nq = index_chunk(csa.index_workspace_bytes(self.cfg, 1, 1, self.N), B * Tq)  # queries per indexer pass
        ws = torch.empty(max(csa.index_workspace_bytes(self.cfg, 1, nq, self.N),
                             csa.index_workspace_bytes(self.cfg, 1, nq, self.N, reindex=True)),
                         dtype=torch.uint8, device=device)
        self.state = csa.GroupState(self.main, self.idx, self.n_entries, self.N, topk, pool, ws, self.status)
        self.outs = {l: torch.empty((B, Tq, 64, 512), dtype=torch.float32, device=device) for l, _ in self.layers}
        self.out = self.outs[self.layers[-1][0]]
        self.stages = ["L%d_%s" % (l, m) for l, m in self.layers]
        chunks = -(-B * Tq // nq)
        self.launches_per_step = sum({"full": 2 + 2 * chunks, "reindex": 1 + 2 * chunks, "reuse": 1}[m]
                                     for _, m in self.layers)
        att = B * Tq * attend_query_bytes(wl.cache, wl.topk, wl.window)
        eb = idx_entry_bytes(wl)
        self.stage_bytes, self.stage_flops = {}, {}
        pairs = (sum(min((ctx + t - (r - 1)) // r + 1, self.N) for t in range(Tq)) * B if Tq > 1 else B * self.N)
        for l, m in self.layers:
            comp = B * (Tq // r if Tq > 1 else 1) * (r * 1024 + 360)
            extra = {"full": B * self.N * eb + comp + (B * Tq * (8192 + 2048) if Tq > 1 else 0),
                     "reindex": B * Tq * wl.hsi_blocks * 8 * eb, "reuse": 0}[m]
            self.stage_bytes["L%d_%s" % (l, m)] = att + extra
            if Tq > 1 and m == "full":
                self.stage_flops["L%d_%s" % (l, m)] = pairs * 8192
        att_k = attend_kernel(wl.topk, wl.window).replace("_kernel", "")
        self.stage_kernels = {st: {"full": "compress + score_tc + select + " + att_k,
                                   "reindex": "score_tc (gather) + select + " + att_k,
                                   "reuse": att_k}[st.split("_")[1]]
                              for st in self.stages}
        self.units = B * Tq
        self.cfg_extra = {"batch_per_gpu": B, "ctx": ctx, "entries": self.N, "layers": len(self.layers),
                          "query_tokens": Tq,
                          "unit": "query token through the %d-layer group" % len(self.layers)}

    def late_inputs(self):
        """The per-layer inputs of every layer after the first."""
        first = self.layers[0][0]
        late = set()
        for k in self.h:
            m = re.fullmatch(r"(q|q_idx|swa)(\d+)", k)
            if m and int(m.group(2)) != first:
                late.add(k)
        return 1, late

    def calls(self, d):
        csa = self.csa
        mode_of = {"full": csa.MODE_FULL, "reindex": csa.MODE_REINDEX, "reuse": csa.MODE_REUSE}
        out = []
        for l, m in self.layers:
            kw = {}
            if m == "full":
                kw = dict(x=d["x"], pos0=d["pos0"], merge_w=self.merge_w, w_idx=self.w_idx)
            out.append(lambda l=l, m=m, kw=kw: csa.layer(
                self.cfg, mode_of[m], self.state, d["q_pos"], d["q%d" % l], d["swa%d" % l], d["swa_len"],
                d["swa_pos0"], self.outs[l], q_idx=d.get("q_idx%d" % l), **kw))
        return out


def make_step(name, device, seed_offset=0):
    wl = synth.WORKLOADS[name]
    if wl.layers:
        return GroupStep(wl, device, seed_offset)
    if wl.tq > 1:
        return PrefillStep(wl, device, seed_offset)
    return DecodeStep(wl, device, seed_offset)


# ------------------------------------------------------------- cpu oracle ----

class OracleStep:
    """The CPU oracle on a bounded sample of the same workload, with its own
    seeded random cache: decode -- up to 4 sequences through the step
    (compress, index, attend); decoder group -- one sequence through all 20
    layers; prefill -- the chunk's compressor and 4 query rows."""

    def __init__(self, wl: synth.Workload):
        import oracle
        self.oracle, self.wl = oracle, wl
        r = wl.ratio
        self.prefill = wl.tq > 1
        self.B = 1 if (wl.layers or self.prefill) else min(wl.batch, 4)
        B = self.B
        N = (wl.ctx + wl.tq) // r if self.prefill else wl.ctx // r
        self.N = N
        self.main = oracle.Cache(B, N, 512, wl.cache)
        self.idx = oracle.Cache(B, N, 128, "fp4g32" if wl.idx68 else wl.cache)
        g = synth.rng(wl.seed, "oracle_cache")
        for c in (self.main, self.idx):
            if c.dtype != "bf16":
                for b in range(B):
                    c.codes[b], c.scales[b] = synth.fp4_bytes(g, N, c.channels, group=32 if c.dtype == "fp4g32" else 16)
            else:
                c.bf16[:] = synth.normal_bf16(g, c.bf16.shape)
        s, ctx = wl.seed, wl.ctx
        self.w = synth.merge_weights(synth.rng(s, "w"), r, 512)
        self.w_idx = synth.normal_bf16(synth.rng(s, "w_idx"), (512, 128), 1 / math.sqrt(512))
        if self.prefill:
            # every row of a short block, else 4 rows: both ends and both sides of position 2048
            rows = np.arange(wl.tq) if wl.tq <= 8 else np.array([0, 2047, 2048, wl.tq - 1], np.int64)
            Tc = wl.tq - wl.tq % r
            self.x = synth.normal_bf16(synth.rng(s, "x_chunk"), (1, Tc, 512))
            self.pos0 = np.array([ctx], np.int64)
            self.q = synth.normal_bf16(synth.rng(s, "q"), (1, wl.tq, 64, 512))[:, rows]
            self.q_idx = synth.normal_bf16(synth.rng(s, "q_idx"), (1, wl.tq, 32, 128))[:, rows]
            S = wl.window - 1 + wl.tq
            self.swa = synth.normal_bf16(synth.rng(s, "swa"), (1, S, 512))
            self.swa_len, self.swa_pos0 = np.array([S], np.int32), np.array([ctx - wl.window + 1], np.int64)
            self.q_pos = (ctx + rows).reshape(1, -1)
            self.n_ent = np.array([N], np.int32)
            self.units = len(rows)
            self.sample = ("all %d query rows of one sequence's block plus its compressor" % wl.tq if wl.tq <= 8 else
                           "4 query rows (0, 2047, 2048, last) of the %d-token chunk plus its compressor" % wl.tq)
            if wl.layers:  # the same rows through every layer of the group, each with its own inputs
                self.per_layer = []
                for layer, mode in wl.layers:
                    ls = s * 1000 + layer
                    self.per_layer.append((layer, mode,
                                           synth.normal_bf16(synth.rng(ls, "q"), (1, wl.tq, 64, 512))[:, rows],
                                           synth.normal_bf16(synth.rng(ls, "swa"), (1, S, 512)),
                                           synth.normal_bf16(synth.rng(ls, "q_idx"), (1, wl.tq, 32, 128))[:, rows]))
                self.sample += ", through the %d-layer group" % len(wl.layers)
        else:
            self.x = synth.normal_bf16(synth.rng(s, "x_step"), (B, r, 512))
            self.pos0 = np.full(B, ctx - r, np.int64)
            self.q_pos = np.full((B, 1), ctx - 1, np.int64)
            self.swa_len, self.swa_pos0 = np.full(B, wl.window, np.int32), np.full(B, ctx - wl.window, np.int64)
            self.n_ent = np.full(B, N, np.int32)
            if wl.layers:
                self.per_layer = []
                for layer, mode in wl.layers:
                    ls = s * 1000 + layer
                    self.per_layer.append((layer, mode,
                                           synth.normal_bf16(synth.rng(ls, "q"), (1, 1, 64, 512)),
                                           synth.normal_bf16(synth.rng(ls, "swa"), (1, wl.window, 512)),
                                           synth.normal_bf16(synth.rng(ls, "q_idx"), (1, 1, 32, 128))))
                self.units = 1
                self.sample = "1 sequence through the %d-layer group" % len(wl.layers)
            else:
                self.q = synth.normal_bf16(synth.rng(s, "q"), (B, 1, 64, 512))
                self.q_idx = synth.normal_bf16(synth.rng(s, "q_idx"), (B, 1, 32, 128))
                self.swa = synth.normal_bf16(synth.rng(s, "swa"), (B, wl.window, 512))
                if wl.swa_fp8:  # resident MXFP8 window; the step encodes the newest row
                    self.swa_new = np.ascontiguousarray(self.swa[:, -1:])
                    self.swa = oracle.swa_encode(self.swa)
                self.units = B
                self.sample = "%d sequences of the step (compress + index over %d entries + attend)" % (B, N)
        self.cores = min(oracle.threads(), max(self.units, 1))

    def step(self):
        o, wl = self.oracle, self.wl
        sc = 1 / math.sqrt(512)
        o.compress(self.x, self.pos0, self.w, self.w_idx, self.main, self.idx, wl.ratio, wl.theta)
        if wl.swa_fp8:
            self.swa[:, -1:] = o.swa_encode(self.swa_new)
        if not wl.layers:
            topk, _, _ = o.index_topk(self.idx, self.n_ent, self.q_idx, self.q_pos, wl.ratio, wl.topk,
                                      hsi_blocks=wl.hsi_blocks if wl.hsi else 0, want_pool=wl.hsi, q_fp4=wl.q_fp4)
            return o.attend(self.main, self.n_ent, self.q, topk, self.swa, self.swa_len, self.swa_pos0, self.q_pos,
                            wl.window, sc)
        topk = pool = None
        for layer, mode, q, swa, q_idx in self.per_layer:
            if mode == "full":
                topk, pool, _ = o.index_topk(self.idx, self.n_ent, q_idx, self.q_pos, wl.ratio, wl.topk,
                                             hsi_blocks=wl.hsi_blocks if wl.hsi else 0, want_pool=wl.hsi)
            elif mode == "reindex":
                topk, _, _ = o.index_topk(self.idx, self.n_ent, q_idx, self.q_pos, wl.ratio, wl.topk,
                                          hsi_blocks=wl.hsi_blocks, pool=pool)
            out = o.attend(self.main, self.n_ent, q, topk, swa, self.swa_len, self.swa_pos0, self.q_pos, wl.window, sc)
        return out


def cpu_baseline(wl, seconds: float):
    st = OracleStep(wl)
    t0 = time.perf_counter()
    n = 0
    while True:
        st.step()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": n * st.units / dt, "unit": UNIT, "cores": st.cores, "kind": "oracle",
            "sample": "%d runs of %s: %s; fp64 C oracle, OpenMP over query tokens" % (n, wl.name, st.sample)}


# -------------------------------------------------------------------- main ----

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, ws, rank):
    """The oracle as it stands, on the host cores, on this arm's workload."""
    wl = synth.WORKLOADS[args.workload]
    if rank != 0:
        return
    st = OracleStep(wl)
    for _ in range(args.warmup):
        st.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.step()
    dt = time.perf_counter() - t0
    v = args.steps * st.units / dt
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name}, "impl": "reference",
            "cpu_baseline": {"value": v, "unit": UNIT, "kind": "oracle", "cores": st.cores,
                             "sample": "%d runs of %s: %s" % (args.steps, wl.name, st.sample)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_step(step, steps, warmup, flush, ws):
    """Warm-up, then K graph replays of the whole step (each after an L2
    flush, bracketed by CUDA events on the launching stream), one graph per
    stage replayed back to back after the same flush, the eager step through
    the Python API, and warm-L2 replays."""
    import torch
    nst = len(step.stages)
    for _ in range(warmup):
        flush_l2(flush, 1)
        step.step()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, "device status %d" % int(step.status.item())
    # the step and each of its stages captured once as CUDA graphs (decode
    # steps are a handful of short kernels: replaying a graph removes the
    # host-side launch gaps between them)
    calls = step.calls(step.d)
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        for c in calls:
            c()
    g_stage = []
    for c in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            c()
        g_stage.append(g)
    for _ in range(2):
        flush_l2(flush, 2)
        g_step.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(steps):
        flush_l2(flush, k & 0xFF)
        evs[k][0].record()
        g_step.replay()
        evs[k][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(ws)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    # per-stage durations (stage graphs back to back after the flush) and
    # the same step launched eagerly through the Python API
    n_stage = min(steps, 50)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(n_stage)]
    for k in range(n_stage):
        flush_l2(flush, k & 0xFF)
        for i, g in enumerate(g_stage):
            sev[k][i].record()
            g.replay()
        sev[k][nst].record()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(n_stage)]
    for k in range(n_stage):
        flush_l2(flush, k & 0xFF)
        step.step(events=eev[k])
    torch.cuda.synchronize()
    # warm variant: the same graph replayed back to back without the L2 flush
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_stage)]
    for k in range(n_stage):
        wev[k][0].record()
        g_step.replay()
        wev[k][1].record()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return {"step_ms": step_ms, "wall": wall, "g_step": g_step,
            "stage_ms": {s: statistics.fmean(e[i].elapsed_time(e[i + 1]) for e in sev)
                         for i, s in enumerate(step.stages)},
            "eager_ms": statistics.fmean(e[0].elapsed_time(e[nst]) for e in eev),
            "eager_stage_ms": {s: statistics.fmean(e[i].elapsed_time(e[i + 1]) for e in eev)
                               for i, s in enumerate(step.stages)},
            "warm_ms": statistics.fmean(a.elapsed_time(b) for a, b in wev)}


def roofline_of(step, stage_ms):
    """Roofline of the dominant stage (the longest): its algorithmic FLOPs
    against the sustained tensor peak where the stage is a contraction with a
    FLOP count (prefill indexer), else its algorithmic bytes against the
    measured HBM copy bandwidth; DRAM traffic per launch from the ncu capture
    named in TRAFFIC, when there is one of the current kernels."""
    hbm, tflops_sus, src = peaks()
    dom = max(stage_ms, key=stage_ms.get)
    flops = getattr(step, "stage_flops", {}).get(dom)
    traffic, traffic_src = TRAFFIC.get(step.wl.name, {}).get(dom, (None, None))
    if step.B != step.wl.batch:
        traffic, traffic_src = None, None  # the captures are of the workload's own batch
    if flops is not None:
        # f16 operands run at the bf16 rate; the sustained figure, the kernel
        # runs inside a long step
        ach = flops / (stage_ms[dom] / 1e3) / 1e12
        return {"bound": "tensor", "kernel": step.stage_kernels[dom], "stage": dom, "achieved": ach,
                "peak": tflops_sus, "unit": "TFLOP/s", "frac": ach / tflops_sus, "traffic": traffic,
                "traffic_source": traffic_src,
                "peak_source": ("of measured (MEASURED_PEAKS.json bf16_tflops_sustained, f16 = bf16 rate)"
                                if src == "measured" else "of fallback"),
                "algorithmic_flops_per_launch": flops, "launch_ms": stage_ms[dom]}
    ach = step.stage_bytes[dom] / (stage_ms[dom] / 1e3) / 1e9
    return {"bound": "hbm", "kernel": step.stage_kernels[dom], "stage": dom, "achieved": ach, "peak": hbm,
            "unit": "GB/s", "frac": ach / hbm, "traffic": traffic, "traffic_source": traffic_src,
            "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "of fallback",
            "algorithmic_bytes_per_launch": step.stage_bytes[dom], "launch_ms": stage_ms[dom]}


def measure_target(name, dev, flush, steps, warmup):
    """One of the workloads with a stated target, measured in the same run:
    whole-step graph replays after an L2 flush, per-stage times, the
    roofline of its dominant stage, and the target beside the figure."""
    import torch
    step = make_step(name, dev)
    t = time_step(step, steps, warmup, flush, 1)
    ms = statistics.fmean(t["step_ms"])
    out = {"value": step.units / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
           "config": dict({"workload": name}, **step.cfg_extra), "stage_ms": t["stage_ms"],
           "roofline": roofline_of(step, t["stage_ms"]), "target": TARGETS[name],
           "gpu_launches": step.launches_per_step * steps}
    del step, t
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences per GPU instead of the workload's own (smaller profiling captures)")
    ap.add_argument("--tq", type=int, default=None,
                    help="query tokens per sequence instead of the workload's own (smaller prefill captures)")
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the decoder-group and prefill target workloads measured beside the default one")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.batch is not None:
        wl = synth.WORKLOADS[args.workload]
        synth.WORKLOADS[args.workload] = dataclasses.replace(wl, batch=args.batch)
    if args.tq is not None:
        wl = synth.WORKLOADS[args.workload]
        synth.WORKLOADS[args.workload] = dataclasses.replace(wl, tq=args.tq)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        barrier(ws)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    step = make_step(args.workload, dev, seed_offset=rank)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    clocks = ClockSampler(local)
    clocks.start()
    t = time_step(step, args.steps, args.warmup, flush, ws)
    clk = clocks.stop()
    step_ms, stage_ms = t["step_ms"], t["stage_ms"]
    total_ms = max_over_ranks(sum(step_ms), ws)
    ms_per_step = total_ms / args.steps
    value = ws * step.units * args.steps / (total_ms / 1e3)
    eager_ms, warm_ms, wall = t["eager_ms"], t["warm_ms"], t["wall"]

    # end to end through the Python API with host buffers: the step's inputs
    # in two pinned host buffers, each copied in with one H2D copy (the
    # device tensors the API is called with are views of two staging
    # buffers): the inputs of the first calls on the step's stream, the rest
    # (the attention's query and window rows) on a second stream so that
    # their upload overlaps the first calls; the step; D2H of the output
    host_in = {k: np.ascontiguousarray(v.view(np.int16) if v.dtype == np.uint16 else v)
               for k, v in step.inputs_host().items()}
    late_from, late_keys = step.late_inputs()
    dbuf, packs, total = {}, [], 0
    for group in ([k for k in host_in if k not in late_keys], [k for k in host_in if k in late_keys]):
        offs, size = {}, 0
        for k in group:
            offs[k] = size
            size += (host_in[k].nbytes + 255) & ~255
        if not size:
            packs.append(None)
            continue
        hpack = torch.empty(size, dtype=torch.uint8).pin_memory()
        dpack = torch.empty(size, dtype=torch.uint8, device=dev)
        for k in group:
            hv = torch.from_numpy(host_in[k])
            hpack[offs[k]:offs[k] + hv.numel() * hv.element_size()].copy_(hv.view(-1).view(torch.uint8))
            dbuf[k] = dpack[offs[k]:offs[k] + hv.numel() * hv.element_size()].view(hv.dtype).view(hv.shape)
        packs.append((hpack, dpack))
        total += size
    hout = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = total
    d2h = hout.numel() * hout.element_size()
    side = torch.cuda.Stream(device=dev)
    late_ready = torch.cuda.Event()

    def e2e_step():
        main = torch.cuda.current_stream()
        if packs[1] is not None:
            side.wait_stream(main)
            with torch.cuda.stream(side):
                packs[1][1].copy_(packs[1][0], non_blocking=True)
                late_ready.record(side)
        if packs[0] is not None:
            packs[0][1].copy_(packs[0][0], non_blocking=True)
        for i, c in enumerate(step.calls(dbuf)):
            if i == late_from and packs[1] is not None:
                main.wait_event(late_ready)
            c()
        hout.copy_(step.out, non_blocking=True)

    # recorded once through the package's public capture helper: one replay
    # per step issues the two H2D copies, the library calls and the D2H copy
    e2e = step.csa.capture(e2e_step)
    e2e_steps = max(3, min(args.steps, 50))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for k in range(e2e_steps):
        flush_l2(flush, k & 0xFF)
        e2e_ev[k][0].record()
        e2e()
        e2e_ev[k][1].record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), ws) / e2e_steps
    # the same, issued call by call through the Python API
    for k in range(e2e_steps):
        flush_l2(flush, k & 0xFF)
        e2e_ev[k][0].record()
        e2e_step()
        e2e_ev[k][1].record()
    torch.cuda.synchronize()
    e2e_eager_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), ws) / e2e_steps
    assert int(step.status.item()) == 0

    roof = roofline_of(step, stage_ms)
    wl_name, units, launches, cfg_extra = step.wl.name, step.units, step.launches_per_step, step.cfg_extra
    wl_obj = step.wl
    targets = None
    if ws == 1 and not args.no_targets and args.workload == DEFAULT_WORKLOAD and args.batch is None and args.tq is None:
        del step, e2e, packs, dbuf
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        targets = {name: measure_target(name, dev, flush, steps=max(10, min(args.steps, 40)), warmup=args.warmup)
                   for name in TARGETS}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl_obj, args.cpu_seconds)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                "config": dict({"workload": wl_name}, **cfg_extra,
                               **{"cache": wl_obj.cache, "topk": wl_obj.topk, "window": wl_obj.window,
                                  "hsi": wl_obj.hsi, "operands": "f16 tensor-core operands, fp32 accumulate",
                                  "l2": "flushed before every step (256 MiB write, then 256 MiB read of a second buffer)",
                                  "launch": "CUDA graph of the step, captured once and replayed per step"}),
                "stage_ms": stage_ms, "eager_stage_ms": t["eager_stage_ms"], "eager_ms_per_step": eager_ms,
                "warm_l2": {"value": ws * units / (max_over_ranks(warm_ms, ws) / 1e3), "unit": UNIT,
                            "ms_per_step": warm_ms},
                "median_ms_per_step": statistics.median(step_ms), "wall_s": wall,
                "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": ws * units / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                        "launch": "csa.capture of the step: H2D of the first calls' inputs, the API calls with the "
                                  "attention inputs' H2D overlapped on a second stream, one D2H copy",
                        "eager_value": ws * units / (e2e_eager_ms / 1e3)},
                "gpu_launches": launches * args.steps, "clocks": clk}
        if targets is not None:
            line["targets"] = targets
        print(json.dumps(line), flush=True)
    barrier(ws)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
