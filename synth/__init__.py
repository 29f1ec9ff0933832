"""Seeded synthetic inputs for CSA2 workloads.

This module only draws random numbers and encodes them as the bit patterns the
path consumes (bf16, fp32, FP4 code/scale bytes).  It holds none of the
method's arithmetic (no merge, RoPE, quantiser, scoring, selection or
softmax), so both the CUDA path and the CPU oracle can take their inputs from
it.  Every array comes from numpy's PCG64 seeded by (config seed, stream name).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "ENCODER_GROUP", "DECODER_GROUP", "rng", "normal_bf16", "merge_weights", "fp4_bytes",
    "bf16_bits_to_f64", "integer_fp4_bytes", "integer_bf16", "decode_inputs",
]


def rng(seed: int, stream: str) -> np.random.Generator:
    """Independent generator per (seed, stream name)."""
    key = zlib.crc32(stream.encode())
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, key])))


def normal_bf16(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) drawn in fp64, rounded to bf16; returned as uint16 bit patterns."""
    x = g.standard_normal(size=shape) * std
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def merge_weights(g: np.random.Generator, r: int, dim: int) -> np.ndarray:
    """Per-channel merge weights [r][dim] fp32.  r = 2: (cos phi, sin phi) with
    phi ~ U(0, pi/2) per channel, so that merging two N(0,1) latents gives an
    N(0,1) entry; r = 1: ones."""
    if r == 1:
        return np.ones((1, dim), dtype=np.float32)
    if r != 2:
        raise ValueError("merge weights are defined for r in {1, 2}")
    phi = g.uniform(0.0, np.pi / 2, size=dim)
    return np.stack([np.cos(phi), np.sin(phi)]).astype(np.float32)


def fp4_bytes(g: np.random.Generator, n: int, channels: int, scale_lo: int = 0x20, scale_hi: int = 0x3C,
              group: int = 16):
    """Random FP4 entries in canonical form: codes [n][channels/2] (uniform bytes,
    i.e. uniform E2M1 codes) and E4M3 scales [n][channels/group] drawn uniformly
    from the byte range [scale_lo, scale_hi] (0x20..0x3C = 0.125..0.875 x 2^0)."""
    codes = g.integers(0, 256, size=(n, channels // 2), dtype=np.uint8)
    scales = g.integers(scale_lo, scale_hi + 1, size=(n, channels // group), dtype=np.uint8)
    return codes, scales


# E2M1 codes whose values are integers: 0, 1, 2, 3, 4, 6 and their negatives.
_INT_E2M1 = np.array([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], dtype=np.uint8)


def integer_fp4_bytes(g: np.random.Generator, n: int, channels: int):
    """FP4 entries whose decoded values are integers: codes from the integer
    E2M1 values, every scale byte 0x38 (= 1.0 in E4M3)."""
    lo = _INT_E2M1[g.integers(0, len(_INT_E2M1), size=(n, channels // 2))]
    hi = _INT_E2M1[g.integers(0, len(_INT_E2M1), size=(n, channels // 2))]
    codes = (lo | (hi << 4)).astype(np.uint8)
    scales = np.full((n, channels // 16), 0x38, dtype=np.uint8)
    return codes, scales


def integer_bf16(g: np.random.Generator, shape, lo: int = -3, hi: int = 3) -> np.ndarray:
    """Integers in [lo, hi] as bf16 bit patterns (exact)."""
    x = g.integers(lo, hi + 1, size=shape).astype(np.float64)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class Workload:
    """One synthetic CSA2 workload; sizes follow the configurations the
    write-ups' model description implies (64 heads x 512 latent, 64 RoPE
    dims, indexer 32 x 128, top-512, SWA-128, HSI 2048 blocks of 8)."""
    name: str
    batch: int
    ctx: int               # tokens already in the context (decode) / prefix (prefill)
    ratio: int             # compress ratio r
    cache: str             # "fp4" or "bf16"
    theta: float
    seed: int
    tq: int = 1            # query tokens per sequence (decode 1)
    hsi: bool = False      # hierarchical sparse indexer (decoder Full layer)
    layers: tuple = ()     # cross-layer group schedule, empty for a single layer
    dim: int = 512
    rope_dims: int = 64
    heads: int = 64
    idx_heads: int = 32
    idx_dim: int = 128
    topk: int = 512
    window: int = 128
    hsi_blocks: int = 2048
    hsi_block: int = 8
    idx68: bool = False    # indexer entries of 68 B (one E4M3 scale per 32 channels)
    swa_fp8: bool = False  # MXFP8 window rows (528 B) instead of bf16
    q_fp4: bool = False    # indexer queries scored in FP4 (E2M1, E4M3 per 16 channels)
    extra: dict = field(default_factory=dict)

    @property
    def entries(self) -> int:
        """Main-KV entries per sequence once the step's tokens are compressed."""
        return (self.ctx + self.tq) // self.ratio if self.tq > 1 else self.ctx // self.ratio


# Decoder group schedule: layer 20 Full (+HSI), 24/28/32/36 Reindex, rest Reuse.
DECODER_GROUP = tuple(
    (l, "full" if l == 20 else "reindex" if l in (24, 28, 32, 36) else "reuse") for l in range(20, 40)
)

# The encoder's first CSA2 macro block: layer 2 Full, layers 3-7 Reuse (r = 2, no HSI).
ENCODER_GROUP = tuple((l, "full" if l == 2 else "reuse") for l in range(2, 8))

WORKLOADS = {
    "decode_b1_ctx4096_r2_bf16": Workload(
        "decode_b1_ctx4096_r2_bf16", batch=1, ctx=4096, ratio=2, cache="bf16", theta=1e4, seed=0),
    "decode_b8_ctx32768_r2_fp4": Workload(
        "decode_b8_ctx32768_r2_fp4", batch=8, ctx=32768, ratio=2, cache="fp4", theta=1e4, seed=1),
    "decode_b32_ctx131072_r1_fp4_hsi": Workload(
        "decode_b32_ctx131072_r1_fp4_hsi", batch=32, ctx=131072, ratio=1, cache="fp4", theta=1.6e5,
        seed=2, hsi=True),
    "decoder_group20_b16_ctx262144_fp4": Workload(
        "decoder_group20_b16_ctx262144_fp4", batch=16, ctx=262144, ratio=1, cache="fp4", theta=1.6e5,
        seed=3, hsi=True, layers=DECODER_GROUP),
    "prefill_4096_on_1m_r2_fp4": Workload(
        "prefill_4096_on_1m_r2_fp4", batch=1, ctx=1048576, ratio=2, cache="fp4", theta=1e4, seed=4,
        tq=4096),
    "mqdecode_b8_q5_ctx32768_r2_fp4": Workload(
        "mqdecode_b8_q5_ctx32768_r2_fp4", batch=8, ctx=32768, ratio=2, cache="fp4", theta=1e4, seed=6, tq=5),
    "decode_b8_ctx32768_r2_fp4_idx68_fp8swa": Workload(
        "decode_b8_ctx32768_r2_fp4_idx68_fp8swa", batch=8, ctx=32768, ratio=2, cache="fp4", theta=1e4, seed=7,
        idx68=True, swa_fp8=True),
    "decode_b8_ctx32768_r2_fp4_qfp4": Workload(
        "decode_b8_ctx32768_r2_fp4_qfp4", batch=8, ctx=32768, ratio=2, cache="fp4", theta=1e4, seed=8, q_fp4=True),
    "encoder_group6_b8_ctx32768_r2_fp4": Workload(
        "encoder_group6_b8_ctx32768_r2_fp4", batch=8, ctx=32768, ratio=2, cache="fp4", theta=1e4, seed=5,
        layers=ENCODER_GROUP),
    "encoder_group6_prefill_4096_on_1m_r2_fp4": Workload(
        "encoder_group6_prefill_4096_on_1m_r2_fp4", batch=1, ctx=1048576, ratio=2, cache="fp4", theta=1e4, seed=9,
        tq=4096, layers=ENCODER_GROUP),
}


def decode_inputs(wl: Workload, batch: int | None = None, seed_offset: int = 0):
    """Per-step query-side inputs of one decode step (one query token per
    sequence at position ctx - 1): q [B][1][64][512], q_idx [B][1][32][128],
    SWA rows [B][W][512] at positions ctx-W..ctx-1, all bf16 bit patterns."""
    B = wl.batch if batch is None else batch
    s = wl.seed + seed_offset
    q = normal_bf16(rng(s, "q"), (B, 1, wl.heads, wl.dim))
    q_idx = normal_bf16(rng(s, "q_idx"), (B, 1, wl.idx_heads, wl.idx_dim))
    swa = normal_bf16(rng(s, "swa"), (B, wl.window, wl.dim))
    return q, q_idx, swa
