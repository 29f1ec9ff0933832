"""Test-side conversion between the oracle's canonical (unpaged) caches and the
library's paged device caches, written from the layout documented in
include/csa2.h.  Index shuffling only: no arithmetic of the method."""
import numpy as np
import torch

import compressed_sparse_attention_07_gb300 as csa

PAGE = 64


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy -> device tensor; uint16 bit patterns travel as int16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


def page_order(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of the page pool (fragmented page tables)."""
    return np.random.default_rng(seed).permutation(n)


def _pad_entries(a: np.ndarray, cap: int) -> np.ndarray:
    B, N = a.shape[:2]
    if N == cap:
        return a
    out = np.zeros((B, cap) + a.shape[2:], a.dtype)
    out[:, :N] = a
    return out


def _group(cache) -> int:
    """Channels per FP4 scale: 16, or 32 for the 68-byte indexer entry."""
    return 32 if cache.cache_dtype == csa.CACHE_FP4_S32 else 16


def _page_bytes(cache: csa.PagedCache, canon_codes: np.ndarray, canon_scales):
    """Canonical [B][cap][...] -> per-page byte rows in block-table order."""
    B, mp = cache.batch, cache.max_pages
    C_ = cache.channels
    codes = _pad_entries(canon_codes, cache.capacity)
    if cache.cache_dtype != csa.CACHE_BF16:
        cb = codes.reshape(B, mp, PAGE, C_ // 2)
        if C_ == 128:  # 16-byte chunk c of slot s at (c*64 + s)*16
            cb = cb.reshape(B, mp, PAGE, 4, 16).transpose(0, 1, 3, 2, 4)
        sb = _pad_entries(canon_scales, cache.capacity).reshape(B, mp, PAGE * (C_ // _group(cache)))
        return cb.reshape(B * mp, -1), sb.reshape(B * mp, -1)
    vb = codes.view(np.uint8).reshape(B, mp, PAGE, C_ * 2)
    if C_ == 128:
        vb = vb.reshape(B, mp, PAGE, 16, 16).transpose(0, 1, 3, 2, 4)
    return vb.reshape(B * mp, -1), None


def upload(cache: csa.PagedCache, ocache) -> None:
    """Copy an oracle.Cache (canonical) into the paged device cache."""
    if cache.cache_dtype != csa.CACHE_BF16:
        d, s = _page_bytes(cache, ocache.codes, ocache.scales)
    else:
        d, s = _page_bytes(cache, ocache.bf16, None)
    bt = cache.block_table.flatten().long()
    cache.data[bt] = torch.from_numpy(np.ascontiguousarray(d)).to(cache.data.device)
    if s is not None:
        cache.scales[bt] = torch.from_numpy(np.ascontiguousarray(s)).to(cache.data.device)


def download(cache: csa.PagedCache, n: int):
    """Paged device cache -> canonical arrays of the first n entries per sequence:
    (codes [B][n][C/2], scales [B][n][C/16]) for FP4, (values [B][n][C] uint16, None) for BF16."""
    B, mp, C_ = cache.batch, cache.max_pages, cache.channels
    bt = cache.block_table.flatten().long()
    d = cache.data[bt].cpu().numpy()
    if cache.cache_dtype != csa.CACHE_BF16:
        cb = d.reshape(B, mp, -1)
        if C_ == 128:
            cb = cb.reshape(B, mp, 4, PAGE, 16).transpose(0, 1, 3, 2, 4)
        codes = np.ascontiguousarray(cb).reshape(B, mp * PAGE, C_ // 2)[:, :n]
        s = cache.scales[bt].cpu().numpy().reshape(B, mp * PAGE, C_ // _group(cache))[:, :n]
        return codes, s
    vb = d.reshape(B, mp, -1)
    if C_ == 128:
        vb = vb.reshape(B, mp, 16, PAGE, 16).transpose(0, 1, 3, 2, 4)
    vals = np.ascontiguousarray(vb).reshape(B, mp * PAGE, C_ * 2).view(np.uint16)[:, :n]
    return vals, None


def cache_pair(B, capacity, channels, dtype: str, seed: int):
    """A paged device cache with a shuffled page table ("fp4", "fp4g32" or "bf16")."""
    cd = {"fp4": csa.CACHE_FP4, "fp4g32": csa.CACHE_FP4_S32, "bf16": csa.CACHE_BF16}[dtype]
    mp = -(-capacity // PAGE)
    order = page_order(seed, B * mp + 3)[: B * mp]
    return csa.PagedCache(B, capacity, channels, cd, page_order=order, spare_pages=3)


def upload_seq(cache: csa.PagedCache, b: int, ocache, ob: int = 0) -> None:
    """Copy sequence ob of an oracle.Cache into sequence b of the paged cache."""
    mp = cache.max_pages
    C_ = cache.channels
    n = ocache.n_cap
    one = type(ocache)(1, cache.capacity, C_, ocache.dtype)
    if ocache.dtype != "bf16":
        one.codes[0, :n], one.scales[0, :n] = ocache.codes[ob], ocache.scales[ob]
    else:
        one.bf16[0, :n] = ocache.bf16[ob]
    view = csa.PagedCache.__new__(csa.PagedCache)
    view.batch, view.channels, view.cache_dtype = 1, C_, cache.cache_dtype
    view.max_pages, view.capacity, view.num_pages = mp, cache.capacity, cache.num_pages
    view.data, view.scales = cache.data, cache.scales
    view.block_table = cache.block_table[b:b + 1]
    if ocache.dtype != "bf16":
        d, s = _page_bytes(view, one.codes, one.scales)
    else:
        d, s = _page_bytes(view, one.bf16, None)
    bt = view.block_table.flatten().long()
    cache.data[bt] = torch.from_numpy(np.ascontiguousarray(d)).to(cache.data.device)
    if s is not None:
        cache.scales[bt] = torch.from_numpy(np.ascontiguousarray(s)).to(cache.data.device)
