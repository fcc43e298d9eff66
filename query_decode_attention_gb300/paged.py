"""Filling and reading paged q8 caches through the public API.

``fill_cache`` writes every token of a workload's sequences into a fresh
``PagedKVCache`` with ``kq8_append_kv`` (the library's write path), drawing
fp32 K/V chunk by chunk on the device so that full-size caches never need
their fp32 form in memory at once.  ``unpack`` reads a pool back into the
logical [T, nkv, 128] view for tests.
"""
from __future__ import annotations

import numpy as np
import torch

from . import kq8
from . import workloads as W

GEN_CHUNK = 65536  # tokens drawn per device generator call


class DeviceCase:
    """A workload's layer resident on the device: cache, page table, lengths, q."""

    def __init__(self, wl: W.Workload, cache: kq8.PagedKVCache, page_table_np: np.ndarray,
                 device, layer: int = 0, q: torch.Tensor = None):
        self.wl = wl
        self.layer = layer
        self.cache = cache
        self.page_table_np = page_table_np
        self.page_table = torch.tensor(page_table_np, dtype=torch.int32, device=device)
        self.seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=device)
        self.q = q if q is not None else W.device_q(wl, layer, device)
        self.device = device

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        return W.slots_for(self.wl, self.page_table_np, b, t0, t1)

    def device_kv(self, b: int, t0: int, t1: int):
        """The fp32 K, V the cache was filled from, tokens [t0, t1) of sequence b
        (t0 a multiple of GEN_CHUNK: the draws are seeded per chunk)."""
        assert t0 % GEN_CHUNK == 0
        n = int(self.wl.seq_lens[b])
        parts = [W.device_kv_chunk(self.wl, self.layer, b, c0, min(c0 + GEN_CHUNK, n), self.device)
                 for c0 in range(t0, t1, GEN_CHUNK)]
        if len(parts) == 1:
            K, V = parts[0]
        else:
            K = torch.cat([p[0] for p in parts])
            V = torch.cat([p[1] for p in parts])
        return K[:t1 - t0], V[:t1 - t0]


def new_cache(wl: W.Workload, extra_pages: int = 0, device="cuda", pt_seed=None, bits: int = 8):
    pt, num_pages = W.page_table(wl, extra_pages=extra_pages, seed=pt_seed)
    cache = kq8.PagedKVCache(num_pages, wl.nkv, wl.kv_bs, device=device, bits=bits)
    return cache, pt


def fill_cache(wl: W.Workload, layer: int = 0, device="cuda", extra_pages: int = 0,
               cache: kq8.PagedKVCache = None, pt=None, status=None, bits: int = 8) -> DeviceCase:
    """Quantise every token of every sequence into a paged cache on `device`
    (q8, or the q4 cache with bits=4)."""
    if cache is None:
        cache, pt = new_cache(wl, extra_pages, device, bits=bits)
    append = kq8.kq8_append_kv if cache.bits == 8 else kq8.kq8_append_kv_q4
    case = DeviceCase(wl, cache, pt, device, layer)
    for b in range(wl.B):
        n = int(wl.seq_lens[b])
        for t0 in range(0, n, GEN_CHUNK):
            t1 = min(n, t0 + GEN_CHUNK)
            K, V = W.device_kv_chunk(wl, layer, b, t0, t1, device)
            sl = torch.tensor(case.slots(b, t0, t1), dtype=torch.int32, device=device)
            append(cache, K, V, sl, status=status)
            del K, V
    return case


def fill_from_host(wl: W.Workload, Ks, Vs, device="cuda", extra_pages: int = 0,
                   q_host: np.ndarray = None, pt_seed=None, bits: int = 8) -> DeviceCase:
    """Quantise host fp32 K/V lists (one [n_b, nkv, 128] array per sequence)."""
    cache, pt = new_cache(wl, extra_pages, device, pt_seed, bits=bits)
    q = torch.tensor(q_host, device=device) if q_host is not None else None
    case = DeviceCase(wl, cache, pt, device, 0, q=q)
    if wl.B and wl.total_tokens:
        K = torch.tensor(np.concatenate([k.reshape(-1, wl.nkv, wl.hd) for k in Ks]), device=device)
        V = torch.tensor(np.concatenate([v.reshape(-1, wl.nkv, wl.hd) for v in Vs]), device=device)
        sl = torch.tensor(W.all_slots(wl, pt), dtype=torch.int32, device=device)
        (kq8.kq8_append_kv if bits == 8 else kq8.kq8_append_kv_q4)(cache, K, V, sl)
    return case


def unpack(cache: kq8.PagedKVCache, slots: np.ndarray):
    """Codes and stored maxima of the given pool slots, logical layout:
    (k8 [T, nkv, 128], ks [T, nkv], v8 [T, nkv, 128], vs [T, nkv]) numpy."""
    s = torch.as_tensor(np.asarray(slots, np.int64), device=cache.k.device)
    page, r = s // cache.kv_bs, s % cache.kv_bs
    # k: [P, nkv, sub, 4, 32, 32] -> row r is [.., r//32, :, kpos(r%32), :] with
    # kpos(x) = (x%4)*8 + x//4 (rows 0, 4, 8, ... adjacent)
    pos = (r % 32 % 4) * 8 + (r % 32) // 4
    k = cache.k[page, :, r // 32]                     # [T, nkv, 4, 32, 32]
    k = k[torch.arange(len(s), device=s.device), :, :, pos, :]  # [T, nkv, 4, 32]
    k8 = k.reshape(len(s), cache.num_kv_heads, 128)
    v8 = cache.v[page, :, r]                          # [T, nkv, 128]
    ks = cache.kscale[page, :, r]
    vs = cache.vscale[page, :, r]
    return (k8.cpu().numpy(), ks.cpu().numpy(), v8.cpu().numpy(), vs.cpu().numpy())


def unpack_q4(cache: kq8.PagedKVCache, slots: np.ndarray):
    """Codes (int8 in [-7, 7]) and stored maxima of a q4 cache's slots, logical
    layout [T, nkv, 128]: element e of a row is nibble e % 8 // 4 of byte
    e % 4 of word e % 32 // 8 of its block's 16 bytes, stored as code + 8."""
    s = torch.as_tensor(np.asarray(slots, np.int64), device=cache.k.device)
    page, r = s // cache.kv_bs, s % cache.kv_bs
    pos = (r % 32 % 4) * 8 + (r % 32) // 4
    k = cache.k[page, :, r // 32]                      # [T, nkv, 4, 32, 16]
    k = k[torch.arange(len(s), device=s.device), :, :, pos, :]  # [T, nkv, 4, 16]
    v = cache.v[page, :, r]                            # [T, nkv, 64]

    def nibbles(b):  # [..., 16 * n] bytes -> [..., 32 * n] codes in element order
        u = b.to(torch.int32) & 0xFF
        w = u.reshape(*u.shape[:-1], -1, 4)            # words of 4 bytes
        lo, hi = w & 0xF, w >> 4
        return (torch.cat([lo, hi], dim=-1).reshape(*u.shape[:-1], -1) - 8).to(torch.int8)
    k4 = nibbles(k).reshape(len(s), cache.num_kv_heads, 128)
    v4 = nibbles(v).reshape(len(s), cache.num_kv_heads, 128)
    ks = cache.kscale[page, :, r]
    vs = cache.vscale[page, :, r]
    return (k4.cpu().numpy(), ks.cpu().numpy(), v4.cpu().numpy(), vs.cpu().numpy())
