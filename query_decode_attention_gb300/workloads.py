"""Seeded synthetic workloads for q8-KV decode attention.

This module only draws inputs (fp32 q, K, V, sequence lengths, page tables,
write slots).  It holds none of the method's arithmetic -- no quantisation, no
scores, no softmax -- so that the CUDA path and the CPU oracle can both be fed
from it without sharing any of the computation they are compared on.

Shapes follow the Qwen3-VL models the pages target (article 9-2 header:
Qwen3-VL-8B / Qwen3-VL-2B, hd = 128, kv_bs = 32) and the block-sparse knobs of
article 10-1 §2 (block 32, k 32, probe 8).  The pages measure on private
prompts that are not available; the distributions below stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

HD = 128
KV_BS = 32


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    nq: int
    nkv: int
    seq_lens: np.ndarray          # int32 [B]; includes the token appended this step
    layers: int = 1
    hd: int = HD
    kv_bs: int = KV_BS
    kind: str = "normal"          # normal | sigma | student_t | planted
    seed: int = 0
    block: int = 32               # block-sparse knobs (article 10-1 §2)
    topk: int = 32
    probe: int = 8
    description: str = ""

    @property
    def G(self) -> int:
        return self.nq // self.nkv

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.hd)))

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def max_pages(self) -> int:
        return max(1, -(-self.max_seq_len // self.kv_bs))

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic KV bytes one exact decode call reads: per (token, KV
        head) 128 B of K codes, 128 B of V codes and two fp32 scales."""
        return self.total_tokens * self.nkv * (2 * self.hd + 8)


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed))


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny(seed: int = 1000) -> Workload:
    """1 sequence, 1 layer, 16 query / 8 KV heads, n = 256 (article 9-3 §3
    experiment shape: L = 256, hd = 128, K/V ~ N(0, 1))."""
    return Workload("tiny_n256", 1, 16, 8, np.array([256], np.int32), seed=seed,
                    description="B=1 nq=16 nkv=8 hd=128 n=256 kv_bs=32, q/K/V ~ N(0,1)")


def qwen3vl_2b(n: int, seed: int = 2000) -> Workload:
    """Qwen3-VL-2B decode at batch 1: 28 layers, 16/8 heads, the three
    context lengths of article 10-1 Table B.  Per (layer, KV head) K and V
    have sigma ~ U[0.5, 3] (independent for K and V)."""
    return Workload(f"qwen3vl2b_n{n}", 1, 16, 8, np.array([n], np.int32), layers=28,
                    kind="sigma", seed=seed + n,
                    description=f"B=1 nq=16 nkv=8 hd=128 28 layers n={n}, K,V ~ N(0, s^2) "
                                "s ~ U[0.5,3] per (layer, kv head)")


def serving_8b(B: int = 64, lo: int = 1024, hi: int = 32768, layers: int = 36,
               seed: int = 3000) -> Workload:
    """Qwen3-VL-8B-shaped batched serving decode: 32 query / 8 KV heads,
    36 layers, ragged lengths uniform in [lo, hi], pages in a shared pool in
    random order."""
    lens = _rng(seed).integers(lo, hi + 1, size=B).astype(np.int32)
    return Workload(f"serving8b_B{B}", B, 32, 8, lens, layers=layers, seed=seed,
                    description=f"B={B} nq=32 nkv=8 hd=128 {layers} layers, n ~ U[{lo},{hi}], "
                                "K/V ~ N(0,1), randomly permuted 32-token pages")


def long_context(B: int = 8, n: int = 131072, seed: int = 4000) -> Workload:
    """Long-context stress: K Student-t (nu = 3) with 1 % of the nkv*hd
    channels scaled x20 (fixed over tokens), V ~ N(0, 1)."""
    return Workload(f"long_B{B}_n{n}", B, 16, 8, np.full(B, n, np.int32), kind="student_t",
                    seed=seed,
                    description=f"B={B} nq=16 nkv=8 hd=128 n={n}, K Student-t(3) with 1% "
                                "channels x20, V ~ N(0,1)")


def sparse_planted(n: int, B: int = 16, seed: int = 5000) -> Workload:
    """Block-sparse decode: block 32, k 32, probe 8; K/V ~ N(0, 1) with
    min(32, nblk) planted blocks per (sequence, KV head) whose K rows align
    with the group's queries (cosine 0.8)."""
    return Workload(f"sparse_n{n}", B, 16, 8, np.full(B, n, np.int32), kind="planted",
                    seed=seed + n,
                    description=f"B={B} nq=16 nkv=8 hd=128 n={n} block=32 k=32 probe=8, "
                                "N(0,1) with 32 planted blocks per (seq, kv head)")


def custom(B, nq, nkv, seq_lens, kind="normal", seed=0, kv_bs=KV_BS, block=32, topk=32,
           probe=8, name="custom") -> Workload:
    return Workload(name, B, nq, nkv, np.asarray(seq_lens, np.int32).reshape(B), kind=kind,
                    seed=seed, kv_bs=kv_bs, block=block, topk=topk, probe=probe)


# ---------------------------------------------------------------------------
# Host (numpy) inputs -- oracle-sized cases
# ---------------------------------------------------------------------------

def _layer_seed(wl: Workload, layer: int, what: int, b: int = 0) -> int:
    return ((wl.seed * 1009 + layer) * 7 + what) * 100003 + b


def host_q(wl: Workload, layer: int = 0) -> np.ndarray:
    """q float32 [B, nq, hd] ~ N(0, 1)."""
    return _rng(_layer_seed(wl, layer, 0)).standard_normal((wl.B, wl.nq, wl.hd)).astype(np.float32)


def _outlier_channels(wl: Workload) -> np.ndarray:
    """10 of the nkv*hd channels (1 %), fixed over tokens."""
    n_out = max(1, round(0.01 * wl.nkv * wl.hd))
    return _rng(_layer_seed(wl, 0, 9)).choice(wl.nkv * wl.hd, size=n_out, replace=False)


def _planted_blocks(wl: Workload, b: int, kh: int, n: int) -> np.ndarray:
    nblk = -(-n // wl.block)
    cnt = min(32, nblk)
    return np.sort(_rng(_layer_seed(wl, 0, 11, b * 64 + kh)).choice(nblk, size=cnt, replace=False))


def host_kv(wl: Workload, b: int, layer: int = 0, q: Optional[np.ndarray] = None):
    """fp32 K, V [n_b, nkv, hd] of sequence b (host, numpy)."""
    n = int(wl.seq_lens[b])
    r = _rng(_layer_seed(wl, layer, 1, b))
    shape = (n, wl.nkv, wl.hd)
    if wl.kind in ("normal", "planted", "ties"):
        K = r.standard_normal(shape, dtype=np.float32)
        V = r.standard_normal(shape, dtype=np.float32)
    elif wl.kind == "sigma":
        rs = _rng(_layer_seed(wl, layer, 2))
        sk = rs.uniform(0.5, 3.0, size=wl.nkv).astype(np.float32)
        sv = rs.uniform(0.5, 3.0, size=wl.nkv).astype(np.float32)
        K = r.standard_normal(shape, dtype=np.float32) * sk[None, :, None]
        V = r.standard_normal(shape, dtype=np.float32) * sv[None, :, None]
    elif wl.kind == "student_t":
        z = r.standard_normal(shape, dtype=np.float32)
        chi2 = (r.standard_normal((3,) + shape, dtype=np.float32) ** 2).sum(0)
        K = (z / np.sqrt(chi2 / 3.0)).astype(np.float32)
        ch = _outlier_channels(wl)
        K.reshape(n, wl.nkv * wl.hd)[:, ch] *= np.float32(20.0)
        V = r.standard_normal(shape, dtype=np.float32)
    else:
        raise ValueError(wl.kind)
    if wl.kind == "planted":
        if q is None:
            q = host_q(wl, layer)
        _plant(wl, b, K, q[b], n)
    if wl.kind == "ties":
        if q is None:
            q = host_q(wl, layer)
        _plant_ties(wl, b, K, q[b], n)
    return K.astype(np.float32), V.astype(np.float32)


def _aligned_rows(rr, u: np.ndarray, rows: int, hd: int, cos: float) -> np.ndarray:
    """`rows` vectors sqrt(hd) * (cos u + sin x_perp), x_perp random unit
    vectors orthogonal to the unit vector u."""
    x = rr.standard_normal((rows, hd))
    x -= (x @ u)[:, None] * u[None, :]
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return math.sqrt(hd) * (cos * u[None, :] + math.sqrt(1.0 - cos * cos) * x)


def tie_mode(b: int) -> int:
    """How sequence b of a "ties" workload is built: 0 all-zero K, 1 every
    block a copy of block 0, 2 a few strong blocks plus more copies of one
    block than the top-k has places left."""
    return b % 3


def tie_counts(wl: Workload, n: int):
    """(strong blocks, copied blocks) of a mode-2 sequence of length n: only
    whole blocks are used, and the copies outnumber the places the strong
    blocks leave in the top-k, so equal block scores straddle the k-th place."""
    full = n // wl.block
    strong = min(10, full // 4, wl.topk // 2)
    copies = min(full - strong, wl.topk - strong + 8)
    return strong, copies


def _plant_ties(wl: Workload, b: int, K: np.ndarray, qb: np.ndarray, n: int) -> None:
    """K of a "ties" sequence (tie_mode): equal K rows give equal int8 codes
    and stored maxima, so their block scores are equal on any implementation
    of the method."""
    mode = tie_mode(b)
    if mode == 0:
        K[:] = 0.0
        return
    if mode == 1:
        for t0 in range(wl.block, n, wl.block):
            K[t0:min(n, t0 + wl.block)] = K[:min(n, t0 + wl.block) - t0]
        return
    G = wl.G
    strong, copies = tie_counts(wl, n)
    for kh in range(wl.nkv):
        u = qb[kh * G:(kh + 1) * G].astype(np.float64).sum(0)
        u /= np.linalg.norm(u)
        rr = _rng(_layer_seed(wl, 0, 13, b * 64 + kh))
        chosen = rr.choice(n // wl.block, size=strong + copies, replace=False)
        for j in chosen[:strong]:
            K[j * wl.block:(j + 1) * wl.block, kh] = _aligned_rows(rr, u, wl.block, wl.hd, 0.9)
        src = _aligned_rows(rr, u, wl.block, wl.hd, 0.8).astype(np.float32)
        for j in chosen[strong:]:
            K[j * wl.block:(j + 1) * wl.block, kh] = src


def _plant(wl: Workload, b: int, K: np.ndarray, qb: np.ndarray, n: int) -> None:
    """K rows of the planted blocks := sqrt(hd) * (0.8 u + 0.6 r_perp), u the
    normalised sum of the group's query heads, r_perp a random unit vector
    orthogonal to u (one per row)."""
    G = wl.G
    for kh in range(wl.nkv):
        u = qb[kh * G:(kh + 1) * G].astype(np.float64).sum(0)
        u /= np.linalg.norm(u)
        rr = _rng(_layer_seed(wl, 0, 12, b * 64 + kh))
        blocks = _planted_blocks(wl, b, kh, n)
        rows = np.concatenate([np.arange(j * wl.block, min((j + 1) * wl.block, n))
                               for j in blocks])
        x = rr.standard_normal((rows.size, wl.hd))
        x -= (x @ u)[:, None] * u[None, :]
        x /= np.linalg.norm(x, axis=1, keepdims=True)
        K[rows, kh] = (math.sqrt(wl.hd) * (0.8 * u[None, :] + 0.6 * x)).astype(np.float32)


def planted_blocks(wl: Workload, b: int, kh: int) -> np.ndarray:
    """Block indices planted for (sequence b, KV head kh) (sorted)."""
    return _planted_blocks(wl, b, kh, int(wl.seq_lens[b]))


# ---------------------------------------------------------------------------
# Paged pool bookkeeping
# ---------------------------------------------------------------------------

def page_table(wl: Workload, extra_pages: int = 0, seed: Optional[int] = None):
    """Random page assignment from a shared pool.

    Returns (page_table int32 [B, max_pages] (-1 where unused), num_pages).
    Pages of all sequences are a seeded random permutation of the pool."""
    need = [max(1, -(-int(n) // wl.kv_bs)) if n > 0 else 0 for n in wl.seq_lens]
    total = int(sum(need)) + extra_pages
    perm = _rng(wl.seed * 31 + 7 if seed is None else seed).permutation(max(total, 1)).astype(np.int32)
    pt = np.full((wl.B, wl.max_pages), -1, np.int32)
    o = 0
    for b in range(wl.B):
        pt[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    return pt, max(total, 1)


def slots_for(wl: Workload, pt: np.ndarray, b: int, t0: int, t1: int) -> np.ndarray:
    """Pool slots (page * kv_bs + row) of tokens [t0, t1) of sequence b."""
    t = np.arange(t0, t1)
    return (pt[b, t // wl.kv_bs].astype(np.int64) * wl.kv_bs + t % wl.kv_bs).astype(np.int32)


def all_slots(wl: Workload, pt: np.ndarray) -> np.ndarray:
    """Slots of every token of every sequence, sequences concatenated."""
    if wl.B == 0:
        return np.zeros(0, np.int32)
    return np.concatenate([slots_for(wl, pt, b, 0, int(wl.seq_lens[b])) for b in range(wl.B)])


# ---------------------------------------------------------------------------
# Device (torch) inputs -- full-size cases
# ---------------------------------------------------------------------------

def device_generator(device, seed: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def device_q(wl: Workload, layer: int, device):
    import torch
    g = device_generator(device, _layer_seed(wl, layer, 0))
    return torch.randn((wl.B, wl.nq, wl.hd), generator=g, device=device, dtype=torch.float32)


def device_kv_chunk(wl: Workload, layer: int, b: int, t0: int, t1: int, device, out_k=None,
                    out_v=None):
    """fp32 K, V [t1 - t0, nkv, hd] for tokens [t0, t1) of sequence b drawn
    on the device (same distributions as host_kv; different random stream)."""
    import torch
    n = t1 - t0
    shape = (n, wl.nkv, wl.hd)
    g = device_generator(device, _layer_seed(wl, layer, 5, b) * 4099 + t0)
    K = out_k if out_k is not None else torch.empty(shape, device=device, dtype=torch.float32)
    V = out_v if out_v is not None else torch.empty(shape, device=device, dtype=torch.float32)
    K.normal_(generator=g)
    V.normal_(generator=g)
    if wl.kind == "sigma":
        rs = _rng(_layer_seed(wl, layer, 2))
        sk = torch.tensor(rs.uniform(0.5, 3.0, size=wl.nkv).astype(np.float32), device=device)
        sv = torch.tensor(rs.uniform(0.5, 3.0, size=wl.nkv).astype(np.float32), device=device)
        K.mul_(sk[None, :, None])
        V.mul_(sv[None, :, None])
    elif wl.kind == "student_t":
        chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
        tmp = torch.empty(shape, device=device, dtype=torch.float32)
        for _ in range(3):
            tmp.normal_(generator=g)
            chi2.addcmul_(tmp, tmp)
        K.div_(torch.sqrt(chi2 / 3.0))
        ch = torch.tensor(_outlier_channels(wl), device=device, dtype=torch.long)
        Kf = K.view(n, -1)
        Kf[:, ch] *= 20.0
    elif wl.kind == "planted":
        raise ValueError("planted workloads are drawn on the host")
    return K, V


def describe(wl: Workload) -> dict:
    return {"workload": wl.name, "B": wl.B, "nq": wl.nq, "nkv": wl.nkv, "hd": wl.hd,
            "kv_bs": wl.kv_bs, "layers": wl.layers, "max_seq_len": wl.max_seq_len,
            "mean_seq_len": float(wl.seq_lens.mean()) if wl.B else 0.0,
            "distribution": wl.description}


ALL_NAMES: List[str] = ["tiny", "qwen3vl_2b", "serving_8b", "long_context", "sparse_planted"]
