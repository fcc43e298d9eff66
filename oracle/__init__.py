"""Plain CPU oracle for q8-KV single-query decode attention.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The CUDA product never imports this package, and this package never
imports the product.

The arithmetic lives in ``kq8_oracle.c`` (plain C99, fp32 exactly as the pages
write it, compiled with ``-ffp-contract=off``; fp64 brute-force references
beside it).  This module only compiles it with gcc and marshals numpy arrays.

Cache layout seen by the oracle is the pages' own (article 9-2,
flash_attn_single_q_q8_neon, §2 signature and segment 2): per sequence a list
of blocks of ``kv_bs`` token rows, each row ``nkv*hd`` int8 codes (token-major,
head ``kh`` at column ``kh*hd``), and per-(token, head) float scales laid out
``[token][nkv]`` holding the row's max |x|.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kq8_oracle.c")
_HDR = os.path.join(_HERE, "kq8_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkq8_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_D = ctypes.c_double
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkq8_oracle.so`` (gcc, -O2,
    no FMA contraction; OpenMP when the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    base = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-Wall", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.kq8o_kv_quantize_row.argtypes = [_P, _I, _P, _P]
            L.kq8o_kv_quantize_rows.argtypes = [_P, _I64, _I, _I, _P, _P]
            L.kq8o_dequant.argtypes = [ctypes.c_int8, _F]
            L.kq8o_dequant.restype = _F
            L.kq8o_quantize_q.argtypes = [_P, _I, _P, _P]
            L.kq8o_block_dots.argtypes = [_P, _P, _I, _P]
            L.kq8o_score.argtypes = [_P, _P, _I, _F, _F]
            L.kq8o_score.restype = _F
            L.kq8o_attn_single_q.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                                             _P, _I, _P, _P]
            L.kq8o_stream_reset.argtypes = [_P, _P, _P, _I]
            L.kq8o_attn_stream.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                           _I, _F]
            L.kq8o_stream_output.argtypes = [_P, _F, _P, _I]
            L.kq8o_attn_two_pass_f64.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                 _F, _P, _I]
            L.kq8o_attn_ref_f64.argtypes = [_P, _P, _P, _P, _I, _I, _D]
            L.kq8o_attn_exact_sum.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F]
            L.kq8o_probe_block_scores.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                                                  _I]
            L.kq8o_topk_blocks.argtypes = [_P, _P, _I, _I]
            L.kq8o_topk_blocks.restype = _I
            L.kq8o_sparse_attn_head.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                _F, _I, _I, _I, _P]
            L.kq8o_sparse_attn_head.restype = _I
            L.kq8o_decode_batch.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                            _F, _I, _I, _I, _I, _P, _I]
            L.kq8o_decode_batch.restype = _I
            L.kq8o_prefill_batch.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                             _I, _F, _I, _I, _I, _I, _P, _I]
            L.kq8o_prefill_batch.restype = _I
            L.kq8o_kv_quantize_rows_q4.argtypes = [_P, _I64, _I, _I, _P, _P]
            L.kq8o_attn_single_q_q4.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                _F]
            L.kq8o_decode_batch_q4.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                               _I, _F, _I]
            L.kq8o_decode_batch_q4.restype = _I
            L.kq8o_sparse_attn_group.argtypes = [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                                 _I, _F, _I, _I, _I, _P]
            L.kq8o_sparse_attn_group.restype = _I
            L.kq8o_decode_batch_shared.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                                   _I, _I, _F, _I, _I, _I, _P, _I]
            L.kq8o_decode_batch_shared.restype = _I
            L.kq8o_has_openmp.restype = _I
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(_P)


# --------------------------------------------------------------------------
# Write path and quantisers
# --------------------------------------------------------------------------

def kv_quantize_rows(x):
    """Write path (article 9-3, §2): x[..., hd] float32 -> (codes int8
    [..., hd], stored max float32 [...]) per row."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hd = x.shape[-1]
    rows = x.reshape(-1, hd)
    codes = np.empty(rows.shape, np.int8)
    maxima = np.empty(rows.shape[0], np.float32)
    lib().kq8o_kv_quantize_rows(rows.ctypes.data_as(_P), rows.shape[0], 1, hd,
                                codes.ctypes.data_as(_P), maxima.ctypes.data_as(_P))
    return codes.reshape(x.shape), maxima.reshape(x.shape[:-1])


def kv_quantize_rows_q4(x):
    """q4 write path (the q8 rule with 7 for 127; the pages name --kv-q4 but
    give no format): x[..., hd] float32 -> (codes int8 in [-7, 7] [..., hd],
    stored max float32 [...])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hd = x.shape[-1]
    rows = x.reshape(-1, hd)
    codes = np.empty(rows.shape, np.int8)
    maxima = np.empty(rows.shape[0], np.float32)
    lib().kq8o_kv_quantize_rows_q4(rows.ctypes.data_as(_P), rows.shape[0], 1, hd,
                                   codes.ctypes.data_as(_P), maxima.ctypes.data_as(_P))
    return codes.reshape(x.shape), maxima.reshape(x.shape[:-1])


def dequant(codes, maxima):
    """q * (stored_max * (1/127)) element by element (article 9-3, §2)."""
    codes = np.asarray(codes, np.int8)
    maxima = np.asarray(maxima, np.float32)
    out = np.empty(codes.shape, np.float32)
    L = lib()
    flat_c = codes.reshape(-1, codes.shape[-1])
    flat_m = maxima.reshape(-1)
    flat_o = out.reshape(-1, codes.shape[-1])
    for r in range(flat_c.shape[0]):
        m = float(flat_m[r])
        for i in range(flat_c.shape[1]):
            flat_o[r, i] = L.kq8o_dequant(int(flat_c[r, i]), m)
    return out


def quantize_q(q):
    """Q quantisation (article 9-2, §2 segment 1): q[..., hd] -> (qi int8
    [..., hd], qsc float32 [..., hd/32])."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    hd = q.shape[-1]
    rows = q.reshape(-1, hd)
    qi = np.empty(rows.shape, np.int8)
    qsc = np.empty((rows.shape[0], hd // 32), np.float32)
    L = lib()
    for r in range(rows.shape[0]):
        L.kq8o_quantize_q(rows[r].ctypes.data_as(_P), hd, qi[r].ctypes.data_as(_P),
                          qsc[r].ctypes.data_as(_P))
    return qi.reshape(q.shape), qsc.reshape(q.shape[:-1] + (hd // 32,))


def block_dots(qi, krow):
    qi, pq = _c(qi, np.int8)
    krow, pk = _c(krow, np.int8)
    out = np.empty(qi.shape[-1] // 32, np.int32)
    lib().kq8o_block_dots(pq, pk, qi.shape[-1], out.ctypes.data_as(_P))
    return out


def score(dots, qsc, kscale_stored, scale):
    dots, pd = _c(dots, np.int32)
    qsc, pq = _c(qsc, np.float32)
    return np.float32(lib().kq8o_score(pd, pq, dots.shape[0], float(np.float32(kscale_stored)),
                                       float(np.float32(scale))))


# --------------------------------------------------------------------------
# One query head over one sequence in the pages' blocked layout
# --------------------------------------------------------------------------

class SeqCache:
    """One sequence's quantised cache of one layer in the pages' layout.

    k8, v8: int8 [n, nkv, hd] token rows; ks, vs: float32 [n, nkv] stored
    maxima.  ``blocks`` splits the rows into kv_bs-token blocks; when
    ``shuffle_seed`` is given the blocks are copied to a pool in a random
    order and reached through the block-pointer array, as on article 9-2 §2.
    """

    def __init__(self, k8, ks, v8, vs, kv_bs=32, shuffle_seed=None):
        self.n, self.nkv, self.hd = k8.shape
        self.kv_bs = kv_bs
        self.kv_dim = self.nkv * self.hd
        nb = max(1, -(-self.n // kv_bs))
        pad = nb * kv_bs - self.n
        k = np.concatenate([k8.reshape(self.n, self.kv_dim), np.zeros((pad, self.kv_dim), np.int8)])
        v = np.concatenate([v8.reshape(self.n, self.kv_dim), np.zeros((pad, self.kv_dim), np.int8)])
        kb = k.reshape(nb, kv_bs, self.kv_dim)
        vb = v.reshape(nb, kv_bs, self.kv_dim)
        order = np.arange(nb)
        if shuffle_seed is not None:
            order = np.random.default_rng(shuffle_seed).permutation(nb)
        # pool slot order[j] holds block j
        self.k_pool = np.empty_like(kb)
        self.v_pool = np.empty_like(vb)
        self.k_pool[order] = kb
        self.v_pool[order] = vb
        stride = kv_bs * self.kv_dim
        kbase = self.k_pool.ctypes.data
        vbase = self.v_pool.ctypes.data
        self.k_ptrs = (ctypes.c_void_p * nb)(*[kbase + int(order[j]) * stride for j in range(nb)])
        self.v_ptrs = (ctypes.c_void_p * nb)(*[vbase + int(order[j]) * stride for j in range(nb)])
        self.ks = np.ascontiguousarray(ks, np.float32).reshape(self.n, self.nkv)
        self.vs = np.ascontiguousarray(vs, np.float32).reshape(self.n, self.nkv)
        if self.n == 0:
            self.ks = np.zeros((1, self.nkv), np.float32)
            self.vs = np.zeros((1, self.nkv), np.float32)

    def scale_ptrs(self, kh):
        off = kh * 4
        return (ctypes.c_void_p(self.ks.ctypes.data + off), ctypes.c_void_p(self.vs.ctypes.data + off))


def attn_single_q(q, cache: SeqCache, kh, scale, tokens=None, trace=False):
    """One-pass q8 attention of one query head (article 9-2, §1-§2).
    Returns out float32 [hd] (and (m_trace, n_visited) when trace)."""
    q, pq = _c(q, np.float32)
    out = np.empty(cache.hd, np.float32)
    kp, vp = cache.scale_ptrs(kh)
    if tokens is not None:
        tokens, pt = _c(tokens, np.int32)
        nt = tokens.shape[0]
    else:
        pt, nt = None, 0
    n_list = nt if tokens is not None else cache.n
    mtr = np.empty(max(1, n_list), np.float32) if trace else None
    nv = ctypes.c_int(0)
    lib().kq8o_attn_single_q(out.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs, kp, vp,
                             cache.n, cache.kv_dim, cache.kv_bs, cache.nkv, kh * cache.hd,
                             cache.hd, float(np.float32(scale)), pt, nt,
                             mtr.ctypes.data_as(_P) if trace else None, ctypes.byref(nv))
    if trace:
        return out, mtr[:n_list], nv.value
    return out


class StreamState:
    """Running one-pass state (M, S, acc[hd]) of one query head, kept between
    calls (article 9-2 §3, streaming form)."""

    def __init__(self, hd=128):
        self.M = np.zeros(1, np.float32)
        self.S = np.zeros(1, np.float32)
        self.acc = np.zeros(hd, np.float32)
        lib().kq8o_stream_reset(self.M.ctypes.data_as(_P), self.S.ctypes.data_as(_P),
                                self.acc.ctypes.data_as(_P), hd)

    def output(self):
        out = np.empty_like(self.acc)
        lib().kq8o_stream_output(out.ctypes.data_as(_P), float(self.S[0]),
                                 self.acc.ctypes.data_as(_P), self.acc.shape[0])
        return out


def attn_stream(state: StreamState, q, cache: SeqCache, kh, scale, t_begin, t_end):
    """Continue the one-pass loop of `state` over tokens [t_begin, t_end)."""
    q, pq = _c(q, np.float32)
    kp, vp = cache.scale_ptrs(kh)
    lib().kq8o_attn_stream(state.M.ctypes.data_as(_P), state.S.ctypes.data_as(_P),
                           state.acc.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs, kp, vp,
                           int(t_begin), int(t_end), cache.kv_dim, cache.kv_bs, cache.nkv,
                           kh * cache.hd, cache.hd, float(np.float32(scale)))
    return state


def attn_two_pass_f64(q, cache: SeqCache, kh, scale, tokens=None):
    """Two-pass brute force in fp64 over the same codes (article 9-2, §3)."""
    q, pq = _c(q, np.float32)
    out = np.empty(cache.hd, np.float64)
    kp, vp = cache.scale_ptrs(kh)
    if tokens is not None:
        tokens, pt = _c(tokens, np.int32)
        nt = tokens.shape[0]
    else:
        pt, nt = None, 0
    lib().kq8o_attn_two_pass_f64(out.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs, kp, vp,
                                 cache.n, cache.kv_dim, cache.kv_bs, cache.nkv, kh * cache.hd,
                                 cache.hd, float(np.float32(scale)), pt, nt)
    return out


def attn_exact_sum(q, cache: SeqCache, kh, scale):
    """The method's result with exact sums (article 9-2 §3: one pass and two
    passes are the same computation): the method's fp32 scores and V steps,
    then the softmax and the weighted V sum in fp64, two passes.  The value the
    fp32 one-pass loop (attn_single_q) approximates; over very long sequences
    that loop's own rounding can exceed the output tolerance."""
    q, pq = _c(q, np.float32)
    out = np.empty(cache.hd, np.float64)
    kp, vp = cache.scale_ptrs(kh)
    lib().kq8o_attn_exact_sum(out.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs, kp, vp,
                              cache.n, cache.kv_dim, cache.kv_bs, cache.nkv, kh * cache.hd,
                              cache.hd, float(np.float32(scale)))
    return out


def attn_ref_f64(q, K, V, scale):
    """Standard attention on float K/V [n, hd] in fp64 (article 9-3, §1)."""
    q, pq = _c(q, np.float32)
    K, pk = _c(K, np.float32)
    V, pv = _c(V, np.float32)
    out = np.empty(q.shape[-1], np.float64)
    lib().kq8o_attn_ref_f64(out.ctypes.data_as(_P), pq, pk, pv, K.shape[0], q.shape[-1],
                            float(scale))
    return out


def probe_block_scores(q, cache: SeqCache, kh, scale, block, probe):
    q, pq = _c(q, np.float32)
    nb = -(-cache.n // block)
    out = np.empty(max(nb, 1), np.float32)
    kp, _ = cache.scale_ptrs(kh)
    lib().kq8o_probe_block_scores(out.ctypes.data_as(_P), pq, cache.k_ptrs, kp, cache.n,
                                  cache.kv_dim, cache.kv_bs, cache.nkv, kh * cache.hd, cache.hd,
                                  float(np.float32(scale)), block, probe)
    return out[:nb]


def topk_blocks(scores, k):
    scores, ps = _c(scores, np.float32)
    sel = np.empty(max(1, min(k, scores.shape[0])), np.int32)
    m = lib().kq8o_topk_blocks(sel.ctypes.data_as(_P), ps, scores.shape[0], k)
    return sel[:m]


def sparse_attn_head(q, cache: SeqCache, kh, scale, block, topk, probe):
    """Block-sparse one-head kernel (article 10-1, §1-§2, with the readings in
    kq8_oracle.c).  Returns (out [hd], sel [topk] -1 padded, used_sparse)."""
    q, pq = _c(q, np.float32)
    out = np.empty(cache.hd, np.float32)
    sel = np.empty(max(1, topk), np.int32)
    kp, vp = cache.scale_ptrs(kh)
    used = lib().kq8o_sparse_attn_head(out.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs,
                                       kp, vp, cache.n, cache.kv_dim, cache.kv_bs, cache.nkv,
                                       kh * cache.hd, cache.hd, float(np.float32(scale)), block,
                                       topk, probe, sel.ctypes.data_as(_P))
    return out, sel[:topk], bool(used)


# --------------------------------------------------------------------------
# Batch driver (OpenMP over (sequence, query head) when available)
# --------------------------------------------------------------------------

def attn_single_q_q4(q, cache: SeqCache, kh, scale):
    """One-pass attention of one query head over a q4 cache (codes in [-7, 7])."""
    q, pq = _c(q, np.float32)
    out = np.empty(cache.hd, np.float32)
    kp, vp = cache.scale_ptrs(kh)
    lib().kq8o_attn_single_q_q4(out.ctypes.data_as(_P), pq, cache.k_ptrs, cache.v_ptrs, kp, vp,
                                cache.n, cache.kv_dim, cache.kv_bs, cache.nkv, kh * cache.hd,
                                cache.hd, float(np.float32(scale)))
    return out


def _pack_layer(k8_list, ks_list, v8_list, vs_list, hd, kv_bs):
    """One layer's sequences as the token-major rows the C drivers walk."""
    B = len(k8_list)
    nkv = k8_list[0].shape[1] if B else 1
    lens = np.array([k.shape[0] for k in k8_list], np.int32)
    offs = np.zeros(B, np.int64)
    offs[1:] = np.cumsum(lens.astype(np.int64))[:-1]
    total = int(lens.astype(np.int64).sum())
    pad_rows = kv_bs  # last block pointer of the last sequence stays in range
    k_rows = np.zeros((total + pad_rows, nkv * hd), np.int8)
    v_rows = np.zeros((total + pad_rows, nkv * hd), np.int8)
    ks = np.zeros((total + pad_rows, nkv), np.float32)
    vs = np.zeros((total + pad_rows, nkv), np.float32)
    for b in range(B):
        o, n = int(offs[b]), int(lens[b])
        k_rows[o:o + n] = k8_list[b].reshape(n, nkv * hd)
        v_rows[o:o + n] = v8_list[b].reshape(n, nkv * hd)
        ks[o:o + n] = ks_list[b]
        vs[o:o + n] = vs_list[b]
    return k_rows, v_rows, ks, vs, offs, lens, nkv


def decode_batch(q, k8_list, ks_list, v8_list, vs_list, scale, kv_bs=32, sparse=False, block=32,
                 topk=32, probe=8, nthreads=0):
    """Exact (or block-sparse) decode for B sequences of one layer.

    q: float32 [B, nq, hd]; k8_list[b]: int8 [n_b, nkv, hd]; ks_list[b]:
    float32 [n_b, nkv] (same for V).  Returns out float32 [B, nq, hd] and,
    for sparse, sel int32 [B, nq, topk] (-1 padded)."""
    q = np.ascontiguousarray(q, np.float32)
    B, nq, hd = q.shape
    k_rows, v_rows, ks, vs, offs, lens, nkv = _pack_layer(k8_list, ks_list, v8_list, vs_list, hd,
                                                          kv_bs)
    out = np.empty((B, nq, hd), np.float32)
    sel = np.full((B, nq, max(1, topk)), -1, np.int32) if sparse else None
    rc = lib().kq8o_decode_batch(out.ctypes.data_as(_P), q.ctypes.data_as(_P),
                                 k_rows.ctypes.data_as(_P), v_rows.ctypes.data_as(_P),
                                 ks.ctypes.data_as(_P), vs.ctypes.data_as(_P),
                                 offs.ctypes.data_as(_P), lens.ctypes.data_as(_P), B, nq, nkv, hd,
                                 kv_bs, float(np.float32(scale)), int(sparse), block, topk, probe,
                                 sel.ctypes.data_as(_P) if sparse else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle: unsupported shape")
    return (out, sel[:, :, :topk]) if sparse else out


def sparse_attn_group(q, cache: SeqCache, kh, scale, block, topk, probe):
    """One selection for the G query heads q [G, hd] of KV head kh (the max
    of their block scores); returns (out [G, hd], sel [topk], used)."""
    q, pq = _c(q, np.float32)
    G = q.shape[0]
    out = np.empty((G, cache.hd), np.float32)
    sel = np.full(max(1, topk), -1, np.int32)
    kp, vp = cache.scale_ptrs(kh)
    used = lib().kq8o_sparse_attn_group(out.ctypes.data_as(_P), pq, G, cache.k_ptrs, cache.v_ptrs,
                                        kp, vp, cache.n, cache.kv_dim, cache.kv_bs, cache.nkv,
                                        kh * cache.hd, cache.hd, float(np.float32(scale)), block,
                                        topk, probe, sel.ctypes.data_as(_P))
    return out, sel[:topk], bool(used)


def decode_batch_shared(q, k8_list, ks_list, v8_list, vs_list, scale, kv_bs=32, block=32,
                        topk=32, probe=8, nthreads=0):
    """Block-sparse decode with one selection per KV head; returns (out
    [B, nq, hd], sel [B, nq, topk])."""
    q = np.ascontiguousarray(q, np.float32)
    B, nq, hd = q.shape
    k_rows, v_rows, ks, vs, offs, lens, nkv = _pack_layer(k8_list, ks_list, v8_list, vs_list, hd,
                                                          kv_bs)
    out = np.empty((B, nq, hd), np.float32)
    sel = np.full((B, nq, max(1, topk)), -1, np.int32)
    rc = lib().kq8o_decode_batch_shared(out.ctypes.data_as(_P), q.ctypes.data_as(_P),
                                        k_rows.ctypes.data_as(_P), v_rows.ctypes.data_as(_P),
                                        ks.ctypes.data_as(_P), vs.ctypes.data_as(_P),
                                        offs.ctypes.data_as(_P), lens.ctypes.data_as(_P), B, nq,
                                        nkv, hd, kv_bs, float(np.float32(scale)), block, topk,
                                        probe, sel.ctypes.data_as(_P), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: unsupported shape")
    return out, sel[:, :, :topk]


def decode_batch_q4(q, k4_list, ks_list, v4_list, vs_list, scale, kv_bs=32, nthreads=0):
    """Exact decode over q4 caches (codes int8 in [-7, 7]); as decode_batch."""
    q = np.ascontiguousarray(q, np.float32)
    B, nq, hd = q.shape
    k_rows, v_rows, ks, vs, offs, lens, nkv = _pack_layer(k4_list, ks_list, v4_list, vs_list, hd,
                                                          kv_bs)
    out = np.empty((B, nq, hd), np.float32)
    rc = lib().kq8o_decode_batch_q4(out.ctypes.data_as(_P), q.ctypes.data_as(_P),
                                    k_rows.ctypes.data_as(_P), v_rows.ctypes.data_as(_P),
                                    ks.ctypes.data_as(_P), vs.ctypes.data_as(_P),
                                    offs.ctypes.data_as(_P), lens.ctypes.data_as(_P), B, nq, nkv,
                                    hd, kv_bs, float(np.float32(scale)), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: unsupported shape")
    return out


def prefill_batch(q, q_lens, k8_list, ks_list, v8_list, vs_list, scale, kv_bs=32, sparse=False,
                  block=32, topk=32, probe=8, nthreads=0):
    """Batched causal prefill for B sequences of one layer (see kq8o_prefill_batch).

    q: float32 [total_q, nq, hd], packed by sequence; q_lens[b] = nb_b new
    tokens of sequence b, the last nb_b of its cache (k8_list[b] etc. as in
    decode_batch).  Returns out float32 [total_q, nq, hd] and, for sparse,
    sel int32 [total_q, nq, topk] (-1 padded)."""
    q = np.ascontiguousarray(q, np.float32)
    T, nq, hd = q.shape
    q_off = np.zeros(len(k8_list) + 1, np.int32)
    q_off[1:] = np.cumsum(np.asarray(q_lens, np.int64))
    assert int(q_off[-1]) == T
    k_rows, v_rows, ks, vs, offs, lens, nkv = _pack_layer(k8_list, ks_list, v8_list, vs_list, hd,
                                                          kv_bs)
    out = np.empty((T, nq, hd), np.float32)
    sel = np.full((T, nq, max(1, topk)), -1, np.int32) if sparse else None
    rc = lib().kq8o_prefill_batch(out.ctypes.data_as(_P), q.ctypes.data_as(_P),
                                  k_rows.ctypes.data_as(_P), v_rows.ctypes.data_as(_P),
                                  ks.ctypes.data_as(_P), vs.ctypes.data_as(_P),
                                  offs.ctypes.data_as(_P), lens.ctypes.data_as(_P),
                                  q_off.ctypes.data_as(_P), len(k8_list), nq, nkv, hd, kv_bs,
                                  float(np.float32(scale)), int(sparse), block, topk, probe,
                                  sel.ctypes.data_as(_P) if sparse else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle: unsupported shape or q_lens")
    return (out, sel[:, :, :topk]) if sparse else out


def openmp_threads() -> int:
    """Threads the batch driver may use (0: built without OpenMP)."""
    return int(lib().kq8o_has_openmp())
