"""Thin ctypes binding of libkq8 (include/kq8.h), same entry-point names.

Only argument marshalling happens here: tensors become device pointers, the
current torch stream becomes the cudaStream_t.  Every step of the method runs
in the library's CUDA kernels; there is no fallback.  Importing this module
raises ImportError when libkq8.so has not been built.

PyTorch provides device memory and streams: ``PagedKVCache`` allocates the
pool tensors in the layout include/kq8.h documents, and ``Workspace`` holds a
caller-owned scratch buffer.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

if not os.path.exists(_build.LIB):
    raise ImportError(
        f"libkq8.so is not built ({_build.LIB}); run `python -m query_decode_attention_gb300.build`"
        " or __graft_entry__.build() first")

_lib = ctypes.CDLL(_build.LIB)

KQ8_OK = 0
KQ8_ERR_INVALID_ARG = -1
KQ8_ERR_UNSUPPORTED = -2
KQ8_ERR_WORKSPACE = -3
KQ8_ERR_CUDA = -4

KQ8_STATUS_BAD_PAGE = 0x1
KQ8_STATUS_BAD_SEQLEN = 0x2
KQ8_STATUS_BAD_SLOT = 0x4
KQ8_STATUS_TIMEOUT = 0x8

HEAD_DIM = 128


class kq8_cache_t(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("kscale", ctypes.c_void_p),
                ("vscale", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("kv_bs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_CP = ctypes.POINTER(kq8_cache_t)

_lib.kq8_append_kv.argtypes = [_CP, _P, _P, _P, _I32, _P, _P]
_lib.kq8_decode_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
_lib.kq8_decode_workspace_bytes.restype = _SZ
_lib.kq8_sparse_decode_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32]
_lib.kq8_sparse_decode_workspace_bytes.restype = _SZ
_lib.kq8_decode_plan.argtypes = [_I32, _I32, _I32, _I32, ctypes.POINTER(_I32),
                                 ctypes.POINTER(_I32)]
_lib.kq8_sparse_decode_plan.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, ctypes.POINTER(_I32),
                                        ctypes.POINTER(_I32)]
_lib.kq8_workspace_init.argtypes = [_P, _SZ, _P]
_lib.kq8_decode_attn.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float, _P,
                                 _SZ, _P]
_lib.kq8_sparse_decode_attn.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32,
                                        ctypes.c_float, _I32, _I32, _I32, _P, _P, _SZ, _P]
_lib.kq8_decode_attn_noalloc.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32,
                                         ctypes.c_float, _P]
_lib.kq8_state_reset.argtypes = [_P, _P, _I32, _P]
_lib.kq8_decode_attn_update.argtypes = [_P, _P, _P, _CP, _P, _I32, _P, _P, _I32, _I32, _I32,
                                        _I32, ctypes.c_float, _P, _SZ, _P]
_lib.kq8_state_finalize.argtypes = [_P, _P, _P, _I32, _P]
_lib.kq8_state_merge.argtypes = [_P, _P, _P, _P, _I32, _I32, _P]
_lib.kq8_prefill_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32]
_lib.kq8_prefill_workspace_bytes.restype = _SZ
_lib.kq8_prefill_attn.argtypes = [_P, _P, _I32, _CP, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                  ctypes.c_float, _P, _SZ, _P]
_lib.kq8_debug_prefill_withhold.argtypes = [_P, _P, _I32, _CP, _P, _I32, _P, _P, _I32, _I32,
                                            _I32, _I32, ctypes.c_float, _P, _SZ, _I32, _P]
_lib.kq8_debug_decode_withhold.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32,
                                           ctypes.c_float, _P, _SZ, _I32, _P]
_lib.kq8_sparse_prefill_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32]
_lib.kq8_sparse_prefill_workspace_bytes.restype = _SZ
_lib.kq8_sparse_prefill_attn.argtypes = [_P, _P, _I32, _CP, _P, _I32, _P, _P, _I32, _I32, _I32,
                                         _I32, ctypes.c_float, _I32, _I32, _I32, _P, _P, _SZ, _P]
_lib.kq8_append_kv_q4.argtypes = [_CP, _P, _P, _P, _I32, _P, _P]
_lib.kq8_decode_attn_q4.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float,
                                    _P, _SZ, _P]
_lib.kq8_sparse_decode_attn_shared.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32,
                                               ctypes.c_float, _I32, _I32, _I32, _P, _P, _SZ, _P]
_lib.kq8_read_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), _P]
_lib.kq8_strerror.argtypes = [ctypes.c_int]
_lib.kq8_strerror.restype = ctypes.c_char_p
_lib.kq8_version.restype = ctypes.c_int
_lib.kq8_debug_quantize_q.argtypes = [_P, _P, _P, _I32, _I32, _P]
_lib.kq8_debug_block_dots.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32, _P]
_lib.kq8_debug_probe_scores.argtypes = [_P, _P, _CP, _P, _I32, _P, _I32, _I32, _I32,
                                        ctypes.c_float, _I32, _I32, _P]


class Kq8Error(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {kq8_strerror(code)} ({code})" if what else kq8_strerror(code))


def _check(rc: int, what: str) -> None:
    if rc != KQ8_OK:
        raise Kq8Error(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("kq8 takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("kq8 takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype(t: torch.Tensor, dt, name: str) -> None:
    if t.dtype != dt:
        raise TypeError(f"{name} must be {dt}, got {t.dtype}")


def kq8_strerror(code: int) -> str:
    return _lib.kq8_strerror(int(code)).decode()


def kq8_version() -> int:
    return int(_lib.kq8_version())


class PagedKVCache:
    """Device pool of one layer in the kq8_cache_t layout (torch-allocated).

    bits=8: k int8 [num_pages, nkv, kv_bs/32, 4, 32, 32], v int8 [num_pages,
    nkv, kv_bs, 128]; bits=4 (q4 cache, packed nibbles): k [.., 4, 32, 16],
    v [num_pages, nkv, kv_bs, 64]; kscale/vscale: float32 [num_pages, nkv,
    kv_bs]."""

    def __init__(self, num_pages: int, num_kv_heads: int, kv_bs: int = 32, device="cuda",
                 k=None, v=None, kscale=None, vscale=None, bits: int = 8):
        if bits not in (8, 4):
            raise ValueError("bits must be 8 or 4")
        self.num_pages, self.num_kv_heads, self.kv_bs = int(num_pages), int(num_kv_heads), int(kv_bs)
        self.head_dim = HEAD_DIM
        self.bits = bits
        sub = kv_bs // 32
        row = HEAD_DIM if bits == 8 else HEAD_DIM // 2
        self.k = k if k is not None else torch.zeros(
            (num_pages, num_kv_heads, sub, 4, 32, row // 4), dtype=torch.int8, device=device)
        self.v = v if v is not None else torch.zeros(
            (num_pages, num_kv_heads, kv_bs, row), dtype=torch.int8, device=device)
        self.kscale = kscale if kscale is not None else torch.zeros(
            (num_pages, num_kv_heads, kv_bs), dtype=torch.float32, device=device)
        self.vscale = vscale if vscale is not None else torch.zeros(
            (num_pages, num_kv_heads, kv_bs), dtype=torch.float32, device=device)
        self._struct = kq8_cache_t(self.k.data_ptr(), self.v.data_ptr(), self.kscale.data_ptr(),
                                   self.vscale.data_ptr(), self.num_pages, self.kv_bs,
                                   self.num_kv_heads, self.head_dim)

    @property
    def struct(self) -> kq8_cache_t:
        return self._struct

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k, self.v, self.kscale, self.vscale))


def _append_args(cache, k, v, slot, status, bits):
    if cache.bits != bits:
        raise ValueError(f"this call writes a q{bits} cache, got q{cache.bits}")
    _dtype(k, torch.float32, "k")
    _dtype(v, torch.float32, "v")
    _dtype(slot, torch.int32, "slot")
    T = slot.numel()
    if k.numel() != T * cache.num_kv_heads * HEAD_DIM or v.numel() != k.numel():
        raise ValueError("k/v must be [T, nkv, 128] with T = len(slot)")
    if status is not None:
        _dtype(status, torch.int32, "status")
    return T


def kq8_append_kv(cache: PagedKVCache, k: torch.Tensor, v: torch.Tensor, slot: torch.Tensor,
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write path: k, v float32 [T, nkv, 128]; slot int32 [T]."""
    T = _append_args(cache, k, v, slot, status, 8)
    _check(_lib.kq8_append_kv(ctypes.byref(cache.struct), _ptr(k), _ptr(v), _ptr(slot), T,
                              _ptr(status), _stream(stream)), "kq8_append_kv")


def kq8_append_kv_q4(cache: PagedKVCache, k: torch.Tensor, v: torch.Tensor, slot: torch.Tensor,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q4 write path (include/kq8.h) into a PagedKVCache(bits=4)."""
    T = _append_args(cache, k, v, slot, status, 4)
    _check(_lib.kq8_append_kv_q4(ctypes.byref(cache.struct), _ptr(k), _ptr(v), _ptr(slot), T,
                                 _ptr(status), _stream(stream)), "kq8_append_kv_q4")


def kq8_decode_workspace_bytes(B: int, nq: int, nkv: int, max_seq_len: int) -> int:
    return int(_lib.kq8_decode_workspace_bytes(B, nq, nkv, max_seq_len))


def kq8_decode_plan(B: int, nq: int, nkv: int, max_seq_len: int):
    """(chunk_tiles, num_chunks) of the exact decode's KV split."""
    ct, nc = _I32(0), _I32(0)
    _check(_lib.kq8_decode_plan(B, nq, nkv, max_seq_len, ctypes.byref(ct), ctypes.byref(nc)),
           "kq8_decode_plan")
    return int(ct.value), int(nc.value)


def kq8_sparse_decode_plan(B: int, nq: int, nkv: int, max_seq_len: int, block: int, topk: int):
    """(chunk_tiles, num_chunks) of the sparse decode's bounded attention."""
    ct, nc = _I32(0), _I32(0)
    _check(_lib.kq8_sparse_decode_plan(B, nq, nkv, max_seq_len, block, topk, ctypes.byref(ct),
                                       ctypes.byref(nc)), "kq8_sparse_decode_plan")
    return int(ct.value), int(nc.value)


def kq8_sparse_decode_workspace_bytes(B: int, nq: int, nkv: int, max_seq_len: int, block: int,
                                      topk: int) -> int:
    return int(_lib.kq8_sparse_decode_workspace_bytes(B, nq, nkv, max_seq_len, block, topk))


def kq8_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(_lib.kq8_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kq8_workspace_init")


def new_workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A caller-owned workspace (uint8 tensor) with its status word cleared."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    kq8_workspace_init(ws, stream)
    return ws


def _decode_args(out, q, cache, page_table, seq_lens, bits=8):
    if cache.bits != bits:
        raise ValueError(f"this call reads a q{bits} cache, got q{cache.bits}")
    _dtype(out, torch.float32, "out")
    _dtype(q, torch.float32, "q")
    _dtype(page_table, torch.int32, "page_table")
    _dtype(seq_lens, torch.int32, "seq_lens")
    if q.dim() != 3 or q.shape[2] != HEAD_DIM or out.shape != q.shape:
        raise ValueError("q and out must be [B, nq, 128]")
    B, nq = q.shape[0], q.shape[1]
    if page_table.dim() != 2 or page_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("page_table must be [B, max_pages] and seq_lens [B]")
    return B, nq, page_table.shape[1]


def kq8_decode_attn(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                    page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                    scale: float, workspace: torch.Tensor, stream=None) -> None:
    """Exact q8 decode attention (include/kq8.h)."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens)
    _check(_lib.kq8_decode_attn(_ptr(out), _ptr(q), ctypes.byref(cache.struct), _ptr(page_table),
                                max_pages, _ptr(seq_lens), int(max_seq_len), B, nq, float(scale),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)), "kq8_decode_attn")


def kq8_decode_attn_q4(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                       page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                       scale: float, workspace: torch.Tensor, stream=None) -> None:
    """Exact decode over a q4 cache (include/kq8.h)."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens, bits=4)
    _check(_lib.kq8_decode_attn_q4(_ptr(out), _ptr(q), ctypes.byref(cache.struct),
                                   _ptr(page_table), max_pages, _ptr(seq_lens), int(max_seq_len),
                                   B, nq, float(scale), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "kq8_decode_attn_q4")


def kq8_decode_attn_noalloc(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                            page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                            scale: float, stream=None) -> None:
    """kq8_decode_attn without a workspace, for callers that may not allocate
    device memory (the library's fixed scratch array is used instead; calls
    that overlap on the GPU race)."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens)
    _check(_lib.kq8_decode_attn_noalloc(_ptr(out), _ptr(q), ctypes.byref(cache.struct),
                                        _ptr(page_table), max_pages, _ptr(seq_lens),
                                        int(max_seq_len), B, nq, float(scale), _stream(stream)),
           "kq8_decode_attn_noalloc")


def kq8_debug_decode_withhold(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                              page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                              scale: float, workspace: torch.Tensor, withhold_tile: int,
                              stream=None) -> None:
    """Failure-detection hook (include/kq8.h): the exact decode with one tile
    copy of every warp's walk never issued, so its bounded wait runs out."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens)
    _check(_lib.kq8_debug_decode_withhold(_ptr(out), _ptr(q), ctypes.byref(cache.struct),
                                          _ptr(page_table), max_pages, _ptr(seq_lens),
                                          int(max_seq_len), B, nq, float(scale), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          int(withhold_tile), _stream(stream)),
           "kq8_debug_decode_withhold")


def kq8_sparse_decode_attn(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                           page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                           scale: float, block: int, topk: int, probe: int,
                           workspace: torch.Tensor, sel_blocks: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """Block-sparse q8 decode attention (include/kq8.h)."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens)
    if sel_blocks is not None:
        _dtype(sel_blocks, torch.int32, "sel_blocks")
        if sel_blocks.numel() != B * nq * topk:
            raise ValueError("sel_blocks must be [B, nq, topk]")
    _check(_lib.kq8_sparse_decode_attn(_ptr(out), _ptr(q), ctypes.byref(cache.struct),
                                       _ptr(page_table), max_pages, _ptr(seq_lens),
                                       int(max_seq_len), B, nq, float(scale), int(block),
                                       int(topk), int(probe), _ptr(sel_blocks), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "kq8_sparse_decode_attn")


class AttnState:
    """A running attention state for B sequences x nq query heads (the
    streaming form): acc float32 [B, nq, 128], ms float32 [B, nq, 2]."""

    def __init__(self, B: int, nq: int, device="cuda", stream=None):
        self.acc = torch.empty((B, nq, HEAD_DIM), dtype=torch.float32, device=device)
        self.ms = torch.empty((B, nq, 2), dtype=torch.float32, device=device)
        kq8_state_reset(self, stream)


def kq8_state_reset(state: AttnState, stream=None) -> None:
    rows = state.acc.numel() // HEAD_DIM
    _check(_lib.kq8_state_reset(_ptr(state.acc), _ptr(state.ms), rows, _stream(stream)),
           "kq8_state_reset")


def kq8_decode_attn_update(state: AttnState, q: torch.Tensor, cache: PagedKVCache,
                           page_table: torch.Tensor, seq_begin: Optional[torch.Tensor],
                           seq_end: torch.Tensor, max_seq_len: int, scale: float,
                           workspace: torch.Tensor, stream=None, max_range_len: int = 0) -> None:
    """Fold tokens [seq_begin, seq_end) of each sequence into `state`;
    max_range_len bounds seq_end - seq_begin (0: max_seq_len)."""
    B, nq, max_pages = _decode_args(state.acc, q, cache, page_table, seq_end)
    if seq_begin is not None:
        _dtype(seq_begin, torch.int32, "seq_begin")
        if seq_begin.numel() != B:
            raise ValueError("seq_begin must be [B]")
    _check(_lib.kq8_decode_attn_update(_ptr(state.acc), _ptr(state.ms), _ptr(q),
                                       ctypes.byref(cache.struct), _ptr(page_table), max_pages,
                                       _ptr(seq_begin), _ptr(seq_end), int(max_seq_len),
                                       int(max_range_len), B, nq,
                                       float(scale), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "kq8_decode_attn_update")


def kq8_state_finalize(out: torch.Tensor, state: AttnState, stream=None) -> None:
    _dtype(out, torch.float32, "out")
    if out.shape != state.acc.shape:
        raise ValueError("out must match the state's [B, nq, 128]")
    rows = state.acc.numel() // HEAD_DIM
    _check(_lib.kq8_state_finalize(_ptr(out), _ptr(state.acc), _ptr(state.ms), rows,
                                   _stream(stream)), "kq8_state_finalize")


def kq8_state_merge(state: AttnState, part_acc: torch.Tensor, part_ms: torch.Tensor,
                    stream=None) -> None:
    """Fold partial states part_acc [parts, B, nq, 128] / part_ms [parts, B, nq, 2]
    (this library's state format, e.g. other ranks' states) into `state`."""
    _dtype(part_acc, torch.float32, "part_acc")
    _dtype(part_ms, torch.float32, "part_ms")
    if (part_acc.dim() != 4 or part_acc.shape[1:] != state.acc.shape
            or part_ms.shape != (part_acc.shape[0],) + tuple(state.ms.shape)):
        raise ValueError("part_acc must be [parts, B, nq, 128] and part_ms [parts, B, nq, 2]")
    if not (part_acc.is_contiguous() and part_ms.is_contiguous()):
        raise ValueError("partial states must be contiguous")
    rows = state.acc.numel() // HEAD_DIM
    _check(_lib.kq8_state_merge(_ptr(state.acc), _ptr(state.ms), _ptr(part_acc), _ptr(part_ms),
                                part_acc.shape[0], rows, _stream(stream)), "kq8_state_merge")


def kq8_prefill_workspace_bytes(B: int, nq: int, nkv: int, max_seq_len: int,
                                max_q_len: int) -> int:
    return int(_lib.kq8_prefill_workspace_bytes(B, nq, nkv, max_seq_len, max_q_len))


def kq8_prefill_attn(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                     page_table: torch.Tensor, seq_lens: torch.Tensor, q_offsets: torch.Tensor,
                     max_seq_len: int, max_q_len: int, scale: float, workspace: torch.Tensor,
                     stream=None) -> None:
    """Batched causal prefill attention (include/kq8.h): q and out are
    [total_q, nq, 128], packed by sequence per q_offsets [B+1]; seq_lens
    counts each sequence's cached tokens including its new ones."""
    if cache.bits != 8:
        raise ValueError("prefill reads a q8 cache")
    _dtype(out, torch.float32, "out")
    _dtype(q, torch.float32, "q")
    _dtype(page_table, torch.int32, "page_table")
    _dtype(seq_lens, torch.int32, "seq_lens")
    _dtype(q_offsets, torch.int32, "q_offsets")
    if q.dim() != 3 or q.shape[2] != HEAD_DIM or out.shape != q.shape:
        raise ValueError("q and out must be [total_q, nq, 128]")
    B = seq_lens.numel()
    if q_offsets.numel() != B + 1 or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("q_offsets must be [B+1] and page_table [B, max_pages]")
    _check(_lib.kq8_prefill_attn(_ptr(out), _ptr(q), q.shape[0], ctypes.byref(cache.struct),
                                 _ptr(page_table), page_table.shape[1], _ptr(seq_lens),
                                 _ptr(q_offsets), int(max_seq_len), int(max_q_len), B, q.shape[1],
                                 float(scale), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "kq8_prefill_attn")


def kq8_debug_prefill_withhold(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                               page_table: torch.Tensor, seq_lens: torch.Tensor,
                               q_offsets: torch.Tensor, max_seq_len: int, max_q_len: int,
                               scale: float, workspace: torch.Tensor, withhold_sub: int,
                               stream=None) -> None:
    """Failure-detection hook (include/kq8.h): the prefill with one raw
    sub-tile's copy never issued, so its bounded wait runs out."""
    if cache.bits != 8:
        raise ValueError("prefill reads a q8 cache")
    B = seq_lens.numel()
    _check(_lib.kq8_debug_prefill_withhold(_ptr(out), _ptr(q), q.shape[0],
                                           ctypes.byref(cache.struct), _ptr(page_table),
                                           page_table.shape[1], _ptr(seq_lens), _ptr(q_offsets),
                                           int(max_seq_len), int(max_q_len), B, q.shape[1],
                                           float(scale), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           int(withhold_sub), _stream(stream)),
           "kq8_debug_prefill_withhold")


def kq8_sparse_decode_attn_shared(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                                  page_table: torch.Tensor, seq_lens: torch.Tensor,
                                  max_seq_len: int, scale: float, block: int, topk: int,
                                  probe: int, workspace: torch.Tensor,
                                  sel_blocks: Optional[torch.Tensor] = None, stream=None) -> None:
    """Block-sparse decode with one selection per KV head (include/kq8.h)."""
    B, nq, max_pages = _decode_args(out, q, cache, page_table, seq_lens)
    if sel_blocks is not None:
        _dtype(sel_blocks, torch.int32, "sel_blocks")
        if sel_blocks.numel() != B * nq * topk:
            raise ValueError("sel_blocks must be [B, nq, topk]")
    _check(_lib.kq8_sparse_decode_attn_shared(_ptr(out), _ptr(q), ctypes.byref(cache.struct),
                                              _ptr(page_table), max_pages, _ptr(seq_lens),
                                              int(max_seq_len), B, nq, float(scale), int(block),
                                              int(topk), int(probe), _ptr(sel_blocks),
                                              _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream)), "kq8_sparse_decode_attn_shared")


def kq8_sparse_prefill_workspace_bytes(total_q: int, nq: int, nkv: int, max_seq_len: int,
                                       block: int, topk: int) -> int:
    return int(_lib.kq8_sparse_prefill_workspace_bytes(total_q, nq, nkv, max_seq_len, block, topk))


def kq8_sparse_prefill_attn(out: torch.Tensor, q: torch.Tensor, cache: PagedKVCache,
                            page_table: torch.Tensor, seq_lens: torch.Tensor,
                            q_offsets: torch.Tensor, max_seq_len: int, max_q_len: int,
                            scale: float, block: int, topk: int, probe: int,
                            workspace: torch.Tensor, sel_blocks: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """Block-sparse batched prefill (include/kq8.h); arguments as
    kq8_prefill_attn plus the block-sparse knobs of kq8_sparse_decode_attn."""
    if cache.bits != 8:
        raise ValueError("sparse prefill reads a q8 cache")
    _dtype(out, torch.float32, "out")
    _dtype(q, torch.float32, "q")
    _dtype(page_table, torch.int32, "page_table")
    _dtype(seq_lens, torch.int32, "seq_lens")
    _dtype(q_offsets, torch.int32, "q_offsets")
    if q.dim() != 3 or q.shape[2] != HEAD_DIM or out.shape != q.shape:
        raise ValueError("q and out must be [total_q, nq, 128]")
    B = seq_lens.numel()
    if q_offsets.numel() != B + 1 or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("q_offsets must be [B+1] and page_table [B, max_pages]")
    if sel_blocks is not None:
        _dtype(sel_blocks, torch.int32, "sel_blocks")
        if sel_blocks.numel() != q.shape[0] * q.shape[1] * topk:
            raise ValueError("sel_blocks must be [total_q, nq, topk]")
    _check(_lib.kq8_sparse_prefill_attn(_ptr(out), _ptr(q), q.shape[0], ctypes.byref(cache.struct),
                                        _ptr(page_table), page_table.shape[1], _ptr(seq_lens),
                                        _ptr(q_offsets), int(max_seq_len), int(max_q_len), B,
                                        q.shape[1], float(scale), int(block), int(topk),
                                        int(probe), _ptr(sel_blocks), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "kq8_sparse_prefill_attn")


def kq8_read_status(word: torch.Tensor, stream=None) -> int:
    """Fetch and clear a status word (the workspace's first word, or an
    append status tensor).  Synchronises the stream."""
    st = ctypes.c_uint32(0)
    _check(_lib.kq8_read_status(_ptr(word), ctypes.byref(st), _stream(stream)), "kq8_read_status")
    return int(st.value)


# ---- test-only exports -------------------------------------------------------

def kq8_debug_quantize_q(q: torch.Tensor, stream=None):
    """q float32 [..., 128] -> (qi int8 [..., 128], qsc float32 [..., 4])."""
    _dtype(q, torch.float32, "q")
    rows = q.numel() // HEAD_DIM
    qi = torch.empty(q.shape, dtype=torch.int8, device=q.device)
    qsc = torch.empty(q.shape[:-1] + (HEAD_DIM // 32,), dtype=torch.float32, device=q.device)
    _check(_lib.kq8_debug_quantize_q(_ptr(qi), _ptr(qsc), _ptr(q), rows, HEAD_DIM, _stream(stream)),
           "kq8_debug_quantize_q")
    return qi, qsc


def kq8_debug_block_dots(q, cache, page_table, seq_lens, max_seq_len, stream=None):
    B, nq, max_pages = _decode_args(torch.empty_like(q), q, cache, page_table, seq_lens)
    dots = torch.zeros((B, nq, max(1, max_seq_len), HEAD_DIM // 32), dtype=torch.int32,
                       device=q.device)
    _check(_lib.kq8_debug_block_dots(_ptr(dots), _ptr(q), ctypes.byref(cache.struct),
                                     _ptr(page_table), max_pages, _ptr(seq_lens), int(max_seq_len),
                                     B, nq, _stream(stream)), "kq8_debug_block_dots")
    return dots


def kq8_debug_probe_scores(q, cache, page_table, seq_lens, max_seq_len, scale, block, probe,
                           stream=None):
    B, nq, max_pages = _decode_args(torch.empty_like(q), q, cache, page_table, seq_lens)
    nblk = max(1, -(-int(max_seq_len) // int(block)))
    scores = torch.full((B, nq, nblk), float("nan"), dtype=torch.float32, device=q.device)
    _check(_lib.kq8_debug_probe_scores(_ptr(scores), _ptr(q), ctypes.byref(cache.struct),
                                       _ptr(page_table), max_pages, _ptr(seq_lens),
                                       int(max_seq_len), B, nq, float(scale), int(block),
                                       int(probe), _stream(stream)), "kq8_debug_probe_scores")
    return scores
