"""The bench's byte and rate arithmetic, checked on hand-counted cases (CPU)."""
import importlib.util
import os
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

TILE_BYTES = 32 * 2 * 128 + 2 * 32 * 4  # K and V codes of 32 tokens + their maxima


def test_sparse_call_bytes_hand_counted():
    # B = 2, 2 KV heads x 2 query heads, block 64, probe 8 (stride 8), hd 128.
    # Sequence 0 (100 tokens <= 2 * 64) is gated: all of its 4 tiles, both heads.
    # Sequence 1 (300 tokens, 5 blocks): blocks 0-3 have 8 probe rows, block 4
    # (tokens 256..299) has 6 (256, 264, ..., 296); KV head 0 keeps blocks
    # {0, 2} u {2, 4} = 2 + 2 + 2 tiles (block 4 holds 44 tokens: 2 tiles), KV
    # head 1 keeps {1} = 2 tiles.
    wl = SimpleNamespace(B=2, seq_lens=np.array([100, 300]), block=64, probe=8, nkv=2, hd=128,
                         G=2)
    sel = -np.ones((2, 4, 3), np.int32)
    sel[1, 0, :2] = [0, 2]
    sel[1, 1, :2] = [2, 4]
    sel[1, 2, :1] = [1]
    want = (4 * 2 * TILE_BYTES            # gated sequence
            + 38 * 2 * (128 + 4)          # probe rows: K row + its maximum
            + (6 + 2) * TILE_BYTES)       # kept tiles of the two KV heads
    assert TILE_BYTES == 8448
    assert bench.sparse_call_bytes(wl, sel) == want


def test_job_rate_is_all_ranks_bytes_over_the_slowest_time():
    # 2 GB a step, 10 steps, 4 replicas, 20 ms -> 4000 GB/s
    assert abs(bench.job_rate_gbs(2e9, 10, 4, 20.0) - 4000.0) < 1e-9


def test_kernel_source_hash_follows_the_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "query_decode_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cuh").write_text("x")
    (csrc / "b.cu").write_text("y")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_source_hash(["a.cuh", "b.cu"])
    assert h1 == bench.kernel_source_hash(["b.cu", "a.cuh"])  # order-free
    (csrc / "b.cu").write_text("y ")
    assert bench.kernel_source_hash(["a.cuh", "b.cu"]) != h1
