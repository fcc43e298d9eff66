"""Host-side split plans of the decode kernels (no GPU needed: without a
device the plans assume a GB300's 152 SMs).  The properties the kernels and
the workspace layout rely on, over a grid of shapes:

- chunks are whole multiples of the CTA's 4 warps, 4 to 128 tiles (a warp
  holds at most 32 tile ids, one per lane), and they cover the longest list
  with no empty chunk at its end;
- exact walks: when one wave of resident CTAs can hold every list in chunks
  of at most 128 tiles, the plan stays within that wave (at most 16 chunks a
  list); otherwise it uses more than one wave;
- block-sparse walks: the chunks cover a list of min(G * topk, blocks)
  blocks, and the grid stays within one wave (or one chunk a list) unless a
  list needs more chunks of at most 128 tiles;
- dealt out in turn, a sparse list of any length up to that gives no chunk
  more than 128 entries.
"""
import math

import pytest

from query_decode_attention_gb300 import kq8

SMS = 152
SHAPES = [(B, nq, nkv) for B in (1, 2, 8, 16, 64, 256, 4096)
          for nq, nkv in ((8, 8), (16, 8), (32, 8), (64, 8), (16, 2), (40, 8))]
LENS = (0, 1, 31, 32, 33, 506, 4059, 32768, 131072)


def _per_sm(G):
    return 3 if G <= 4 else 2


def _chunk_shape(ct, nc, tiles):
    assert ct % 4 == 0 and 4 <= ct <= 128, (ct, nc, tiles)
    assert nc >= 1
    assert nc * ct >= tiles, (ct, nc, tiles)
    if tiles > 0:
        assert (nc - 1) * ct < tiles, (ct, nc, tiles)


@pytest.mark.parametrize("B,nq,nkv", SHAPES)
def test_exact_plan(B, nq, nkv):
    G = nq // nkv
    slots = SMS * _per_sm(G)
    pairs = B * nkv
    for n in LENS:
        ct, nc = kq8.kq8_decode_plan(B, nq, nkv, n)
        tiles = math.ceil(n / 32)
        _chunk_shape(ct, nc, tiles)
        per = min(16, slots // pairs)
        if per >= 1 and math.ceil(tiles / per) <= 128:
            assert nc <= per and pairs * nc <= slots, (B, nq, nkv, n, ct, nc)
        else:
            assert pairs * nc > slots, (B, nq, nkv, n, ct, nc)


@pytest.mark.parametrize("B,nq,nkv", SHAPES)
@pytest.mark.parametrize("block,topk", [(32, 32), (64, 16), (32, 4), (96, 8)])
def test_sparse_plan(B, nq, nkv, block, topk):
    G = nq // nkv
    slots = SMS * _per_sm(G)
    pairs = B * nkv
    for n in LENS:
        ct, nc = kq8.kq8_sparse_decode_plan(B, nq, nkv, n, block, topk)
        tiles = math.ceil(n / 32)
        nblk = math.ceil(n / block)
        cap = min(tiles, min(nblk, G * topk) * (block // 32))
        _chunk_shape(ct, nc, cap)
        # one wave of CTAs (at least one chunk a list), unless a list needs more
        # chunks of at most 128 tiles
        assert nc <= max(max(1, slots // pairs), math.ceil(cap / 128)), (B, nq, nkv, n, ct, nc)
        # entries dealt out in turn: chunk c of an e-entry list takes
        # ceil((e - c) / nc) of them
        for e in {1, cap // 2, cap}:
            if e > 0:
                assert max(math.ceil((e - c) / nc) for c in range(min(nc, e))) <= 128


def test_plan_argument_errors():
    with pytest.raises(Exception):
        kq8.kq8_decode_plan(1, 16, 0, 100)
    with pytest.raises(Exception):
        kq8.kq8_sparse_decode_plan(1, 16, 8, 100, 48, 32)  # block not a multiple of 32
