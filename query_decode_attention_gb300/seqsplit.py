"""One long sequence's KV split over several ranks (one process per GPU).

The one-pass form (article 9-2 §3: KV may arrive piece by piece) lets each
rank attend only the tokens it holds: rank r folds its token range
[begin_r, end_r) of every sequence into a running state with
kq8_decode_attn_update, the ranks exchange their states -- per (sequence,
query head) one (max, sum) pair and a 128-float accumulator, the path's only
exchange -- and every rank folds the gathered states in rank order with
kq8_state_merge and finalises.  The result is the whole sequence's attention up
to rounding, whatever the split.

Only host logic lives here (the ranges and the exchange through
torch.distributed); every step of the method runs in the library's kernels.
"""
from __future__ import annotations

from typing import Tuple

import torch

TILE = 32  # tokens per cache sub-tile: ranges start on sub-tile boundaries


def kv_range(n: int, rank: int, world: int, tile: int = TILE) -> Tuple[int, int]:
    """Token range [begin, end) of a length-n sequence that `rank` of `world`
    attends: consecutive, disjoint ranges of whole tiles covering [0, n)."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("need 0 <= rank < world and n >= 0")
    tiles = -(-n // tile)
    t0, t1 = tiles * rank // world, tiles * (rank + 1) // world
    return min(n, t0 * tile), min(n, t1 * tile)


def all_gather_states(acc: torch.Tensor, ms: torch.Tensor, group=None):
    """Every rank's running state, stacked in rank order on acc's device:
    (acc [world, B, nq, 128], ms [world, B, nq, 2]).  With a CPU backend
    (gloo) the states travel through host memory."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    via_host = dist.get_backend(group) != "nccl"
    send_acc = acc.cpu() if via_host else acc.contiguous()
    send_ms = ms.cpu() if via_host else ms.contiguous()
    got_acc = [torch.empty_like(send_acc) for _ in range(world)]
    got_ms = [torch.empty_like(send_ms) for _ in range(world)]
    dist.all_gather(got_acc, send_acc, group=group)
    dist.all_gather(got_ms, send_ms, group=group)
    return (torch.stack(got_acc).to(acc.device), torch.stack(got_ms).to(ms.device))


def merge_gathered(out: torch.Tensor, part_acc: torch.Tensor, part_ms: torch.Tensor,
                   stream=None) -> None:
    """out [B, nq, 128] = the finalised fold of the gathered states."""
    from . import kq8
    B, nq = out.shape[0], out.shape[1]
    state = kq8.AttnState(B, nq, out.device, stream)
    kq8.kq8_state_merge(state, part_acc.contiguous(), part_ms.contiguous(), stream)
    kq8.kq8_state_finalize(out, state, stream)
