"""One sequence's KV split over ranks, through the library's kernels: each
rank folds its token range into a running state (kq8_decode_attn_update), the
states are gathered, and kq8_state_merge + kq8_state_finalize give the whole
sequence's attention -- compared with the oracle's one pass over all tokens.
The two-rank case runs two processes that exchange their states over `gloo`;
both use the one GPU (their kernels never wait on each other)."""
import os
import socket

import numpy as np
import pytest

import oracle
from kq8_testlib import assert_out_close, host_inputs, oracle_decode
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from query_decode_attention_gb300 import kq8, paged, seqsplit  # noqa: E402

DEV = "cuda:0"


def _rank_state(case, wl, rank, world):
    """This rank's state: tokens kv_range(n_b, rank, world) of every sequence."""
    rng = [seqsplit.kv_range(int(n), rank, world) for n in wl.seq_lens]
    begin = torch.tensor([r[0] for r in rng], dtype=torch.int32, device=DEV)
    end = torch.tensor([r[1] for r in rng], dtype=torch.int32, device=DEV)
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                           DEV)
    longest = max(r[1] - r[0] for r in rng)
    kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, begin, end,
                               wl.max_seq_len, wl.scale, ws, max_range_len=max(1, longest))
    assert kq8.kq8_read_status(ws) == 0
    return state


@pytest.mark.parametrize("world", [2, 3, 5])
def test_split_states_merge_to_the_whole_sequence(world):
    wl = W.custom(3, 32, 8, [9000, 4001, 300], seed=60 + world)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    states = [_rank_state(case, wl, r, world) for r in range(world)]
    pa = torch.stack([s.acc for s in states]).contiguous()
    pm = torch.stack([s.ms for s in states]).contiguous()
    out = torch.empty((wl.B, wl.nq, 128), device=DEV)
    seqsplit.merge_gathered(out, pa, pm)
    assert_out_close(out.cpu().numpy(), oracle_decode(wl, q, Ks, Vs), f"{world}-way split")


def test_merge_of_no_parts_and_of_empty_states_changes_nothing():
    wl = W.custom(1, 16, 8, [500], seed=7)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    state = _rank_state(case, wl, 0, 1)
    acc0, ms0 = state.acc.clone(), state.ms.clone()
    empty = kq8.AttnState(wl.B, wl.nq, DEV)
    kq8.kq8_state_merge(state, empty.acc[None].contiguous(), empty.ms[None].contiguous())
    kq8.kq8_state_merge(state, torch.empty((0,) + tuple(state.acc.shape), device=DEV),
                        torch.empty((0,) + tuple(state.ms.shape), device=DEV))
    assert torch.equal(state.acc, acc0) and torch.equal(state.ms, ms0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        wl = W.custom(2, 16, 8, [20000, 7777], seed=70)
        q, Ks, Vs = host_inputs(wl)              # every rank draws the same inputs
        case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
        state = _rank_state(case, wl, rank, world)
        pa, pm = seqsplit.all_gather_states(state.acc, state.ms)
        out = torch.empty((wl.B, wl.nq, 128), device=DEV)
        seqsplit.merge_gathered(out, pa, pm)
        q_out.put((rank, out.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_sequence():
    world = 2
    ctx = mp.get_context("spawn")
    qo = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, qo)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((qo.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    wl = W.custom(2, 16, 8, [20000, 7777], seed=70)
    q, Ks, Vs = host_inputs(wl)
    ref = oracle_decode(wl, q, Ks, Vs)
    for rank, out in res:
        assert_out_close(out, ref, f"rank {rank} after the exchange")
    assert np.array_equal(res[0][1], res[1][1])   # both ranks finish with the same result
