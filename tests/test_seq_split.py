"""Host logic of one sequence's KV split over ranks, on CPU: the token ranges
cover the sequence exactly in whole tiles, and two `gloo` ranks all-gather
their running states in rank order.  The kernels' part (each rank's update,
the merge) is stood in for by the oracle's streaming form here; the GPU test
runs the library's own kernels."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from query_decode_attention_gb300 import seqsplit  # noqa: E402


@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 1000, 131072])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_ranges_cover_the_sequence_in_whole_tiles(n, world):
    rs = [seqsplit.kv_range(n, r, world) for r in range(world)]
    assert rs[0][0] == 0 and rs[-1][1] == n
    for (b0, e0), (b1, e1) in zip(rs, rs[1:]):
        assert e0 == b1                                   # consecutive, disjoint
    for b, e in rs:
        assert b <= e and b % 32 == 0 and (e % 32 == 0 or e == n)


def test_range_arguments_are_checked():
    with pytest.raises(ValueError):
        seqsplit.kv_range(10, 2, 2)
    with pytest.raises(ValueError):
        seqsplit.kv_range(-1, 0, 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from query_decode_attention_gb300 import workloads as W
        n = 3000
        wl = W.custom(1, 4, 2, [n], seed=17)
        qh = W.host_q(wl)
        K, V = W.host_kv(wl, 0)
        k8, ks = oracle.kv_quantize_rows(K)
        v8, vs = oracle.kv_quantize_rows(V)
        c = oracle.SeqCache(k8, ks, v8, vs)
        b, e = seqsplit.kv_range(n, rank, world)
        acc = torch.zeros((1, wl.nq, 128))
        ms = torch.zeros((1, wl.nq, 2))
        for h in range(wl.nq):                      # this rank's range only
            st = oracle.StreamState()
            oracle.attn_stream(st, qh[0, h], c, h // wl.G, np.float32(wl.scale), b, e)
            acc[0, h] = torch.tensor(st.acc)
            ms[0, h] = torch.tensor([float(st.M[0]), float(st.S[0])])
        pa, pm = seqsplit.all_gather_states(acc, ms)
        q.put((rank, pa.numpy(), pm.numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_states_in_rank_order():
    import oracle
    from query_decode_attention_gb300 import workloads as W
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted((q.get(timeout=10) for _ in range(world)), key=lambda x: x[0])
    assert np.array_equal(res[0][1], res[1][1]) and np.array_equal(res[0][2], res[1][2])
    pa, pm = res[0][1], res[0][2]                   # [world, 1, nq, 128], [world, 1, nq, 2]
    # fold the gathered states (natural-log maxima, as the oracle keeps them)
    # and compare with one pass over the whole sequence
    wl = W.custom(1, 4, 2, [3000], seed=17)
    qh = W.host_q(wl)
    K, V = W.host_kv(wl, 0)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    c = oracle.SeqCache(k8, ks, v8, vs)
    for h in range(wl.nq):
        m = pm[:, 0, h, 0].astype(np.float64)
        M = m.max()
        f = np.exp(m - M)
        out = (f[:, None] * pa[:, 0, h]).sum(0) / (f * pm[:, 0, h, 1]).sum()
        ref = oracle.attn_single_q(qh[0, h], c, h // wl.G, np.float32(wl.scale))
        assert np.abs(out - ref).max() <= 1e-5
