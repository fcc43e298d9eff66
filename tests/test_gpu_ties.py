"""Block-sparse top-k with equal block scores, CUDA library vs CPU oracle.

The selection rule (article 10-1 §1-§2, this library's reading): per query
head the topk highest block scores are kept, and among equal scores the lower
block index wins.  Random inputs almost never produce equal fp32 scores, so
these inputs force them ("ties" workloads): all-zero K (every block scores
+0), K repeating one block (every whole block scores the same), and a few
strong blocks plus more copies of one block than the top-k has places left,
so that equal scores straddle the k-th place.  Kept block ids must match the
oracle bit for bit, outputs within the usual tolerance.
"""
import numpy as np
import pytest

import oracle
from kq8_testlib import assert_out_close, host_inputs, oracle_decode, oracle_quantized
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _sparse(case, shared=False):
    wl = case.wl
    out = torch.empty((wl.B, wl.nq, wl.hd), dtype=torch.float32, device=DEV)
    ws = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(
        wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block, wl.topk), DEV)
    sb = torch.full((wl.B, wl.nq, wl.topk), -7, dtype=torch.int32, device=DEV)
    fn = kq8.kq8_sparse_decode_attn_shared if shared else kq8.kq8_sparse_decode_attn
    fn(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len, wl.scale,
       wl.block, wl.topk, wl.probe, ws, sel_blocks=sb)
    assert kq8.kq8_read_status(ws) == 0
    return out.cpu().numpy(), sb.cpu().numpy()


def _assert_ties_straddle(wl, q, Ks, Vs):
    """The inputs do what they are for: in every sequence past the gate with more
    blocks than topk, every query head's k-th best score is shared by more
    blocks than the places left for it (checked on the oracle's scores)."""
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    checked = 0
    for b in range(wl.B):
        n = int(wl.seq_lens[b])
        if n <= 2 * wl.block or -(-n // wl.block) <= wl.topk:
            continue
        c = oracle.SeqCache(k8s[b], kss[b], v8s[b], vss[b], kv_bs=wl.kv_bs)
        for h in range(wl.nq):
            sc = oracle.probe_block_scores(q[b, h], c, h // wl.G, np.float32(wl.scale),
                                           wl.block, wl.probe)
            kth = np.sort(sc)[::-1][wl.topk - 1]
            assert (sc == kth).sum() > wl.topk - (sc > kth).sum(), (b, h)
            checked += 1
    assert checked > 0


@pytest.mark.parametrize("n", [4059, 65536])
def test_topk_ties_per_query_head(n):
    # n = 4059: 127 blocks, one radix bucket partly kept; n = 65536: 2048 blocks,
    # the tie bucket narrowed through all four radix passes
    wl = W.custom(3, 16, 8, [n] * 3, kind="ties", seed=n + 1)
    q, Ks, Vs = host_inputs(wl)
    _assert_ties_straddle(wl, q, Ks, Vs)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    got, sel = _sparse(case)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, f"ties n={n}")
    # all-zero K and a repeated block: every head keeps blocks 0 .. topk-1
    for b in range(wl.B):
        if W.tie_mode(b) in (0, 1):
            assert np.array_equal(sel[b], np.broadcast_to(np.arange(wl.topk), sel[b].shape))


@pytest.mark.parametrize("nq,nkv", [(16, 8), (32, 8)])
def test_topk_ties_shared_selection(nq, nkv):
    wl = W.custom(3, nq, nkv, [5000, 3001, 9000], kind="ties", seed=nq + 5)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    got, sel = _sparse(case, shared=True)
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref, rsel = oracle.decode_batch_shared(q, k8s, kss, v8s, vss, wl.scale, kv_bs=wl.kv_bs,
                                           block=wl.block, topk=wl.topk, probe=wl.probe)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, f"ties, shared selection G={wl.G}")


def test_topk_ties_knobs_and_block_64():
    # other knobs: block 64 / probe 16 / topk 5, and block 32 / probe 1 / topk 7
    for block, topk, probe in ((64, 5, 16), (32, 7, 1)):
        wl = W.custom(3, 16, 4, [4000, 2500, 3333], kind="ties", seed=block + topk,
                      block=block, topk=topk, probe=probe)
        q, Ks, Vs = host_inputs(wl)
        _assert_ties_straddle(wl, q, Ks, Vs)
        case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
        got, sel = _sparse(case)
        ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
        assert np.array_equal(sel, rsel), (block, topk, probe)
        assert_out_close(got, ref, f"ties block={block} topk={topk} probe={probe}")


def test_topk_ties_one_cta_per_kv_head():
    # more (sequence, KV head) pairs than the workspace has ticket counters: the
    # top-k takes its one-CTA-per-KV-head path, which must break ties the same way
    B = 2050
    lens = np.random.default_rng(91).integers(200, 400, B)
    wl = W.custom(B, 16, 8, [int(x) for x in lens], kind="ties", seed=92, topk=3, probe=4)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    got, sel = _sparse(case)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, "ties, 2050 sequences")
