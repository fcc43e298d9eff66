"""Stream order through the library's programmatic launches: each decode,
append and probe kernel may be scheduled while the kernel before it on the
stream finishes, and waits for that kernel's completion before it uses global
memory (the plain exact walk reads its inputs earlier only as a guess, which it
checks after the wait).  These cases put other work between and around the
calls on one stream and check that every call sees exactly what stream order
promises, against the oracle or against the same call after a
synchronisation."""
import numpy as np
import pytest

from kq8_testlib import assert_out_close, host_inputs, oracle_decode
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _case(lens, seed):
    wl = W.custom(len(lens), 16, 8, lens, seed=seed)
    q, Ks, Vs = host_inputs(wl)
    return wl, q, Ks, Vs


def test_append_then_rewritten_q_then_decode():
    # the last token of every sequence is appended, then a PyTorch kernel
    # rewrites q in place, then the decode: it must see both
    wl, q, Ks, Vs = _case([600, 1000, 33, 2], seed=90)
    cache, pt = paged.new_cache(wl, device=DEV)
    first = np.concatenate([W.slots_for(wl, pt, b, 0, n - 1) for b, n in enumerate(wl.seq_lens)])
    last = np.concatenate([W.slots_for(wl, pt, b, n - 1, n) for b, n in enumerate(wl.seq_lens)])
    k_first = np.concatenate([K[:-1].reshape(-1, wl.nkv, 128) for K in Ks])
    v_first = np.concatenate([V[:-1].reshape(-1, wl.nkv, 128) for V in Vs])
    k_last = np.concatenate([K[-1:].reshape(-1, wl.nkv, 128) for K in Ks])
    v_last = np.concatenate([V[-1:].reshape(-1, wl.nkv, 128) for V in Vs])
    kq8.kq8_append_kv(cache, torch.tensor(k_first, device=DEV), torch.tensor(v_first, device=DEV),
                      torch.tensor(first, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    kl, vl = torch.tensor(k_last, device=DEV), torch.tensor(v_last, device=DEV)
    sl = torch.tensor(last, dtype=torch.int32, device=DEV)
    qd = torch.tensor(q, device=DEV)
    page_table = torch.tensor(pt, dtype=torch.int32, device=DEV)
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=DEV)
    out = torch.empty((wl.B, wl.nq, 128), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_append_kv(cache, kl, vl, sl)
    qd.mul_(-1.5)
    kq8.kq8_decode_attn(out, qd, cache, page_table, seq_lens, wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    q2 = (q.astype(np.float32) * np.float32(-1.5)).astype(np.float32)
    assert_out_close(out.cpu().numpy(), oracle_decode(wl, q2, Ks, Vs), "append, q rewritten, decode")


def test_back_to_back_decodes_sharing_output_and_workspace():
    wl, q, Ks, Vs = _case([4000, 1500, 700], seed=91)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    q1 = case.q
    q2 = torch.tensor(np.random.default_rng(5).standard_normal(q.shape).astype(np.float32),
                      device=DEV)
    out = torch.empty((wl.B, wl.nq, 128), device=DEV)
    out_b = torch.empty_like(out)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    args = (case.cache, case.page_table, case.seq_lens, wl.max_seq_len, wl.scale, ws)
    kq8.kq8_decode_attn(out, q1, *args)
    snap = out.clone()                  # another kernel between the two calls
    kq8.kq8_decode_attn(out, q2, *args)  # same output and workspace
    kq8.kq8_decode_attn(out_b, q1, *args)  # and directly after it, no kernel between
    torch.cuda.synchronize()
    assert kq8.kq8_read_status(ws) == 0
    ref1 = oracle_decode(wl, q, Ks, Vs)
    ref2 = oracle_decode(wl, q2.cpu().numpy(), Ks, Vs)
    assert_out_close(snap.cpu().numpy(), ref1, "first decode")
    assert_out_close(out.cpu().numpy(), ref2, "second decode, same buffers")
    assert np.array_equal(out_b.cpu().numpy(), snap.cpu().numpy()), "third decode = first"


def test_sparse_exact_sparse_on_one_stream():
    wl = W.sparse_planted(4059, B=3)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    out_s, out_e, out_s2 = (torch.empty((wl.B, wl.nq, 128), device=DEV) for _ in range(3))
    sel, sel2 = (torch.full((wl.B, wl.nq, wl.topk), -7, dtype=torch.int32, device=DEV)
                 for _ in range(2))
    wss = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(
        wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block, wl.topk), DEV)
    wse = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                            DEV)
    sargs = (case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len, wl.scale,
             wl.block, wl.topk, wl.probe, wss)
    kq8.kq8_sparse_decode_attn(out_s, *sargs, sel_blocks=sel)
    kq8.kq8_decode_attn(out_e, case.q, case.cache, case.page_table, case.seq_lens,
                        wl.max_seq_len, wl.scale, wse)
    kq8.kq8_sparse_decode_attn(out_s2, *sargs, sel_blocks=sel2)
    torch.cuda.synchronize()
    assert kq8.kq8_read_status(wss) == 0 and kq8.kq8_read_status(wse) == 0
    ref_s, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel.cpu().numpy(), rsel) and np.array_equal(sel2.cpu().numpy(), rsel)
    assert_out_close(out_s.cpu().numpy(), ref_s, "sparse, first")
    assert np.array_equal(out_s2.cpu().numpy(), out_s.cpu().numpy()), "sparse, again"
    assert_out_close(out_e.cpu().numpy(), oracle_decode(wl, q, Ks, Vs), "exact between")


def _exact(out, q, case, wl, ws):
    kq8.kq8_decode_attn(out, q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, ws)


def _sparse(out, q, case, wl, ws):
    kq8.kq8_sparse_decode_attn(out, q, case.cache, case.page_table, case.seq_lens,
                               wl.max_seq_len, wl.scale, wl.block, wl.topk, wl.probe, ws)


@pytest.mark.parametrize("nq", [16, 32])
@pytest.mark.parametrize("first,second", [("exact", "exact"), ("exact", "sparse"),
                                          ("sparse", "exact"), ("sparse", "sparse")])
def test_query_is_the_previous_calls_output(first, second, nq):
    # The second call's query is the first call's output, with no other kernel
    # between them: the second call's CTAs may be resident while the first
    # call's last CTAs still write that output, and must not use it before the
    # first call has completed.  The first call is many waves long (its rows
    # are written up to its very end) and its output starts as NaN, so an early
    # read shows.  At 16 query heads (2 per KV head) the exact walk reads its
    # inputs before the wait as a guess and checks them after it: the guess is
    # then stale, and the walk has to start over from the values read after the
    # wait.  Reference: the same second call after a synchronisation.
    lens = list(W._rng(93).integers(4096, 16384, 32))
    wl = W.custom(32, nq, 8, lens, seed=93)
    case = paged.fill_cache(wl, 0, DEV)
    run = {"exact": _exact, "sparse": _sparse}
    nbytes = max(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                 kq8.kq8_sparse_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len,
                                                       wl.block, wl.topk))
    ws1, ws2 = kq8.new_workspace(nbytes, DEV), kq8.new_workspace(nbytes, DEV)
    a = torch.empty((wl.B, wl.nq, 128), device=DEV)
    c = torch.empty_like(a)
    ref = torch.empty_like(a)
    for rep in range(3):
        a.fill_(float("nan"))
        c.fill_(0.0)
        run[first](a, case.q, case, wl, ws1)
        run[second](c, a, case, wl, ws2)
        torch.cuda.synchronize()
        run[second](ref, a, case, wl, ws2)
        torch.cuda.synchronize()
        assert kq8.kq8_read_status(ws1) == 0 and kq8.kq8_read_status(ws2) == 0
        assert not torch.isnan(a).any(), "first call left rows unwritten"
        got, want = c.cpu().numpy(), ref.cpu().numpy()
        assert np.array_equal(got, want), (
            f"rep {rep}: {int((got != want).any(axis=2).sum())} of {wl.B * wl.nq} rows "
            "computed from a query read before the previous call completed")


def test_streamed_start_written_by_the_previous_call():
    # A streamed update whose start index is an int32 the call just before it
    # writes (the first block a sparse call selects, read as a token index), with
    # nothing between: the update may read its start early, as a guess, while the
    # sparse call's selection is still to come, and must then start over from the
    # value read after the wait.  Reference: the same update after a
    # synchronisation.
    wl = W.custom(1, 16, 8, [4059], seed=94)
    case = paged.fill_cache(wl, 0, DEV)
    ws_s = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(
        wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block, wl.topk), DEV)
    ws_u = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                             DEV)
    out_s = torch.empty((wl.B, wl.nq, 128), device=DEV)
    sel = torch.empty((wl.B, wl.nq, wl.topk), dtype=torch.int32, device=DEV)
    start = sel.view(-1)[:1]  # [B] = [1]: head 0's first selected block
    for rep in range(3):
        sel.fill_(-7)
        s1, s2 = kq8.AttnState(wl.B, wl.nq, DEV), kq8.AttnState(wl.B, wl.nq, DEV)  # reset
        kq8.kq8_sparse_decode_attn(out_s, case.q, case.cache, case.page_table, case.seq_lens,
                                   wl.max_seq_len, wl.scale, wl.block, wl.topk, wl.probe, ws_s,
                                   sel_blocks=sel)
        kq8.kq8_decode_attn_update(s1, case.q, case.cache, case.page_table, start, case.seq_lens,
                                   wl.max_seq_len, wl.scale, ws_u)
        torch.cuda.synchronize()
        kq8.kq8_decode_attn_update(s2, case.q, case.cache, case.page_table, start, case.seq_lens,
                                   wl.max_seq_len, wl.scale, ws_u)
        torch.cuda.synchronize()
        assert kq8.kq8_read_status(ws_s) == 0 and kq8.kq8_read_status(ws_u) == 0
        assert int(start.item()) >= 0
        assert torch.equal(s1.acc, s2.acc) and torch.equal(s1.ms, s2.ms), f"rep {rep}"
