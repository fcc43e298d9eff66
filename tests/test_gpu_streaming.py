"""Streaming form through the C ABI (article 9-2 §3: the one-pass kernel can
compute while KV arrives piece by piece): running states folded over token
ranges match the oracle's one pass over the whole sequence, within the fp32
output tolerance."""
import numpy as np
import pytest

import oracle
from kq8_testlib import assert_out_close, host_inputs, oracle_decode
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _ws(wl):
    return kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                             DEV)


def _finalize(state, wl):
    out = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    kq8.kq8_state_finalize(out, state)
    return out.cpu().numpy()


@pytest.mark.parametrize("nq,nkv,lens,pieces", [
    (32, 8, [1000, 37, 2500], 3),
    (16, 8, [5000, 1, 64], 5),
    (8, 2, [300], 7),
])
def test_pieces_match_one_pass(nq, nkv, lens, pieces):
    wl = W.custom(len(lens), nq, nkv, lens, seed=sum(lens) + pieces)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    rng = np.random.default_rng(pieces)
    cuts = np.stack([np.concatenate([[0], np.sort(rng.integers(0, n + 1, pieces - 1)), [n]])
                     for n in lens]).astype(np.int32)          # [B, pieces + 1]
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    ws = _ws(wl)
    for k in range(pieces):
        b0 = torch.tensor(cuts[:, k], dtype=torch.int32, device=DEV)
        b1 = torch.tensor(cuts[:, k + 1], dtype=torch.int32, device=DEV)
        kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, b0, b1,
                                   wl.max_seq_len, wl.scale, ws,
                                   max_range_len=int((cuts[:, k + 1] - cuts[:, k]).max()))
    assert kq8.kq8_read_status(ws) == 0
    assert_out_close(_finalize(state, wl), oracle_decode(wl, q, Ks, Vs), f"{pieces} pieces")


def test_one_update_equals_decode_call():
    wl = W.custom(3, 32, 8, [4000, 100, 32], seed=31)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    out = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, _ws(wl))
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, None, case.seq_lens,
                               wl.max_seq_len, wl.scale, _ws(wl))
    assert_out_close(_finalize(state, wl), out.cpu().numpy(), "one update")


def test_kv_appended_between_updates():
    # the cache grows piece by piece; each update attends only the new piece
    wl = W.custom(2, 16, 8, [3000, 700], seed=41)
    q, Ks, Vs = host_inputs(wl)
    cache, pt = paged.new_cache(wl, device=DEV)
    pt_t = torch.tensor(pt, device=DEV)
    qd = torch.tensor(q, device=DEV)
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    ws = _ws(wl)
    done = np.zeros(wl.B, np.int32)
    for step in (500, 1200, 3000):
        new_end = np.minimum(wl.seq_lens, step).astype(np.int32)
        for b in range(wl.B):
            if new_end[b] > done[b]:
                sl = torch.tensor(W.slots_for(wl, pt, b, int(done[b]), int(new_end[b])), device=DEV)
                kq8.kq8_append_kv(cache, torch.tensor(Ks[b][done[b]:new_end[b]], device=DEV),
                                  torch.tensor(Vs[b][done[b]:new_end[b]], device=DEV), sl)
        kq8.kq8_decode_attn_update(state, qd, cache, pt_t, torch.tensor(done, device=DEV),
                                   torch.tensor(new_end, device=DEV), wl.max_seq_len, wl.scale, ws)
        done = new_end
    assert_out_close(_finalize(state, wl), oracle_decode(wl, q, Ks, Vs), "growing cache")


def test_empty_pieces_and_bad_start():
    wl = W.custom(2, 16, 8, [200, 90], seed=51)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    ws = _ws(wl)
    assert not _finalize(state, wl).any()
    same = torch.tensor([50, 90], dtype=torch.int32, device=DEV)
    kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, same, same,
                               wl.max_seq_len, wl.scale, ws)
    assert not _finalize(state, wl).any()                 # empty ranges change nothing
    bad = torch.tensor([0, 95], dtype=torch.int32, device=DEV)  # 95 > seq_end 90
    kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, bad, case.seq_lens,
                               wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == kq8.KQ8_STATUS_BAD_SEQLEN
    got = _finalize(state, wl)
    assert not got[1].any()                               # the bad sequence was skipped
    k8, ks = oracle.kv_quantize_rows(Ks[0])
    v8, vs = oracle.kv_quantize_rows(Vs[0])
    c = oracle.SeqCache(k8, ks, v8, vs)
    for h in range(wl.nq):
        assert_out_close(got[0, h], oracle.attn_single_q(q[0, h], c, h // wl.G, wl.scale), "seq 0")


def test_range_longer_than_the_hint_is_reported_and_skipped():
    wl = W.custom(2, 16, 8, [3000, 500], seed=61)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    ws = _ws(wl)
    # hint 500 tokens: sequence 0's 3000-token range exceeds what the grid covers
    kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, None, case.seq_lens,
                               wl.max_seq_len, wl.scale, ws, max_range_len=500)
    assert kq8.kq8_read_status(ws) == kq8.KQ8_STATUS_BAD_SEQLEN
    got = _finalize(state, wl)
    ref = oracle_decode(wl, q, Ks, Vs)
    assert_out_close(got[1], ref[1], "the in-bound sequence")


def test_long_context_full_size_eight_pieces_sampled():
    # the bench's streaming line: 8 sequences of 131072 tokens (Student-t keys
    # with outlier channels) folded in 8 equal pieces, in its launch
    # configuration; sampled (sequence, head) pairs against the oracle's one
    # pass, every output against the one-call decode
    wl = W.long_context()
    case = paged.fill_cache(wl, 0, DEV)
    ws = _ws(wl)
    pieces = 8
    state = kq8.AttnState(wl.B, wl.nq, DEV)
    kq8.kq8_state_reset(state)
    for k in range(pieces):
        b0 = torch.full((wl.B,), (wl.max_seq_len * k) // pieces, dtype=torch.int32, device=DEV)
        b1 = torch.full((wl.B,), (wl.max_seq_len * (k + 1)) // pieces, dtype=torch.int32,
                        device=DEV)
        kq8.kq8_decode_attn_update(state, case.q, case.cache, case.page_table, b0, b1,
                                   wl.max_seq_len, wl.scale, ws,
                                   max_range_len=-(-wl.max_seq_len // pieces))
    assert kq8.kq8_read_status(ws) == 0
    got = _finalize(state, wl)
    one = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    kq8.kq8_decode_attn(one, case.q, case.cache, case.page_table, case.seq_lens,
                        wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    assert_out_close(got, one.cpu().numpy(), "8 pieces vs one call")
    qh = case.q.cpu().numpy()
    # (3, 14): a head whose fp32 one-pass oracle is itself ~9e-4 from the exact
    # sums (long tail of small weights); there the exact-sum reference decides
    for b, h in [(0, 0), (2, 9), (3, 14), (7, 15)]:
        n = int(wl.seq_lens[b])
        K, V = case.device_kv(b, 0, n)
        kh = h // wl.G
        k8, ks = oracle.kv_quantize_rows(K[:, kh:kh + 1].cpu().numpy())
        v8, vs = oracle.kv_quantize_rows(V[:, kh:kh + 1].cpu().numpy())
        c = oracle.SeqCache(k8, ks, v8, vs, kv_bs=wl.kv_bs)
        ref = oracle.attn_single_q(qh[b, h], c, 0, np.float32(wl.scale))
        exact = oracle.attn_exact_sum(qh[b, h], c, 0, np.float32(wl.scale))
        assert_out_close(got[b, h], ref, f"streamed b={b} h={h}", exact=exact)
