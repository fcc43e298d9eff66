"""q4 KV cache through the C ABI (the --kv-q4 switch of article 10-1 §2; the
format is this library's reading: the q8 rule of article 9-3 §2 with 7 levels a
side).  Codes and stored maxima bit-exact against the oracle's q4 write path;
decode outputs within max abs error <= min(1e-4, 1e-3 * max|out|)."""
import numpy as np
import pytest

import oracle
from kq8_testlib import assert_out_close, host_inputs
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _oracle_q4(Ks, Vs):
    out = [], [], [], []
    for K, V in zip(Ks, Vs):
        k4, ks = oracle.kv_quantize_rows_q4(K)
        v4, vs = oracle.kv_quantize_rows_q4(V)
        for lst, a in zip(out, (k4, ks, v4, vs)):
            lst.append(a)
    return out


@pytest.mark.parametrize("kv_bs", [32, 64])
def test_q4_append_bit_exact(kv_bs):
    wl = W.custom(3, 16, 8, [100, 33, 257], kind="student_t", seed=61, kv_bs=kv_bs)
    _, Ks, Vs = host_inputs(wl)
    Ks[0][5] = 0.0                                   # an all-zero row
    Ks[1][:, :, 7] *= np.float32(1e30)               # huge and tiny rows
    Vs[2][9] *= np.float32(1e-30)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, bits=4, pt_seed=2)
    for b in range(wl.B):
        n = int(wl.seq_lens[b])
        got = paged.unpack_q4(case.cache, case.slots(b, 0, n))
        k4, ks = oracle.kv_quantize_rows_q4(Ks[b])
        v4, vs = oracle.kv_quantize_rows_q4(Vs[b])
        for g, e, name in zip(got, (k4, ks, v4, vs), ("k codes", "k max", "v codes", "v max")):
            assert np.array_equal(g, e), (b, name)


@pytest.mark.parametrize("nq,nkv,lens,kv_bs", [
    (16, 8, [506, 1, 0, 33], 32),     # G = 2, empty and one-token sequences
    (32, 8, [2046, 777], 32),         # G = 4
    (8, 8, [300], 64),                # G = 1, kv_bs 64
    (64, 8, [1000, 64], 32),          # G = 8
    (6, 2, [129], 32),                # G = 3
    (16, 8, [1500, 257], 128),        # large pages
    (16, 8, [700], 256),
])
def test_q4_decode_matches_oracle(nq, nkv, lens, kv_bs):
    wl = W.custom(len(lens), nq, nkv, lens, kind="sigma", seed=sum(lens) + nq, kv_bs=kv_bs)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q, bits=4)
    out = torch.full((wl.B, wl.nq, wl.hd), float("nan"), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn_q4(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                           wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    k4, ks, v4, vs = _oracle_q4(Ks, Vs)
    ref = oracle.decode_batch_q4(q, k4, ks, v4, vs, wl.scale, kv_bs=wl.kv_bs)
    assert_out_close(out.cpu().numpy(), ref, f"q4 G={wl.G}")


def test_q4_serving_shape_sampled_sequences():
    # the serving shape (32/8 heads, ragged 1K-32K) on 6 sequences, every head
    # of every sequence against the oracle
    serv = W.serving_8b(B=6, layers=1, seed=3100)
    wl = W.custom(serv.B, 32, 8, serv.seq_lens, seed=3100)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q, bits=4)
    out = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn_q4(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                           wl.scale, ws)
    k4, ks, v4, vs = _oracle_q4(Ks, Vs)
    ref = oracle.decode_batch_q4(q, k4, ks, v4, vs, wl.scale)
    assert_out_close(out.cpu().numpy(), ref, "q4 serving shape")


def test_q4_bad_page_sets_status_and_caches_are_not_mixed():
    wl = W.custom(2, 16, 8, [200, 90], seed=71)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q, bits=4)
    pt = case.page_table.clone()
    pt[1, 1] = case.cache.num_pages + 5
    out = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn_q4(out, case.q, case.cache, pt, case.seq_lens, wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) & kq8.KQ8_STATUS_BAD_PAGE
    k4, ks, v4, vs = _oracle_q4(Ks[:1], Vs[:1])
    ref = oracle.decode_batch_q4(q[:1], k4, ks, v4, vs, wl.scale)
    assert_out_close(out[:1].cpu().numpy(), ref, "the good sequence")
    with pytest.raises(ValueError):
        kq8.kq8_decode_attn(out, case.q, case.cache, pt, case.seq_lens, wl.max_seq_len, wl.scale,
                            ws)


def test_q4_serving_full_size_sampled():
    # the bench's q4 line: the whole batch-64 serving layer in a q4 cache, in
    # its launch configuration; sampled (sequence, head) pairs against the
    # oracle's q4 write path and decode
    wl = W.serving_8b(layers=1)
    case = paged.fill_cache(wl, 0, DEV, bits=4)
    out = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn_q4(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                           wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    got = out.cpu().numpy()
    qh = case.q.cpu().numpy()
    hi, lo = int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens))
    for b, h in [(hi, 0), (hi, 30), (lo, 6), (21, 13), (63, 27)]:
        n = int(wl.seq_lens[b])
        K, V = case.device_kv(b, 0, n)
        kh = h // wl.G
        k4, ks = oracle.kv_quantize_rows_q4(K[:, kh:kh + 1].cpu().numpy())
        v4, vs = oracle.kv_quantize_rows_q4(V[:, kh:kh + 1].cpu().numpy())
        c = oracle.SeqCache(k4, ks, v4, vs, kv_bs=wl.kv_bs)
        ref = oracle.attn_single_q_q4(qh[b, h], c, 0, np.float32(wl.scale))
        assert_out_close(got[b, h], ref, f"q4 full size b={b} h={h}")
