"""CUDA library vs CPU oracle on the same seeded inputs, through the C ABI.

Integer work (int8 K/V/Q codes, stored scales, Q block scales, int32 block
dots, probe scores and kept block ids) must match bit for bit; fp32 outputs
within max abs error 1e-4 and 1e-3 * max|out|.
"""
import math

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


def _decode(case, sparse=False, sel=False):
    wl = case.wl
    out = torch.empty((wl.B, wl.nq, wl.hd), dtype=torch.float32, device=DEV)
    if sparse:
        nb = kq8.kq8_sparse_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block,
                                                   wl.topk)
        ws = kq8.new_workspace(nb, DEV)
        sb = torch.full((wl.B, wl.nq, wl.topk), -7, dtype=torch.int32, device=DEV) if sel else None
        kq8.kq8_sparse_decode_attn(out, case.q, case.cache, case.page_table, case.seq_lens,
                                   wl.max_seq_len, wl.scale, wl.block, wl.topk, wl.probe, ws,
                                   sel_blocks=sb)
        st = kq8.kq8_read_status(ws)
        assert st == 0, st
        return out.cpu().numpy(), (sb.cpu().numpy() if sel else None)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, ws)
    st = kq8.kq8_read_status(ws)
    assert st == 0, st
    return out.cpu().numpy()


def _host_case(wl, extra_pages=0, pt_seed=None):
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, extra_pages=extra_pages, q_host=q, pt_seed=pt_seed)
    return case, q, Ks, Vs


# ---------------------------------------------------------------------------
# write path, Q quantisation, block dots: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind,kv_bs", [("normal", 32), ("student_t", 32), ("sigma", 64),
                                        ("normal", 128)])
def test_append_bit_exact(kind, kv_bs):
    wl = W.custom(4, 16, 8, [1, 45, 300, 97], kind=kind, seed=7, kv_bs=kv_bs)
    case, q, Ks, Vs = _host_case(wl, extra_pages=3)
    for b in range(wl.B):
        n = int(wl.seq_lens[b])
        k8, ks, v8, vs = paged.unpack(case.cache, case.slots(b, 0, n))
        ok8, oks = oracle.kv_quantize_rows(Ks[b])
        ov8, ovs = oracle.kv_quantize_rows(Vs[b])
        assert np.array_equal(k8, ok8) and np.array_equal(v8, ov8)
        assert np.array_equal(ks.view(np.uint32), oks.view(np.uint32))
        assert np.array_equal(vs.view(np.uint32), ovs.view(np.uint32))


def test_append_8x4096_full_size_sampled():
    # the bench's write-path line: 8 x 4096 new tokens x 8 KV heads in one call
    # (its launch configuration); sampled token rows bit-exact against the oracle
    T, nkv = 8 * 4096, 8
    wl = W.custom(8, 16, nkv, [4096] * 8, seed=99)
    cache, pt = paged.new_cache(wl, device=DEV)
    case = paged.DeviceCase(wl, cache, pt, DEV, 0)
    g = W.device_generator(DEV, 99)
    kn = torch.randn((T, nkv, 128), generator=g, device=DEV)
    vn = torch.randn((T, nkv, 128), generator=g, device=DEV)
    sl = np.concatenate([case.slots(b, 0, 4096) for b in range(8)]).astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kq8.kq8_append_kv(cache, kn, vn, torch.tensor(sl, device=DEV), status=st)
    assert kq8.kq8_read_status(st) == 0
    rows = np.unique(np.concatenate([[0, 31, 32, 4095, 4096, T - 1],
                                     np.random.default_rng(99).integers(0, T, 250)]))
    k8, ks, v8, vs = paged.unpack(cache, sl[rows])
    ok8, oks = oracle.kv_quantize_rows(kn[rows].cpu().numpy())
    ov8, ovs = oracle.kv_quantize_rows(vn[rows].cpu().numpy())
    assert np.array_equal(k8, ok8) and np.array_equal(v8, ov8)
    assert np.array_equal(ks.view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), ovs.view(np.uint32))


def test_append_edge_rows_and_skipped_slots():
    nkv, T = 2, 6
    K = np.random.default_rng(1).standard_normal((T, nkv, 128)).astype(np.float32)
    K[0, 0] = 0.0                               # zero row -> zero codes, scale 0
    K[1, 1] = 1e-38                             # denormal-scale row
    K[2, 0, :4] = [2.0, 1.0, -1.0, -0.5]        # near-tie at 63.5 decided by fl(1/127)
    K[2, 0, 4:] = 0.0
    K[3, 1] *= np.float32(1e30)
    V = -K
    cache = kq8.PagedKVCache(2, nkv, 32, DEV)
    slots = np.array([0, 5, 33, -1, 63, 7], np.int32)  # -1 is skipped
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kq8.kq8_append_kv(cache, torch.tensor(K, device=DEV), torch.tensor(V, device=DEV),
                      torch.tensor(slots, device=DEV), status=st)
    assert kq8.kq8_read_status(st) == 0
    keep = slots >= 0
    k8, ks, v8, vs = paged.unpack(cache, slots[keep])
    ok8, oks = oracle.kv_quantize_rows(K[keep])
    ov8, ovs = oracle.kv_quantize_rows(V[keep])
    assert np.array_equal(k8, ok8) and np.array_equal(v8, ov8)
    assert np.array_equal(ks, oks) and np.array_equal(vs, ovs)
    assert list(k8[2, 0, :4]) == [127, 64, -64, -32]
    # the skipped token's slot (none) and untouched slots stay zero
    k8u, ksu, _, _ = paged.unpack(cache, np.array([1, 2], np.int32))
    assert not k8u.any() and not ksu.any()


def test_append_bad_slot_sets_status_and_skips():
    cache = kq8.PagedKVCache(1, 1, 32, DEV)
    K = torch.ones((2, 1, 128), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kq8.kq8_append_kv(cache, K, K, torch.tensor([3, 32], dtype=torch.int32, device=DEV), status=st)
    assert kq8.kq8_read_status(st) == kq8.KQ8_STATUS_BAD_SLOT
    assert kq8.kq8_read_status(st) == 0  # cleared
    assert int(cache.k.ne(0).sum()) == 128  # only slot 3 written


def test_quantize_q_bit_exact():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((64, 128)).astype(np.float32)
    q *= rng.choice([1e-8, 1e-6, 1e-3, 1.0, 7.0, 1e20], size=(64, 1)).astype(np.float32)
    q[0] = 0.0
    q[1, :32] = [1.0, 0.5, -0.5, 0.25] + [0.0] * 28
    qi, qsc = kq8.kq8_debug_quantize_q(torch.tensor(q, device=DEV))
    oqi, oqsc = oracle.quantize_q(q)
    assert np.array_equal(qi.cpu().numpy(), oqi)
    assert np.array_equal(qsc.cpu().numpy().view(np.uint32), oqsc.view(np.uint32))


def test_block_dots_bit_exact():
    wl = W.custom(3, 24, 8, [31, 64, 130], seed=11)   # G = 3
    case, q, Ks, Vs = _host_case(wl)
    dots = kq8.kq8_debug_block_dots(case.q, case.cache, case.page_table, case.seq_lens,
                                    wl.max_seq_len).cpu().numpy()
    qi, _ = oracle.quantize_q(q)
    k8s, _, _, _ = oracle_quantized(Ks, Vs)
    for b in range(wl.B):
        for h in range(wl.nq):
            for t in range(int(wl.seq_lens[b])):
                ref = oracle.block_dots(qi[b, h], k8s[b][t, h // wl.G])
                assert np.array_equal(dots[b, h, t], ref), (b, h, t)


# ---------------------------------------------------------------------------
# exact decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nq,nkv,lens", [
    (8, 8, [1, 32, 33, 700]),                 # G = 1
    (16, 8, [0, 5, 256, 1000]),               # G = 2, an empty sequence
    (12, 4, [64, 129, 2047]),                 # G = 3
    (32, 8, [31, 4096, 300]),                 # G = 4
    (10, 2, [100, 3000]),                     # G = 5
    (64, 8, [1, 2500]),                       # G = 8
])
def test_decode_small(nq, nkv, lens):
    wl = W.custom(len(lens), nq, nkv, lens, seed=sum(lens) + nq)
    case, q, Ks, Vs = _host_case(wl)
    got = _decode(case)
    ref = oracle_decode(wl, q, Ks, Vs)
    assert_out_close(got, ref, f"nq={nq} nkv={nkv} lens={lens}")
    for b, n in enumerate(lens):
        if n == 0:
            assert not got[b].any()


@pytest.mark.parametrize("kv_bs", [64, 256])
def test_decode_page_sizes(kv_bs):
    wl = W.custom(2, 16, 8, [500, 1531], seed=5, kv_bs=kv_bs)
    case, q, Ks, Vs = _host_case(wl)
    assert_out_close(_decode(case), oracle_decode(wl, q, Ks, Vs), f"kv_bs={kv_bs}")


def test_decode_tiny_config_and_precision():
    wl = W.tiny()
    case, q, Ks, Vs = _host_case(wl)
    got = _decode(case)
    assert_out_close(got, oracle_decode(wl, q, Ks, Vs), "tiny")
    # article 9-3 §3: fp32-KV attention vs this q8 path, about 0.01
    d = max(np.abs(got[0, h] - oracle.attn_ref_f64(q[0, h], Ks[0][:, h // wl.G],
                                                    Vs[0][:, h // wl.G], 1 / math.sqrt(128))).max()
            for h in range(wl.nq))
    assert d <= 0.02


@pytest.mark.parametrize("k_factor", [8.0, 64.0])
def test_decode_large_scores(k_factor):
    # Student-t keys with x20 outlier channels, scaled once more by a power of
    # two (every score scales exactly): scores in the hundreds and thousands
    wl = W.custom(3, 32, 8, [6000, 2500, 700], kind="student_t", seed=19)
    q, Ks, Vs = host_inputs(wl)
    Ks = [(K * np.float32(k_factor)).astype(np.float32) for K in Ks]
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    assert_out_close(_decode(case), oracle_decode(wl, q, Ks, Vs), f"keys x{k_factor}")


@pytest.mark.parametrize("n", [506, 2046, 4059])
def test_decode_qwen3vl_2b_all_layers(n):
    wl = W.qwen3vl_2b(n)
    for layer in range(wl.layers):
        q = W.host_q(wl, layer)
        K, V = W.host_kv(wl, 0, layer)
        case = paged.fill_from_host(wl, [K], [V], DEV, q_host=q)
        got = _decode(case)
        ref = oracle_decode(wl, q, [K], [V])
        assert_out_close(got, ref, f"n={n} layer={layer}")


def _sampled_full_size(wl, samples, layer=0):
    """Full-size cache on the device; the oracle checks a sample of (b, h),
    regenerating each sampled sequence's fp32 K/V once."""
    case = paged.fill_cache(wl, layer, DEV)
    got = _decode(case)
    qh = case.q.cpu().numpy()
    by_seq = {}
    for b, h in samples:
        by_seq.setdefault(b, []).append(h)
    for b, heads in by_seq.items():
        n = int(wl.seq_lens[b])
        K, V = case.device_kv(b, 0, n)
        caches = {}
        for kh in sorted({h // wl.G for h in heads}):
            k8, ks = oracle.kv_quantize_rows(K[:, kh:kh + 1].cpu().numpy())
            v8, vs = oracle.kv_quantize_rows(V[:, kh:kh + 1].cpu().numpy())
            caches[kh] = oracle.SeqCache(k8, ks, v8, vs, kv_bs=wl.kv_bs)
        for h in heads:
            c = caches[h // wl.G]
            ref = oracle.attn_single_q(qh[b, h], c, 0, np.float32(wl.scale))
            exact = oracle.attn_exact_sum(qh[b, h], c, 0, np.float32(wl.scale))
            assert_out_close(got[b, h], ref, f"{wl.name} b={b} h={h}", exact=exact)
        del K, V
    return case, got


def test_decode_serving_full_size_sampled():
    # every query head of the longest and the shortest sequence (all four heads
    # of each KV group, so a slip confined to some heads of a group shows), and
    # a spread of (sequence, head) pairs elsewhere
    wl = W.serving_8b()
    hi = int(np.argmax(wl.seq_lens))
    lo = int(np.argmin(wl.seq_lens))
    samples = [(hi, h) for h in range(wl.nq)] + [(lo, h) for h in range(wl.nq)]
    samples += [(7, 9), (33, 22), (63, 12), (20, 3), (50, 30)]
    _sampled_full_size(wl, samples)


def test_decode_long_context_full_size_sampled():
    # all 16 query heads of one 131072-token sequence, and heads of two others
    wl = W.long_context()
    _sampled_full_size(wl, [(3, h) for h in range(wl.nq)] + [(0, 0), (7, 15)])


# ---------------------------------------------------------------------------
# block-sparse decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [64, 65, 506, 4059])
def test_sparse_matches_oracle(n):
    wl = W.sparse_planted(n, B=3)
    case, q, Ks, Vs = _host_case(wl)
    got, sel = _decode(case, sparse=True, sel=True)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, f"sparse n={n}")


def test_sparse_rows_that_keep_every_block_next_to_probed_rows():
    # rows past the gate (n > 2 * block) but with no more blocks than topk keep
    # every block, in order, without a probe; they share the batch with rows
    # that are probed and selected, and with a gated and an empty row
    wl = W.custom(5, 16, 8, [506, 4059, 100, 64, 0], seed=81, block=32, topk=32, probe=8)
    case, q, Ks, Vs = _host_case(wl)
    got, sel = _decode(case, sparse=True, sel=True)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert (sel[0, :, :16] == np.arange(16)).all() and (sel[0, :, 16:] == -1).all()
    assert_out_close(got, ref, "sparse, kept-all rows among probed rows")


def test_sparse_many_sequences_one_topk_cta_per_kv_head():
    # more (sequence, KV head) pairs than the workspace header has counters
    # (16384): the top-k runs one CTA per KV head selecting its G heads in
    # turn instead of one CTA per query head; selections and outputs as before
    B = 2050
    lens = np.random.default_rng(77).integers(65, 200, B)
    wl = W.custom(B, 16, 8, [int(x) for x in lens], seed=78, block=32, topk=3, probe=4)
    case, q, Ks, Vs = _host_case(wl)
    got, sel = _decode(case, sparse=True, sel=True)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, "sparse, 2050 sequences")


@pytest.mark.parametrize("block,topk,probe", [(32, 4, 8), (64, 3, 5), (32, 7, 32), (96, 2, 1),
                                               (64, 5, 16), (128, 6, 32)])
def test_sparse_knobs(block, topk, probe):
    wl = W.custom(3, 16, 4, [2000, 700, 3001], seed=block + topk + probe, block=block, topk=topk,
                  probe=probe)
    case, q, Ks, Vs = _host_case(wl)
    scores = kq8.kq8_debug_probe_scores(case.q, case.cache, case.page_table, case.seq_lens,
                                        wl.max_seq_len, wl.scale, block, probe).cpu().numpy()
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    for b in range(wl.B):
        c = oracle.SeqCache(k8s[b], kss[b], v8s[b], vss[b])
        for h in range(wl.nq):
            ref = oracle.probe_block_scores(q[b, h], c, h // wl.G, np.float32(wl.scale), block,
                                            probe)
            assert np.array_equal(scores[b, h, :len(ref)], ref), (b, h)
    got, sel = _decode(case, sparse=True, sel=True)
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, f"sparse knobs {block},{topk},{probe}")


def test_sparse_gate_is_bit_identical_to_exact():
    wl = W.custom(4, 16, 8, [1, 40, 64, 63], seed=9)
    case, q, Ks, Vs = _host_case(wl)
    ex = _decode(case)
    sp, sel = _decode(case, sparse=True, sel=True)
    assert np.array_equal(ex, sp)
    assert np.all(sel == -1)


def test_sparse_planted_full_size():
    for n in (16384, 65536):
        wl = W.sparse_planted(n, B=16)
        case, q, Ks, Vs = _host_case(wl)
        got, sel = _decode(case, sparse=True, sel=True)
        ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
        assert np.array_equal(sel, rsel)
        assert_out_close(got, ref, f"sparse n={n}")
        for b in range(wl.B):
            for h in range(wl.nq):
                assert set(sel[b, h].tolist()) == set(W.planted_blocks(wl, b, h // wl.G).tolist())


def _decode_shared(case):
    wl = case.wl
    out = torch.empty((wl.B, wl.nq, wl.hd), dtype=torch.float32, device=DEV)
    nb = kq8.kq8_sparse_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len, wl.block,
                                               wl.topk)
    ws = kq8.new_workspace(nb, DEV)
    sb = torch.full((wl.B, wl.nq, wl.topk), -7, dtype=torch.int32, device=DEV)
    kq8.kq8_sparse_decode_attn_shared(out, case.q, case.cache, case.page_table, case.seq_lens,
                                      wl.max_seq_len, wl.scale, wl.block, wl.topk, wl.probe, ws,
                                      sel_blocks=sb)
    assert kq8.kq8_read_status(ws) == 0
    return out.cpu().numpy(), sb.cpu().numpy()


@pytest.mark.parametrize("nq,nkv,lens,block,topk,probe", [
    (16, 8, [3000, 65, 800], 32, 4, 8),      # G = 2, one sequence at the gate
    (32, 8, [5000, 2000], 32, 8, 8),         # G = 4
    (64, 8, [1500], 64, 3, 16),              # G = 8, block 64
])
def test_shared_selection_matches_oracle(nq, nkv, lens, block, topk, probe):
    # one selection per KV head (max of its query heads' block scores)
    wl = W.custom(len(lens), nq, nkv, lens, seed=sum(lens) + nq, block=block, topk=topk,
                  probe=probe)
    case, q, Ks, Vs = _host_case(wl)
    got, sel = _decode_shared(case)
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref, rsel = oracle.decode_batch_shared(q, k8s, kss, v8s, vss, wl.scale, kv_bs=wl.kv_bs,
                                           block=block, topk=topk, probe=probe)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, f"shared selection G={wl.G}")
    for b in range(wl.B):                    # the group's heads share their blocks
        for h in range(0, wl.nq, wl.G):
            assert all(np.array_equal(sel[b, h], sel[b, h + g]) for g in range(wl.G))


def test_shared_selection_planted_recall():
    wl = W.sparse_planted(16384, B=4)
    case, q, Ks, Vs = _host_case(wl)
    got, sel = _decode_shared(case)
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref, rsel = oracle.decode_batch_shared(q, k8s, kss, v8s, vss, wl.scale, block=wl.block,
                                           topk=wl.topk, probe=wl.probe)
    assert np.array_equal(sel, rsel)
    assert_out_close(got, ref, "shared selection, planted")
    for b in range(wl.B):
        for h in range(wl.nq):
            assert set(sel[b, h].tolist()) == set(W.planted_blocks(wl, b, h // wl.G).tolist())


# ---------------------------------------------------------------------------
# device-side checks of untrusted metadata
# ---------------------------------------------------------------------------

def test_bad_page_and_seq_len_set_status():
    wl = W.custom(2, 16, 8, [100, 50], seed=2)
    case, q, Ks, Vs = _host_case(wl)
    pt = case.page_table.clone()
    pt[1, 0] = case.cache.num_pages + 5          # out of the pool
    out = torch.empty((2, 16, 128), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(2, 16, 8, wl.max_seq_len), DEV)
    kq8.kq8_decode_attn(out, case.q, case.cache, pt, case.seq_lens, wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) & kq8.KQ8_STATUS_BAD_PAGE
    ref = oracle_decode(wl, q, Ks, Vs)
    assert_out_close(out.cpu().numpy()[0], ref[0], "untouched sequence")
    sl = torch.tensor([100, 5000], dtype=torch.int32, device=DEV)  # > max_seq_len
    kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table, sl, wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == kq8.KQ8_STATUS_BAD_SEQLEN
    assert not out[1].any()


def test_cuda_graph_replay():
    wl = W.custom(3, 32, 8, [3000, 17, 900], seed=4)
    case, q, Ks, Vs = _host_case(wl)
    out = torch.zeros((3, 32, 128), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(3, 32, 8, wl.max_seq_len), DEV)
    s = torch.cuda.Stream()
    kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, ws, stream=s)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kq8.kq8_decode_attn(out, case.q, case.cache, case.page_table, case.seq_lens,
                            wl.max_seq_len, wl.scale, ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_out_close(out.cpu().numpy(), oracle_decode(wl, q, Ks, Vs), "graph replay")
