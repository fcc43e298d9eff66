"""Batched causal prefill through the C ABI against the oracle (article 10-1
§1: nb new tokens against the whole history; each new token is one decode
query of article 9-2 §2 over the tokens up to itself).  fp32 outputs within
max abs error <= min(1e-4, 1e-3 * max|out|), element by element."""
import numpy as np
import pytest

import oracle
from kq8_testlib import assert_out_close, host_inputs, oracle_quantized
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _run(wl, q_lens, seed=0, kind="normal", pt_seed=None, k_factor=1.0):
    """Cache of wl (its seq_lens include the new tokens), packed queries for
    q_lens new tokens per sequence; returns (gpu out, oracle out, status).
    k_factor scales every key (a power of two scales every score exactly)."""
    q_lens = np.asarray(q_lens, np.int32)
    _, Ks, Vs = host_inputs(wl)
    Ks = [(K * np.float32(k_factor)).astype(np.float32) for K in Ks]
    T = int(q_lens.sum())
    qp = np.random.default_rng(seed).standard_normal((T, wl.nq, wl.hd)).astype(np.float32)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, pt_seed=pt_seed)
    q_off = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    out = torch.full((T, wl.nq, wl.hd), float("nan"), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_prefill_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len,
                                                           int(q_lens.max(initial=0))), DEV)
    kq8.kq8_prefill_attn(out, torch.tensor(qp, device=DEV), case.cache, case.page_table,
                         case.seq_lens, torch.tensor(q_off, device=DEV), wl.max_seq_len,
                         int(q_lens.max(initial=0)), wl.scale, ws)
    status = kq8.kq8_read_status(ws)
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref = oracle.prefill_batch(qp, q_lens, k8s, kss, v8s, vss, wl.scale, kv_bs=wl.kv_bs)
    return out.cpu().numpy(), ref, status


@pytest.mark.parametrize("nq,nkv,lens,q_lens", [
    (16, 8, [300, 77, 1000], [300, 5, 130]),      # G = 2 (Qwen3-VL-2B heads), whole prompt + chunks
    (32, 8, [2000, 64], [257, 64]),               # G = 4, ragged tiles on both sides
    (8, 8, [129], [129]),                         # G = 1: 128 tokens per CTA + a tail of 1
    (8, 1, [500, 33], [40, 33]),                  # G = 8: 16 tokens per CTA
    (6, 2, [200], [100]),                         # G = 3: 42 tokens per CTA, 2 idle rows
    (16, 8, [1, 31, 32, 33], [1, 31, 1, 33]),     # sub-tile boundaries
])
def test_prefill_matches_oracle(nq, nkv, lens, q_lens):
    wl = W.custom(len(lens), nq, nkv, lens, seed=sum(lens) + nq)
    got, ref, status = _run(wl, q_lens, seed=len(lens))
    assert status == 0
    assert_out_close(got, ref, f"G={nq // nkv}")


def test_prefill_sigma_kv_and_kv_bs_64():
    wl = W.custom(2, 16, 8, [700, 1500], kind="sigma", seed=7, kv_bs=64)
    got, ref, status = _run(wl, [700, 96], seed=8, pt_seed=3)
    assert status == 0
    assert_out_close(got, ref, "sigma, kv_bs 64")


@pytest.mark.parametrize("kv_bs", [128, 256])
def test_prefill_large_pages(kv_bs):
    wl = W.custom(2, 32, 8, [1100, 300], seed=kv_bs, kv_bs=kv_bs)
    got, ref, status = _run(wl, [333, 300], seed=kv_bs + 1, pt_seed=5)
    assert status == 0
    assert_out_close(got, ref, f"kv_bs {kv_bs}")


def test_prefill_outlier_keys_force_rescales():
    # Student-t keys with x20 channels: the running max jumps often, so the
    # lazy O rescale in tensor memory runs on many rows
    wl = W.custom(1, 16, 8, [3000], kind="student_t", seed=11)
    got, ref, status = _run(wl, [200], seed=12)
    assert status == 0
    assert_out_close(got, ref, "student-t")


def test_prefill_zero_new_tokens_and_single_token():
    wl = W.custom(3, 16, 8, [90, 40, 1], seed=13)
    got, ref, status = _run(wl, [0, 7, 1], seed=14)
    assert status == 0 and got.shape[0] == 8
    assert_out_close(got, ref, "nb = 0 / 7 / 1")


def test_prefill_single_new_token_equals_decode():
    wl = W.custom(3, 32, 8, [5000, 333, 64], seed=15)
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len), DEV)
    dec = torch.empty((wl.B, wl.nq, wl.hd), device=DEV)
    kq8.kq8_decode_attn(dec, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, ws)
    pre = torch.empty_like(dec)
    kq8.kq8_prefill_attn(pre, case.q, case.cache, case.page_table, case.seq_lens,
                         torch.arange(wl.B + 1, dtype=torch.int32, device=DEV), wl.max_seq_len, 1,
                         wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    assert_out_close(pre.cpu().numpy(), dec.cpu().numpy(), "prefill nb=1 vs decode")


def test_prefill_bad_bounds_skip_only_that_sequence():
    wl = W.custom(2, 16, 8, [100, 50], seed=17)
    _, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV)
    # sequence 1 claims 60 new tokens but holds 50
    q_off = torch.tensor([0, 10, 70], dtype=torch.int32, device=DEV)
    qp = np.random.default_rng(18).standard_normal((70, 16, 128)).astype(np.float32)
    out = torch.zeros((70, 16, 128), device=DEV)
    ws = kq8.new_workspace(4096, DEV)
    kq8.kq8_prefill_attn(out, torch.tensor(qp, device=DEV), case.cache, case.page_table,
                         case.seq_lens, q_off, wl.max_seq_len, 60, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == kq8.KQ8_STATUS_BAD_SEQLEN
    got = out.cpu().numpy()
    assert not got[10:].any()                      # the bad sequence was not written
    k8s, kss, v8s, vss = oracle_quantized(Ks[:1], Vs[:1])
    ref = oracle.prefill_batch(qp[:10], [10], k8s, kss, v8s, vss, wl.scale)
    assert_out_close(got[:10], ref, "good sequence")


def test_prefill_qwen2b_prompt_sampled_rows():
    # a whole 4059-token Qwen3-VL-2B prompt in one call, as the prefill bench
    # line runs it; the oracle checks every query head of 64 sampled tokens
    wl = W.qwen3vl_2b(4059)
    _, Ks, Vs = host_inputs(wl)
    n = int(wl.seq_lens[0])
    qp = np.random.default_rng(19).standard_normal((n, wl.nq, wl.hd)).astype(np.float32)
    case = paged.fill_from_host(wl, Ks, Vs, DEV)
    out = torch.empty((n, wl.nq, wl.hd), device=DEV)
    ws = kq8.new_workspace(4096, DEV)
    kq8.kq8_prefill_attn(out, torch.tensor(qp, device=DEV), case.cache, case.page_table,
                         case.seq_lens, torch.tensor([0, n], dtype=torch.int32, device=DEV), n, n,
                         wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    got = out.cpu().numpy()
    rows = np.unique(np.concatenate([[0, 1, 31, 32, 63, 64, n - 1],
                                     np.random.default_rng(20).integers(0, n, 57)]))
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    for i in rows:
        p = int(i) + 1  # token i of the prompt sees tokens 0..i: a 1-token prefill of the prefix
        ref = oracle.prefill_batch(qp[i:i + 1], [1], [k8s[0][:p]], [kss[0][:p]], [v8s[0][:p]],
                                   [vss[0][:p]], wl.scale)
        assert_out_close(got[i:i + 1], ref, f"token {i}")


def test_prefill_qwen8b_prompt_sampled_rows():
    # a whole 8192-token Qwen3-VL-8B prompt (32 query heads on 8 KV heads, G = 4)
    # in one call, the other prefill bench line; 40 sampled tokens, every head
    n = 8192
    wl = W.Workload("qwen3vl8b_prompt_n8192", 1, 32, 8, np.array([n], np.int32), kind="sigma",
                    seed=2100 + n)
    _, Ks, Vs = host_inputs(wl)
    qp = np.random.default_rng(21).standard_normal((n, wl.nq, wl.hd)).astype(np.float32)
    case = paged.fill_from_host(wl, Ks, Vs, DEV)
    out = torch.empty((n, wl.nq, wl.hd), device=DEV)
    ws = kq8.new_workspace(4096, DEV)
    kq8.kq8_prefill_attn(out, torch.tensor(qp, device=DEV), case.cache, case.page_table,
                         case.seq_lens, torch.tensor([0, n], dtype=torch.int32, device=DEV), n, n,
                         wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    got = out.cpu().numpy()
    rows = np.unique(np.concatenate([[0, 31, 32, 63, 64, 4095, n - 1],
                                     np.random.default_rng(22).integers(0, n, 33)]))
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    for i in rows:
        p = int(i) + 1
        ref = oracle.prefill_batch(qp[i:i + 1], [1], [k8s[0][:p]], [kss[0][:p]], [v8s[0][:p]],
                                   [vss[0][:p]], wl.scale)
        assert_out_close(got[i:i + 1], ref, f"token {i}")


# ---------------------------------------------------------------------------
# Block-sparse prefill (article 10-1 §1-§2): per token, the block-sparse decode
# query over its own prefix; selections bit-exact, outputs within tolerance.
# ---------------------------------------------------------------------------

def _run_sparse(wl, q_lens, block, topk, probe, seed=0):
    q_lens = np.asarray(q_lens, np.int32)
    _, Ks, Vs = host_inputs(wl)
    T = int(q_lens.sum())
    qp = np.random.default_rng(seed).standard_normal((T, wl.nq, wl.hd)).astype(np.float32)
    case = paged.fill_from_host(wl, Ks, Vs, DEV)
    q_off = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    out = torch.full((T, wl.nq, wl.hd), float("nan"), device=DEV)
    sel = torch.full((T, wl.nq, topk), -7, dtype=torch.int32, device=DEV)
    mq = int(q_lens.max(initial=0))
    ws = kq8.new_workspace(kq8.kq8_sparse_prefill_workspace_bytes(T, wl.nq, wl.nkv, wl.max_seq_len,
                                                                  block, topk), DEV)
    kq8.kq8_sparse_prefill_attn(out, torch.tensor(qp, device=DEV), case.cache, case.page_table,
                                case.seq_lens, torch.tensor(q_off, device=DEV), wl.max_seq_len, mq,
                                wl.scale, block, topk, probe, ws, sel_blocks=sel)
    status = kq8.kq8_read_status(ws)
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref, ref_sel = oracle.prefill_batch(qp, q_lens, k8s, kss, v8s, vss, wl.scale, kv_bs=wl.kv_bs,
                                        sparse=True, block=block, topk=topk, probe=probe)
    return out.cpu().numpy(), sel.cpu().numpy(), ref, ref_sel, status


@pytest.mark.parametrize("nq,nkv,lens,q_lens,block,topk,probe", [
    (16, 8, [600], [600], 32, 4, 8),             # every prefix: gated (<= 64) and pruned rows
    (32, 8, [1500, 90], [128, 90], 32, 8, 8),    # history + chunk, G = 4
    (8, 2, [700], [64], 64, 3, 16),              # block 64 (two sub-tiles per block)
])
def test_sparse_prefill_matches_oracle(nq, nkv, lens, q_lens, block, topk, probe):
    wl = W.custom(len(lens), nq, nkv, lens, seed=sum(lens) + block)
    got, sel, ref, ref_sel, status = _run_sparse(wl, q_lens, block, topk, probe, seed=topk)
    assert status == 0
    assert np.array_equal(sel, ref_sel), "block selections differ"
    assert_out_close(got, ref, "sparse prefill")


def test_sparse_prefill_full_cover_equals_exact_prefill():
    # k * block >= n: nothing is pruned, so the sparse path is the exact one
    wl = W.custom(1, 16, 8, [500], seed=23)
    got, sel, ref, _, status = _run_sparse(wl, [500], 32, 32, 8, seed=24)
    exact, _, status2 = _run(wl, [500], seed=24)
    assert status == 0 and status2 == 0
    assert_out_close(got, exact, "sparse (all blocks kept) vs exact prefill")
    assert_out_close(got, ref, "sparse vs oracle")


@pytest.mark.parametrize("nq,nkv,n", [(16, 8, 4059), (32, 8, 8192)])
def test_sparse_prefill_bench_prompts_sampled_rows(nq, nkv, n):
    # the bench's block-sparse prefill lines (block 32, k 32, probe 8) on the
    # whole prompt in its launch configuration; the 8192-token prompt has more
    # (row, KV head) pairs than ticket counters, so its top-k runs one CTA per
    # KV head.  Sampled tokens: selections bit-exact, outputs within tolerance
    wl = W.Workload(f"prompt_n{n}", 1, nq, nkv, np.array([n], np.int32), kind="sigma",
                    seed=2100 + n)
    case = paged.fill_cache(wl, 0, DEV)
    g = W.device_generator(DEV, 7 + n)
    q = torch.randn((n, nq, wl.hd), generator=g, device=DEV)
    out = torch.empty_like(q)
    sel = torch.full((n, nq, 32), -7, dtype=torch.int32, device=DEV)
    q_off = torch.tensor([0, n], dtype=torch.int32, device=DEV)
    ws = kq8.new_workspace(kq8.kq8_sparse_prefill_workspace_bytes(n, nq, nkv, n, 32, 32), DEV)
    kq8.kq8_sparse_prefill_attn(out, q, case.cache, case.page_table, case.seq_lens, q_off, n, n,
                                wl.scale, 32, 32, 8, ws, sel_blocks=sel)
    assert kq8.kq8_read_status(ws) == 0
    got, gsel, qh = out.cpu().numpy(), sel.cpu().numpy(), q.cpu().numpy()
    K, V = case.device_kv(0, 0, n)
    k8, ks = oracle.kv_quantize_rows(K.cpu().numpy())
    v8, vs = oracle.kv_quantize_rows(V.cpu().numpy())
    rows = np.unique(np.concatenate([[0, 63, 64, 65, 1024, n - 1],
                                     np.random.default_rng(n).integers(0, n, 18)]))
    for i in rows:
        p = int(i) + 1
        ref, rsel = oracle.prefill_batch(qh[i:i + 1], [1], [k8[:p]], [ks[:p]], [v8[:p]], [vs[:p]],
                                         wl.scale, sparse=True, block=32, topk=32, probe=8)
        assert np.array_equal(gsel[i:i + 1], rsel), f"selection of token {i}"
        assert_out_close(got[i:i + 1], ref, f"sparse token {i}")
