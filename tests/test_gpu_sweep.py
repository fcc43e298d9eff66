"""Seeded random sweep over shapes through the C ABI against the oracle: batch,
GQA ratio, page size, ragged lengths (0 and 1 included), block-sparse knobs and
prefill splits drawn from a fixed seed, so that combinations the hand-written
cases do not name are exercised too.  Same contract as the other parity tests:
integer results bit-exact, fp32 outputs within min(1e-4, 1e-3 * max|out|)."""
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


def _draw(rng, max_len):
    nkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.integers(1, 9))
    B = int(rng.integers(1, 6))
    kv_bs = int(rng.choice([32, 64, 128]))
    lens = rng.integers(0, max_len, B)
    lens[rng.integers(0, B)] = int(rng.choice([0, 1, 31, 32, 33, max_len]))
    kind = str(rng.choice(["normal", "sigma", "student_t"]))
    return nkv, G, B, kv_bs, [int(x) for x in lens], kind


@pytest.mark.parametrize("case", range(8))
def test_sweep_exact_and_sparse_decode(case):
    rng = np.random.default_rng(900 + case)
    nkv, G, B, kv_bs, lens, kind = _draw(rng, 2500)
    block = int(rng.choice([32, 64, 96]))
    topk = int(rng.integers(1, 9))
    probe = int(rng.choice([1, 4, 8, block]))
    wl = W.custom(B, nkv * G, nkv, lens, kind=kind, seed=case, kv_bs=kv_bs, block=block,
                  topk=topk, probe=probe)
    q, Ks, Vs = host_inputs(wl)
    c = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q, pt_seed=case, extra_pages=2)
    out = torch.empty((B, wl.nq, 128), device=DEV)
    mx = max(1, wl.max_seq_len)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(B, wl.nq, nkv, mx), DEV)
    kq8.kq8_decode_attn(out, c.q, c.cache, c.page_table, c.seq_lens, mx, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    assert_out_close(out.cpu().numpy(), oracle_decode(wl, q, Ks, Vs), f"exact sweep {case}")

    wss = kq8.new_workspace(kq8.kq8_sparse_decode_workspace_bytes(B, wl.nq, nkv, mx, block, topk),
                            DEV)
    sel = torch.full((B, wl.nq, topk), -7, dtype=torch.int32, device=DEV)
    kq8.kq8_sparse_decode_attn(out, c.q, c.cache, c.page_table, c.seq_lens, mx, wl.scale, block,
                               topk, probe, wss, sel_blocks=sel)
    assert kq8.kq8_read_status(wss) == 0
    ref, rsel = oracle_decode(wl, q, Ks, Vs, sparse=True)
    assert np.array_equal(sel.cpu().numpy(), rsel), f"sparse selection sweep {case}"
    assert_out_close(out.cpu().numpy(), ref, f"sparse sweep {case}")


@pytest.mark.parametrize("case", range(6))
def test_sweep_prefill(case):
    rng = np.random.default_rng(950 + case)
    nkv, G, B, kv_bs, lens, kind = _draw(rng, 700)
    q_lens = [int(rng.integers(0, n + 1)) for n in lens]
    wl = W.custom(B, nkv * G, nkv, lens, kind=kind, seed=case, kv_bs=kv_bs)
    _, Ks, Vs = host_inputs(wl)
    c = paged.fill_from_host(wl, Ks, Vs, DEV, pt_seed=case)
    T = sum(q_lens)
    qp = np.random.default_rng(case).standard_normal((T, wl.nq, 128)).astype(np.float32)
    q_off = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    out = torch.full((T, wl.nq, 128), float("nan"), device=DEV)
    mx, mq = max(1, wl.max_seq_len), max(q_lens)
    ws = kq8.new_workspace(kq8.kq8_prefill_workspace_bytes(B, wl.nq, nkv, mx, mq), DEV)
    kq8.kq8_prefill_attn(out, torch.tensor(qp, device=DEV), c.cache, c.page_table, c.seq_lens,
                         torch.tensor(q_off, device=DEV), mx, mq, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref = oracle.prefill_batch(qp, q_lens, k8s, kss, v8s, vss, wl.scale, kv_bs=kv_bs)
    assert_out_close(out.cpu().numpy(), ref, f"prefill sweep {case} G={G} kv_bs={kv_bs}")
