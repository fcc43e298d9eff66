"""Pins for the oracle's batched prefill (article 10-1 §1: nb new tokens score
against the whole history, O(nb*n); §2: the prefill gate picks the exact or the
block-sparse batched kernel).  The pages give no formula for the batched kernel;
the oracle's reading is that query i of a sequence with nb new tokens sits at
position p = n - nb + i, sees tokens 0..p, and is computed like one decode
query over that prefix.  The pins below check it against a dense masked-matrix
softmax in fp64, causality, and the decode special case."""
import math

import numpy as np
import pytest
import scipy.special

import oracle

F32_INV127 = np.float32(1.0) / np.float32(127.0)
SCALE = np.float32(1 / math.sqrt(128))


def _layer(lens, nkv, seed):
    rng = np.random.default_rng(seed)
    k8s, kss, v8s, vss = [], [], [], []
    for n in lens:
        k8, ks = oracle.kv_quantize_rows(rng.standard_normal((n, nkv, 128)).astype(np.float32)
                                         * np.float32(1.7))
        v8, vs = oracle.kv_quantize_rows(rng.standard_normal((n, nkv, 128)).astype(np.float32))
        k8s.append(k8)
        kss.append(ks)
        v8s.append(v8)
        vss.append(vs)
    return k8s, kss, v8s, vss


def _dense_masked_f64(q, q_lens, k8s, kss, v8s, vss, nq, nkv):
    """Whole score matrix per (sequence, query head) in fp64 over the
    dequantised operands, a causal mask on it, a row softmax, one matmul."""
    outs = []
    G = nq // nkv
    r0 = 0
    for b, nb in enumerate(q_lens):
        n = k8s[b].shape[0]
        o = np.zeros((nb, nq, 128))
        pos = np.arange(n - nb, n)
        mask = np.arange(n)[None, :] <= pos[:, None]            # [nb, n]
        for h in range(nq):
            kh = h // G
            Qd = np.stack([np.repeat(oracle.quantize_q(q[r0 + i, h])[1], 32)
                           * oracle.quantize_q(q[r0 + i, h])[0] for i in range(nb)]).astype(np.float64)
            Kd = k8s[b][:, kh].astype(np.float64) * (kss[b][:, kh] * F32_INV127)[:, None]
            Vd = v8s[b][:, kh].astype(np.float64) * (vss[b][:, kh] * F32_INV127)[:, None]
            S = (Qd @ Kd.T) * float(SCALE)
            S = np.where(mask, S, -np.inf)
            o[:, h] = scipy.special.softmax(S, axis=1) @ Vd
        outs.append(o)
        r0 += nb
    return np.concatenate(outs)


@pytest.mark.parametrize("lens,q_lens,nq,nkv", [
    ([70, 33, 130], [5, 33, 64], 4, 2),
    ([1, 40], [1, 1], 2, 1),
    ([97], [97], 8, 2),
])
def test_prefill_equals_dense_causal_softmax(lens, q_lens, nq, nkv):
    k8s, kss, v8s, vss = _layer(lens, nkv, seed=sum(lens))
    T = sum(q_lens)
    q = np.random.default_rng(T).standard_normal((T, nq, 128)).astype(np.float32)
    out = oracle.prefill_batch(q, q_lens, k8s, kss, v8s, vss, SCALE)
    ref = _dense_masked_f64(q, q_lens, k8s, kss, v8s, vss, nq, nkv)
    err = np.abs(out - ref).max()
    assert err <= 3e-6 * max(1.0, np.abs(ref).max()), err


def test_prefill_is_causal_and_includes_its_own_token():
    lens, q_lens, nkv, nq = [80], [16], 2, 4
    k8s, kss, v8s, vss = _layer(lens, nkv, seed=7)
    q = np.random.default_rng(8).standard_normal((16, nq, 128)).astype(np.float32)
    base = oracle.prefill_batch(q, q_lens, k8s, kss, v8s, vss, SCALE)
    t = 71                                   # query i = 7 sits at position 64 + 7 = 71
    v8b = [v8s[0].copy()]
    v8b[0][t] = -v8b[0][t]                   # change token 71's values only
    got = oracle.prefill_batch(q, q_lens, k8s, kss, v8b, vss, SCALE)
    assert np.array_equal(got[:7], base[:7])            # queries before 71 never see it
    assert np.all(np.abs(got[7:] - base[7:]).max(axis=(1, 2)) > 0)   # 71 and later do


def test_single_new_token_is_decode():
    lens = [300, 64, 1]
    k8s, kss, v8s, vss = _layer(lens, 2, seed=9)
    q = np.random.default_rng(10).standard_normal((3, 4, 128)).astype(np.float32)
    pre = oracle.prefill_batch(q, [1, 1, 1], k8s, kss, v8s, vss, SCALE)
    dec = oracle.decode_batch(q, k8s, kss, v8s, vss, SCALE)
    assert np.array_equal(pre, dec)


def test_prefill_rows_equal_decodes_of_truncated_prefixes():
    # query i equals a decode of a sequence cut at its own position
    lens, nb = [45], 12
    k8s, kss, v8s, vss = _layer(lens, 1, seed=11)
    q = np.random.default_rng(12).standard_normal((nb, 2, 128)).astype(np.float32)
    pre = oracle.prefill_batch(q, [nb], k8s, kss, v8s, vss, SCALE)
    for i in range(nb):
        p = lens[0] - nb + i
        dec = oracle.decode_batch(q[i:i + 1], [k8s[0][:p + 1]], [kss[0][:p + 1]],
                                  [v8s[0][:p + 1]], [vss[0][:p + 1]], SCALE)
        assert np.array_equal(pre[i], dec[0])


def test_sparse_prefill_gate_and_full_cover():
    # block 32, k 32: a 200-token prompt has 7 blocks, so every query keeps all
    # its blocks and the sparse result equals the exact one bit for bit; queries
    # at n <= 64 take the exact path (no selection).
    lens, nb = [200], 200
    k8s, kss, v8s, vss = _layer(lens, 1, seed=13)
    q = np.random.default_rng(14).standard_normal((nb, 2, 128)).astype(np.float32)
    ex = oracle.prefill_batch(q, [nb], k8s, kss, v8s, vss, SCALE)
    sp, sel = oracle.prefill_batch(q, [nb], k8s, kss, v8s, vss, SCALE, sparse=True)
    assert np.array_equal(ex, sp)
    assert np.all(sel[:64] == -1)
    for i in range(64, nb):
        nblk = -(-(i + 1) // 32)
        assert list(sel[i, 0, :nblk]) == list(range(nblk)) and np.all(sel[i, 0, nblk:] == -1)


def test_prefill_rejects_more_queries_than_tokens():
    k8s, kss, v8s, vss = _layer([4], 1, seed=15)
    q = np.zeros((5, 1, 128), np.float32)
    with pytest.raises(ValueError):
        oracle.prefill_batch(q, [5], k8s, kss, v8s, vss, SCALE)
