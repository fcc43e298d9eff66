"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- exact rational arithmetic, brute force on tiny inputs, closed
forms, invariants, textbook routines (scipy softmax), or the numbers the pages
print.  A plausible slip in the oracle (a dropped scale, a wrong sign or index,
rounding instead of truncation, a transposed operand) fails at least one.

Sources: article 9-2 (flash_attn_single_q_q8_neon) §1-§4, article 9-3 (q8 KV
precision comparison) §1-§4, article 10-1 (why long context must be sparse)
§1-§2.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from query_decode_attention_gb300 import workloads as W

F32_INV127 = np.float32(1.0) / np.float32(127.0)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _round_half_away(fr: Fraction) -> int:
    s = 1 if fr >= 0 else -1
    a = abs(fr)
    f = a.numerator // a.denominator
    return s * (f + (1 if a - f >= Fraction(1, 2) else 0))


def _trunc(fr: Fraction) -> int:
    a = abs(fr)
    return (1 if fr >= 0 else -1) * (a.numerator // a.denominator)


# ---------------------------------------------------------------------------
# Write path (article 9-3 §2)
# ---------------------------------------------------------------------------

def test_append_hand_example():
    # Row [2, 1, -1, -0.5, 0 ...]: max_abs 2, step d = 2 * fl(1/127).  Because
    # fl(1/127) lies just below 1/127, 1/d is just above 63.5 -> 64, and
    # 0.5/d = 31.75... -> 32.  The max element maps to 127.
    x = np.zeros(128, np.float32)
    x[:4] = [2.0, 1.0, -1.0, -0.5]
    x[77] = -2.0  # ties in |x| keep max_abs = 2
    c, m = oracle.kv_quantize_rows(x[None])
    assert m[0] == np.float32(2.0)
    assert list(c[0, :4]) == [127, 64, -64, -32]
    assert c[0, 77] == -127
    assert not c[0, 4:77].any() and not c[0, 78:].any()


def test_append_matches_exact_rational_rounding():
    rng = np.random.default_rng(11)
    rows = rng.standard_normal((64, 128)).astype(np.float32)
    rows *= rng.choice([1e-30, 1e-3, 1.0, 37.0, 1e20], size=(64, 1)).astype(np.float32)
    codes, maxima = oracle.kv_quantize_rows(rows)
    near_ties = 0
    for r in range(rows.shape[0]):
        m = np.abs(rows[r]).max()
        assert maxima[r] == m
        d = Fraction(float(np.float32(m) * F32_INV127))
        for i in range(128):
            ratio = Fraction(float(rows[r, i])) / d
            exp = max(-127, min(127, _round_half_away(ratio)))
            if codes[r, i] != exp:
                # only where fp32 division rounds across a half-integer
                frac = abs(ratio) - math.floor(abs(ratio))
                assert abs(frac - Fraction(1, 2)) < abs(ratio) * Fraction(1, 2**22), (r, i)
                near_ties += 1
    assert near_ties <= 2


def test_append_error_bound_and_max_maps_to_127():
    rng = np.random.default_rng(12)
    rows = (rng.standard_t(3, (200, 128)) * rng.uniform(0.01, 100, (200, 1))).astype(np.float32)
    codes, maxima = oracle.kv_quantize_rows(rows)
    d = (maxima * F32_INV127).astype(np.float64)
    err = np.abs(rows.astype(np.float64) - codes.astype(np.float64) * d[:, None])
    assert np.all(err <= d[:, None] * 0.5 * (1 + 2**-20))
    am = np.abs(rows).argmax(1)
    top = codes[np.arange(200), am]
    assert np.all(np.abs(top) == 127)
    assert np.all(np.sign(top) == np.sign(rows[np.arange(200), am]))
    assert codes.min() >= -127 and codes.max() <= 127


def test_append_power_of_two_scaling_invariance():
    # article 9-3 §4: per-row scaling makes the codes independent of the row's
    # amplitude; for a power-of-two factor this holds bit for bit.
    rng = np.random.default_rng(13)
    rows = rng.standard_normal((32, 128)).astype(np.float32)
    c0, m0 = oracle.kv_quantize_rows(rows)
    for k in (-5, 3, 17):
        c1, m1 = oracle.kv_quantize_rows(rows * np.float32(2.0**k))
        assert np.array_equal(c0, c1)
        assert np.array_equal(m1, m0 * np.float32(2.0**k))


def test_append_zero_row_and_permutation():
    c, m = oracle.kv_quantize_rows(np.zeros((1, 128), np.float32))
    assert m[0] == 0 and not c.any()
    rng = np.random.default_rng(14)
    x = rng.standard_normal(128).astype(np.float32)
    p = rng.permutation(128)
    c0, _ = oracle.kv_quantize_rows(x[None])
    c1, _ = oracle.kv_quantize_rows(x[p][None])
    assert np.array_equal(c0[0][p], c1[0])


def test_dequant_is_code_times_step():
    c = np.array([[127, -64, 3, 0] + [0] * 124], np.int8)
    m = np.array([2.0], np.float32)
    d = oracle.dequant(c, m)
    step = np.float32(2.0) * F32_INV127
    assert d[0, 0] == np.float32(127) * step and d[0, 1] == np.float32(-64) * step
    assert d[0, 3] == 0


# ---------------------------------------------------------------------------
# Q quantisation (article 9-2 §2 segment 1)
# ---------------------------------------------------------------------------

def test_quantize_q_hand_example_truncates():
    q = np.zeros(128, np.float32)
    q[0:4] = [1.0, 0.5, -0.5, 0.25]       # block 0, max 1: 127/1 = 127 exactly
    q[32] = 4.0                            # block 1, max 4: 127/4 = 31.75
    q[33] = 1.0                            # 1 * 31.75 -> 31
    q[34] = -3.0                           # -95.25 -> -95
    qi, qsc = oracle.quantize_q(q)
    # truncation, not rounding: 0.5 * 127 = 63.5 -> 63, 0.25*127 = 31.75 -> 31
    assert list(qi[0:4]) == [127, 63, -63, 31]
    assert list(qi[32:35]) == [127, 31, -95]
    assert qsc[0] == np.float32(1.0) * F32_INV127
    assert qsc[1] == np.float32(4.0) * F32_INV127
    # blocks 2 and 3 are all zero: qm < 1e-6 -> 1, codes 0, qsc = 1/127
    assert qsc[2] == F32_INV127 and qsc[3] == F32_INV127
    assert not qi[64:].any()


def test_quantize_q_exact_rational_truncation():
    rng = np.random.default_rng(21)
    for trial in range(20):
        q = (rng.standard_normal(128) * rng.choice([1e-7, 1e-3, 1.0, 50.0])).astype(np.float32)
        qi, qsc = oracle.quantize_q(q)
        for b in range(4):
            blk = q[b * 32:(b + 1) * 32]
            qm = np.float32(np.abs(blk).max())
            if qm < np.float32(1e-6):
                qm = np.float32(1.0)
            assert qsc[b] == qm * F32_INV127
            iq = Fraction(float(np.float32(127.0) / qm))
            for i in range(32):
                v = Fraction(float(blk[i])) * iq
                exp = max(-128, min(127, _trunc(v)))
                got = int(qi[b * 32 + i])
                if got != exp:
                    # fp32 product rounding onto/off an integer
                    assert abs(v - round(v)) < abs(v) * Fraction(1, 2**22) + Fraction(1, 2**40)
                assert abs(got) <= 127
                assert got == 0 or np.sign(got) == np.sign(blk[i])


def test_quantize_q_blocks_are_independent():
    rng = np.random.default_rng(22)
    q = rng.standard_normal(128).astype(np.float32)
    qi0, s0 = oracle.quantize_q(q)
    q2 = q.copy()
    q2[64:96] *= np.float32(100.0)
    qi1, s1 = oracle.quantize_q(q2)
    for b in (0, 1, 3):
        assert np.array_equal(qi0[b * 32:(b + 1) * 32], qi1[b * 32:(b + 1) * 32])
        assert s0[b] == s1[b]
    assert s1[2] != s0[2]


# ---------------------------------------------------------------------------
# int32 block dots and the score (article 9-2 §2 segment 2, point 1)
# ---------------------------------------------------------------------------

def test_block_dots_brute_force_int64():
    rng = np.random.default_rng(31)
    for _ in range(50):
        a = rng.integers(-127, 128, 128).astype(np.int8)
        k = rng.integers(-127, 128, 128).astype(np.int8)
        d = oracle.block_dots(a, k)
        ref = (a.astype(np.int64).reshape(4, 32) * k.astype(np.int64).reshape(4, 32)).sum(1)
        assert np.array_equal(d.astype(np.int64), ref)
    full = np.full(128, 127, np.int8)
    assert list(oracle.block_dots(full, full)) == [516128] * 4
    assert list(oracle.block_dots(full, -full)) == [-516128] * 4


def test_score_against_exact_product():
    rng = np.random.default_rng(32)
    for _ in range(200):
        dots = rng.integers(-516128, 516129, 4).astype(np.int32)
        qsc = rng.uniform(1e-4, 1.0, 4).astype(np.float32)
        kst = np.float32(rng.uniform(0.01, 50.0))
        scale = np.float32(1 / math.sqrt(128))
        s = oracle.score(dots, qsc, kst, scale)
        exact = (sum(Fraction(int(d)) * Fraction(float(c)) for d, c in zip(dots, qsc))
                 * Fraction(float(kst * F32_INV127)) * Fraction(float(scale)))
        bound = sum(abs(Fraction(int(d)) * Fraction(float(c))) for d, c in zip(dots, qsc)) \
            * Fraction(float(kst * F32_INV127)) * Fraction(float(scale)) * Fraction(6, 2**24)
        assert abs(Fraction(float(s)) - exact) <= bound
    # doubling the stored K scale doubles the score exactly (K scale is used)
    d = np.array([1000, -2000, 30, 7], np.int32)
    c = np.array([0.01, 0.02, 0.03, 0.04], np.float32)
    assert oracle.score(d, c, 4.0, 0.5) == 2 * oracle.score(d, c, 2.0, 0.5)
    assert oracle.score(d, c, 2.0, 0.5) == 2 * oracle.score(d, c, 2.0, 0.25)


# ---------------------------------------------------------------------------
# One-pass online softmax (article 9-2 §1-§4)
# ---------------------------------------------------------------------------

def _cache(n, nkv=2, seed=0, kv_bs=32, scale_k=1.0, shuffle=None):
    rng = np.random.default_rng(seed)
    K = (rng.standard_normal((n, nkv, 128)) * scale_k).astype(np.float32)
    V = rng.standard_normal((n, nkv, 128)).astype(np.float32)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    return oracle.SeqCache(k8, ks, v8, vs, kv_bs=kv_bs, shuffle_seed=shuffle), (k8, ks, v8, vs)


def _textbook(q, k8, ks, v8, vs, kh, scale, tokens=None):
    """softmax(Q' K'^T * scale) V' in float64 via scipy, on dequantised data."""
    qi, qsc = oracle.quantize_q(q)
    qd = (qi.astype(np.float64).reshape(4, 32) * qsc.astype(np.float64)[:, None]).reshape(128)
    idx = np.arange(k8.shape[0]) if tokens is None else np.asarray(tokens)
    kst = (ks[idx, kh] * F32_INV127).astype(np.float64)
    vst = (vs[idx, kh] * F32_INV127).astype(np.float64)
    Kd = k8[idx, kh].astype(np.float64) * kst[:, None]
    Vd = v8[idx, kh].astype(np.float64) * vst[:, None]
    p = scipy.special.softmax(Kd @ qd * float(scale))
    return p @ Vd


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 257, 1000])
def test_one_pass_equals_textbook_softmax(n):
    cache, (k8, ks, v8, vs) = _cache(n, seed=n)
    q = np.random.default_rng(100 + n).standard_normal(128).astype(np.float32)
    scale = np.float32(1 / math.sqrt(128))
    for kh in (0, 1):
        out = oracle.attn_single_q(q, cache, kh, scale)
        ref = _textbook(q, k8, ks, v8, vs, kh, scale)
        tol = 2e-6 * np.abs(ref).max() + 1e-7 * math.sqrt(n)
        assert np.abs(out - ref).max() <= max(tol, 1e-6), (n, kh)
        two = oracle.attn_two_pass_f64(q, cache, kh, scale)
        assert np.abs(two - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_one_pass_heads_are_not_mixed():
    cache, (k8, ks, v8, vs) = _cache(300, nkv=3, seed=5)
    q = np.random.default_rng(6).standard_normal(128).astype(np.float32)
    outs = [oracle.attn_single_q(q, cache, kh, 0.1) for kh in range(3)]
    for kh in range(3):
        ref = _textbook(q, k8, ks, v8, vs, kh, np.float32(0.1))
        assert np.abs(outs[kh] - ref).max() < 1e-5
    assert np.abs(outs[0] - outs[1]).max() > 1e-2


def test_running_max_trace_and_visit_count():
    # article 9-2 §4: the loop visits exactly seq_len tokens and M never decreases
    cache, (k8, ks, v8, vs) = _cache(500, seed=7, scale_k=3.0)
    q = np.random.default_rng(8).standard_normal(128).astype(np.float32)
    out, tr, nv = oracle.attn_single_q(q, cache, 1, 0.088, trace=True)
    assert nv == 500
    assert np.all(np.diff(tr) >= 0)
    qi, qsc = oracle.quantize_q(q)
    s = np.array([oracle.score(oracle.block_dots(qi, k8[t, 1]), qsc, ks[t, 1], 0.088)
                  for t in range(500)], np.float32)
    assert np.array_equal(tr, np.maximum.accumulate(s))


def test_single_token_is_dequantised_v():
    cache, (k8, ks, v8, vs) = _cache(1, seed=9)
    q = np.random.default_rng(10).standard_normal(128).astype(np.float32)
    out = oracle.attn_single_q(q, cache, 0, 0.1)
    assert np.array_equal(out, v8[0, 0].astype(np.float32) * (vs[0, 0] * F32_INV127))


def test_identical_keys_give_mean_of_values():
    n = 200
    rng = np.random.default_rng(15)
    krow = rng.standard_normal(128).astype(np.float32)
    K = np.broadcast_to(krow, (n, 1, 128)).copy()
    V = rng.standard_normal((n, 1, 128)).astype(np.float32)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    cache = oracle.SeqCache(k8, ks, v8, vs)
    out = oracle.attn_single_q(rng.standard_normal(128).astype(np.float32), cache, 0, 0.3)
    mean = (v8[:, 0].astype(np.float64) * (vs[:, 0] * F32_INV127)[:, None]).mean(0)
    assert np.abs(out - mean).max() < 1e-5


def test_empty_sequence_gives_zero():
    cache, _ = _cache(0, seed=1)
    out = oracle.attn_single_q(np.ones(128, np.float32), cache, 0, 0.1)
    assert not out.any()


def test_wide_score_range_stays_finite_and_exact():
    cache, (k8, ks, v8, vs) = _cache(400, seed=16, scale_k=40.0)
    q = (np.random.default_rng(17).standard_normal(128) * 5).astype(np.float32)
    out = oracle.attn_single_q(q, cache, 0, 0.088)
    ref = _textbook(q, k8, ks, v8, vs, 0, np.float32(0.088))
    assert np.all(np.isfinite(out))
    assert np.abs(out - ref).max() < 1e-5 * max(1, np.abs(ref).max())


def test_block_pointer_indirection_and_kv_bs():
    # the same rows behind shuffled block pointers, or other block sizes,
    # give bit-identical results (article 9-2 §2 point 2, block/row split)
    _, (k8, ks, v8, vs) = _cache(333, seed=18)
    q = np.random.default_rng(19).standard_normal(128).astype(np.float32)
    base = oracle.attn_single_q(q, oracle.SeqCache(k8, ks, v8, vs, kv_bs=32), 1, 0.1)
    for kv_bs, sh in ((32, 5), (16, None), (64, 3), (7, 1)):
        o = oracle.attn_single_q(q, oracle.SeqCache(k8, ks, v8, vs, kv_bs=kv_bs, shuffle_seed=sh),
                                 1, 0.1)
        assert np.array_equal(o, base)


def test_token_order_only_changes_rounding():
    cache, (k8, ks, v8, vs) = _cache(300, seed=20)
    q = np.random.default_rng(21).standard_normal(128).astype(np.float32)
    perm = np.random.default_rng(22).permutation(300).astype(np.int32)
    a = oracle.attn_single_q(q, cache, 0, 0.1)
    b = oracle.attn_single_q(q, cache, 0, 0.1, tokens=perm)
    assert np.abs(a - b).max() < 1e-5 * np.abs(a).max()


def test_batch_driver_gqa_mapping_and_threads():
    wl = W.custom(3, 8, 2, [40, 1, 129], seed=3)
    q = W.host_q(wl)
    k8s, kss, v8s, vss = [], [], [], []
    for b in range(wl.B):
        K, V = W.host_kv(wl, b)
        k8, ks = oracle.kv_quantize_rows(K)
        v8, vs = oracle.kv_quantize_rows(V)
        k8s.append(k8); kss.append(ks); v8s.append(v8); vss.append(vs)
    out1 = oracle.decode_batch(q, k8s, kss, v8s, vss, wl.scale, nthreads=1)
    out4 = oracle.decode_batch(q, k8s, kss, v8s, vss, wl.scale, nthreads=4)
    assert np.array_equal(out1, out4)
    for b in range(wl.B):
        c = oracle.SeqCache(k8s[b], kss[b], v8s[b], vss[b])
        for h in range(wl.nq):
            assert np.array_equal(out1[b, h], oracle.attn_single_q(q[b, h], c, h // 4, wl.scale))


# ---------------------------------------------------------------------------
# Precision experiment (article 9-3 §1-§4)
# ---------------------------------------------------------------------------

def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, *v = line.split()
                vals[k] = [float(x) for x in v]
    return vals


def test_precision_experiment_magnitude():
    g = _golden("precision_fp32_vs_q8_kv.txt")
    n, hd = int(g["seq_len"][0]), int(g["head_dim"][0])
    wl = W.tiny()
    assert (wl.seq_lens[0], wl.hd) == (n, hd)
    q = W.host_q(wl)[0]
    K, V = W.host_kv(wl, 0)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    Kd = oracle.dequant(k8, ks)
    Vd = oracle.dequant(v8, vs)
    cache = oracle.SeqCache(k8, ks, v8, vs)
    scale = 1 / math.sqrt(hd)
    d_kv, d_full = [], []
    for h in range(wl.nq):
        kh = h // wl.G
        ref = oracle.attn_ref_f64(q[h], K[:, kh], V[:, kh], scale)
        kvq = oracle.attn_ref_f64(q[h], Kd[:, kh], Vd[:, kh], scale)
        full = oracle.attn_single_q(q[h], cache, kh, np.float32(scale))
        d_kv.append(np.abs(kvq - ref))
        d_full.append(np.abs(full - ref))
    d_kv, d_full = np.array(d_kv), np.array(d_full)
    page_max, page_mean = g["max_abs_dout"][0], g["mean_abs_dout"][0]
    print(f"\n[article 9-3 §3] page: max|dout| {page_max} mean {page_mean}; "
          f"KV-only here: max {d_kv.max():.5f} mean {d_kv.mean():.5f}; "
          f"with Q truncated to int8: max {d_full.max():.5f} mean {d_full.mean():.5f}; "
          f"avg K step {np.mean(ks * F32_INV127):.5f} (page {g['avg_k_scale'][0]})")
    # acceptance band: the same order as the page's ~0.01, never above 0.02
    assert d_kv.max() <= 0.02 and d_full.max() <= 0.02
    assert d_full.max() >= 0.1 * page_max
    assert 0.005 < float(np.mean(ks * F32_INV127)) < 0.05


def test_value_error_is_a_convex_combination():
    # K exact, V quantised: out_q - out_f = sum_t p_t (v'_t - v_t), so each
    # component differs by at most max_t |v'_t - v_t| <= max_t step_t / 2.
    rng = np.random.default_rng(40)
    K = rng.standard_normal((256, 128)).astype(np.float32)
    V = rng.standard_normal((256, 128)).astype(np.float32)
    q = rng.standard_normal(128).astype(np.float32)
    v8, vs = oracle.kv_quantize_rows(V)
    Vd = oracle.dequant(v8, vs)
    a = oracle.attn_ref_f64(q, K, V, 1 / math.sqrt(128))
    b = oracle.attn_ref_f64(q, K, Vd, 1 / math.sqrt(128))
    per_comp = np.abs(Vd.astype(np.float64) - V).max(0)
    assert np.all(np.abs(a - b) <= per_comp + 1e-12)
    assert per_comp.max() <= (vs * F32_INV127).max() / 2 * (1 + 1e-6)


def test_amplitude_scaling_keeps_relative_error():
    # article 9-3 §4: amplifying V leaves the relative error unchanged; for a
    # factor 4 (power of two) exactly, for 3 approximately.
    rng = np.random.default_rng(41)
    K = rng.standard_normal((256, 128)).astype(np.float32)
    V = rng.standard_normal((256, 128)).astype(np.float32)
    q = rng.standard_normal(128).astype(np.float32)
    s = 1 / math.sqrt(128)

    def rel(Vx):
        v8, vs = oracle.kv_quantize_rows(Vx)
        a = oracle.attn_ref_f64(q, K, Vx, s)
        b = oracle.attn_ref_f64(q, K, oracle.dequant(v8, vs), s)
        return np.abs(a - b).max() / np.abs(a).max()

    r1, r4, r3 = rel(V), rel(V * np.float32(4)), rel(V * np.float32(3))
    assert abs(r4 - r1) <= 1e-12 * r1
    assert 0.8 < r3 / r1 < 1.25


# ---------------------------------------------------------------------------
# Block-sparse (article 10-1 §1-§2, with the oracle's stated readings)
# ---------------------------------------------------------------------------

def test_sparse_gate_is_exact_path():
    for n in (1, 33, 64):
        cache, _ = _cache(n, seed=50 + n)
        q = np.random.default_rng(n).standard_normal(128).astype(np.float32)
        out, sel, used = oracle.sparse_attn_head(q, cache, 0, 0.1, 32, 32, 8)
        assert not used and np.all(sel == -1)
        assert np.array_equal(out, oracle.attn_single_q(q, cache, 0, 0.1))
    cache, _ = _cache(65, seed=99)
    _, sel, used = oracle.sparse_attn_head(np.ones(128, np.float32), cache, 0, 0.1, 32, 32, 8)
    assert used and list(sel[:3]) == [0, 1, 2] and np.all(sel[3:] == -1)


def test_sparse_keeps_everything_when_k_covers_all_blocks():
    # n = 506, block 32 -> 16 blocks <= k = 32: nothing can be pruned
    cache, _ = _cache(506, seed=60)
    q = np.random.default_rng(61).standard_normal(128).astype(np.float32)
    out, sel, used = oracle.sparse_attn_head(q, cache, 1, 0.1, 32, 32, 8)
    assert used and list(sel[:16]) == list(range(16)) and np.all(sel[16:] == -1)
    assert np.array_equal(out, oracle.attn_single_q(q, cache, 1, 0.1))


def test_probe_positions_and_max_fusion():
    n, block, probe = 640, 32, 8
    cache, (k8, ks, v8, vs) = _cache(n, nkv=1, seed=70)
    q = np.random.default_rng(71).standard_normal(128).astype(np.float32)
    qi, qsc = oracle.quantize_q(q)
    s = np.array([oracle.score(oracle.block_dots(qi, k8[t, 0]), qsc, ks[t, 0], 0.1)
                  for t in range(n)], np.float32)
    bs = oracle.probe_block_scores(q, cache, 0, 0.1, block, probe)
    # probe p of block j at j*32 + 4p
    ref = np.array([s[j * 32:(j + 1) * 32:4].max() for j in range(n // 32)], np.float32)
    assert np.array_equal(bs, ref)
    full = oracle.probe_block_scores(q, cache, 0, 0.1, block, block)
    assert np.array_equal(full, s.reshape(-1, 32).max(1))
    # a ragged last block only probes tokens < n
    cache2 = oracle.SeqCache(k8[:613], ks[:613], v8[:613], vs[:613])
    bs2 = oracle.probe_block_scores(q, cache2, 0, 0.1, block, probe)
    assert bs2[-1] == s[608:613:4].max()


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(80)
    for trial in range(200):
        nblk = int(rng.integers(1, 90))
        k = int(rng.integers(1, 40))
        sc = rng.integers(-5, 6, nblk).astype(np.float32) * np.float32(0.5)
        got = oracle.topk_blocks(sc, k)
        order = sorted(range(nblk), key=lambda j: (-float(sc[j]), j))
        assert list(got) == sorted(order[:k])


def test_sparse_output_is_one_pass_over_kept_blocks():
    n = 1000
    cache, (k8, ks, v8, vs) = _cache(n, seed=90)
    q = np.random.default_rng(91).standard_normal(128).astype(np.float32)
    out, sel, used = oracle.sparse_attn_head(q, cache, 0, 0.1, 32, 4, 8)
    assert used and np.all(sel >= 0) and np.all(np.diff(sel) > 0)
    bs = oracle.probe_block_scores(q, cache, 0, 0.1, 32, 8)
    assert list(sel) == sorted(sorted(range(len(bs)), key=lambda j: (-bs[j], j))[:4])
    toks = np.concatenate([np.arange(j * 32, min((j + 1) * 32, n)) for j in sel]).astype(np.int32)
    ref = _textbook(q, k8, ks, v8, vs, 0, np.float32(0.1), tokens=toks)
    assert np.abs(out - ref).max() < 1e-5 * max(1, np.abs(ref).max())


def test_planted_blocks_are_recalled():
    wl = W.sparse_planted(4059, B=2)
    q = W.host_q(wl)
    for b in range(wl.B):
        K, V = W.host_kv(wl, b, q=q)
        k8, ks = oracle.kv_quantize_rows(K)
        v8, vs = oracle.kv_quantize_rows(V)
        cache = oracle.SeqCache(k8, ks, v8, vs)
        for h in range(wl.nq):
            kh = h // wl.G
            _, sel, used = oracle.sparse_attn_head(q[b, h], cache, kh, wl.scale, wl.block,
                                                   wl.topk, wl.probe)
            assert used
            assert set(sel.tolist()) == set(W.planted_blocks(wl, b, kh).tolist())


# ---------------------------------------------------------------------------
# Streaming form (article 9-2 §3): KV fed in pieces through a carried state
# ---------------------------------------------------------------------------

def test_streaming_in_pieces_equals_one_call():
    # the carried (M, S, acc) continues the same loop, so any split of the
    # sequence gives the one-call result bit for bit
    n = 700
    cache, (k8, ks, v8, vs) = _cache(n, seed=95)
    q = np.random.default_rng(96).standard_normal(128).astype(np.float32)
    one = oracle.attn_single_q(q, cache, 1, 0.1)
    for cuts in ([0, n], [0, 1, 2, n], [0, 31, 32, 33, 400, 699, n], [0, 350, 350, n]):
        st = oracle.StreamState()
        for a, b in zip(cuts[:-1], cuts[1:]):
            oracle.attn_stream(st, q, cache, 1, 0.1, a, b)
        assert np.array_equal(st.output(), one), cuts
    # the state itself is the textbook pair: acc / S is softmax-weighted V
    ref = _textbook(q, k8, ks, v8, vs, 1, np.float32(0.1))
    assert np.abs(one - ref).max() < 1e-5 * np.abs(ref).max()


def test_streaming_empty_state_and_empty_pieces():
    cache, _ = _cache(10, seed=97)
    q = np.ones(128, np.float32)
    st = oracle.StreamState()
    assert not st.output().any()
    oracle.attn_stream(st, q, cache, 0, 0.1, 5, 5)  # empty piece changes nothing
    assert st.S[0] == 0 and st.M[0] == np.float32(-1e9)


# ---------------------------------------------------------------------------
# Shared selection per KV head (the variant that lets a KV head's G query heads
# read the same blocks; its reading is the oracle's: max of their block scores)
# ---------------------------------------------------------------------------

def test_shared_selection_is_topk_of_the_heads_max_and_one_pass_each():
    n, block, topk, probe = 700, 32, 5, 8
    cache, _ = _cache(n, nkv=1, seed=80)
    q = np.random.default_rng(81).standard_normal((4, 128)).astype(np.float32)
    out, sel, used = oracle.sparse_attn_group(q, cache, 0, 0.1, block, topk, probe)
    assert used
    scores = np.max([oracle.probe_block_scores(q[g], cache, 0, 0.1, block, probe)
                     for g in range(4)], axis=0)
    want = sorted(sorted(range(len(scores)), key=lambda j: (-scores[j], j))[:topk])
    assert list(sel) == want
    toks = np.concatenate([np.arange(j * block, min((j + 1) * block, n)) for j in want])
    for g in range(4):
        assert np.array_equal(out[g], oracle.attn_single_q(q[g], cache, 0, 0.1, tokens=toks))


def test_shared_selection_one_head_equals_per_head_and_gate():
    cache, _ = _cache(500, nkv=1, seed=82)
    q = np.random.default_rng(83).standard_normal((1, 128)).astype(np.float32)
    o1, s1, _ = oracle.sparse_attn_group(q, cache, 0, 0.1, 32, 4, 8)
    o2, s2, _ = oracle.sparse_attn_head(q[0], cache, 0, 0.1, 32, 4, 8)
    assert np.array_equal(o1[0], o2) and np.array_equal(s1, s2)
    small, _ = _cache(64, nkv=1, seed=84)
    q2 = np.random.default_rng(85).standard_normal((2, 128)).astype(np.float32)
    o3, s3, used = oracle.sparse_attn_group(q2, small, 0, 0.1, 32, 4, 8)
    assert not used and np.all(s3 == -1)
    assert np.array_equal(o3[1], oracle.attn_single_q(q2[1], small, 0, 0.1))


def test_shared_selection_batch_driver_matches_group_calls():
    lens = [400, 50]
    rng = np.random.default_rng(86)
    caches, raw = [], []
    for b, n in enumerate(lens):
        c, r = _cache(n, nkv=2, seed=87 + b)
        caches.append(c)
        raw.append(r)
    q = rng.standard_normal((2, 4, 128)).astype(np.float32)
    out, sel = oracle.decode_batch_shared(q, [r[0] for r in raw], [r[1] for r in raw],
                                          [r[2] for r in raw], [r[3] for r in raw], 0.1,
                                          block=32, topk=3, probe=8)
    for b in range(2):
        for kh in range(2):
            o, s, _ = oracle.sparse_attn_group(q[b, 2 * kh:2 * kh + 2], caches[b], kh, 0.1, 32, 3, 8)
            assert np.array_equal(out[b, 2 * kh:2 * kh + 2], o)
            assert np.array_equal(sel[b, 2 * kh], s) and np.array_equal(sel[b, 2 * kh + 1], s)


# ---------------------------------------------------------------------------
# exact-sum reference (article 9-2 §3: the one pass and the two passes are the
# same computation, differing only by rounding)
# ---------------------------------------------------------------------------

def _integer_case(n, seed):
    """q, K, V whose quantisation is the identity: every 32-element block of q
    and every K/V row holds a +-127 (so qsc = stored max * (1/127) = 1 and the
    codes are the integers themselves); the other entries are small integers."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-2, 3, 128).astype(np.float32)
    q[0::32] = 127.0
    K = rng.integers(-2, 3, (n, 1, 128)).astype(np.float32)
    K[:, 0, 1::32] = 127.0                      # a +-127 where q is small
    K[:, 0, 1] *= np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    V = rng.integers(-127, 128, (n, 1, 128)).astype(np.float32)
    V[:, 0, 5] = 127.0
    return q, K, V


def test_exact_sum_is_the_textbook_softmax_when_scores_are_exact():
    n = 777
    q, K, V = _integer_case(n, 3)
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    assert np.array_equal(k8[:, 0].astype(np.float32), K[:, 0])   # identity quantisation
    qi, qsc = oracle.quantize_q(q)
    assert np.array_equal(qsc, np.ones(4, np.float32)) and np.array_equal(qi.astype(np.float32), q)
    scale = 2.0 ** -6                           # every score is exact in fp32
    s = (K[:, 0].astype(np.float64) @ q.astype(np.float64)) * scale
    want = scipy.special.softmax(s) @ V[:, 0].astype(np.float64)
    got = oracle.attn_exact_sum(q, oracle.SeqCache(k8, ks, v8, vs), 0, np.float32(scale))
    assert np.abs(got - want).max() <= 1e-11 * np.abs(want).max()


@pytest.mark.parametrize("n", [1, 33, 1000])
def test_exact_sum_agrees_with_one_pass_on_short_sequences(n):
    cache, _ = _cache(n, seed=n)
    q = np.random.default_rng(n).standard_normal(128).astype(np.float32)
    for kh in range(2):
        a = oracle.attn_exact_sum(q, cache, kh, np.float32(0.088))
        b = oracle.attn_single_q(q, cache, kh, np.float32(0.088))
        # the fp32 loop's rounding: ~1e-6 of the output at these lengths
        assert np.abs(a - b).max() <= 1e-5 * max(1.0, np.abs(a).max())


def test_one_pass_rounding_grows_on_long_sequences_and_exact_sum_does_not():
    # token 0 scores highest (weight 1); n - 1 equal tokens each weigh ~1.5e-6.
    # The fp32 loop adds each small weight to a running sum near 1, whose unit
    # in the last place is 1.2e-7: every add rounds, the same way, so the sum
    # drifts.  The exact sum matches the closed form.
    n = 200000
    q = np.zeros(128, np.float32)
    q[0::32] = 127.0
    K = np.zeros((n, 1, 128), np.float32)
    K[0, 0, 0::32] = 127.0                      # dot 127 * 508
    K[1:, 0, 0::32] = 100.0                     # dot 127 * 400
    K[1:, 0, 2] = 127.0                         # stored max 127 (q is 0 there)
    V = np.zeros((n, 1, 128), np.float32)
    V[0, 0, 0] = 127.0
    V[1:, 0, 1] = 127.0
    k8, ks = oracle.kv_quantize_rows(K)
    v8, vs = oracle.kv_quantize_rows(V)
    scale = 2.0 ** -10
    cache = oracle.SeqCache(k8, ks, v8, vs)
    w = math.exp((127 * 400 - 127 * 508) * scale)
    den = 1.0 + (n - 1) * w
    want = np.zeros(128)
    want[0], want[1] = 127.0 / den, 127.0 * (n - 1) * w / den
    exact = oracle.attn_exact_sum(q, cache, 0, np.float32(scale))
    assert np.abs(exact - want).max() <= 1e-9 * 127
    one_pass = oracle.attn_single_q(q, cache, 0, np.float32(scale))
    assert np.abs(one_pass - want).max() > 1e-4
