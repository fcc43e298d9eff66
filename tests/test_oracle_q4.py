"""Pins for the oracle's q4 KV variant.  Article 10-1 §2 names the --kv-q4
switch (and keeps it out of the sparse path) but no page gives the format; the
oracle reads it as the q8 write rule of article 9-3 §2 with 7 in place of 127:
stored max m, step m * (1/7), codes roundf(x / step) clamped to [-7, 7],
readers multiply the stored max by 1/7, Q quantised to int8 as in article 9-2
§2.  Each pin checks the oracle against exact arithmetic, a textbook routine or
the q8 path, not against itself."""
import math
from fractions import Fraction

import numpy as np
import scipy.special

import oracle

F32_INV7 = np.float32(1.0) / np.float32(7.0)
SCALE = np.float32(1 / math.sqrt(128))


def _round_half_away(fr: Fraction) -> int:
    s = 1 if fr >= 0 else -1
    a = abs(fr)
    f = a.numerator // a.denominator
    return s * (f + (1 if a - f >= Fraction(1, 2) else 0))


def test_q4_hand_example():
    # row [2, 1, -1, -0.5, 0, ...]: m = 2, step d = 2 * fl(1/7).  fl(1/7) lies
    # just above 1/7, so 1/d is just below 3.5 -> 3, and 0.5/d = 1.75 -> 2; the
    # max maps to 7.
    x = np.zeros(128, np.float32)
    x[:4] = [2.0, 1.0, -1.0, -0.5]
    assert Fraction(float(F32_INV7)) > Fraction(1, 7)
    c, m = oracle.kv_quantize_rows_q4(x[None])
    assert m[0] == 2.0 and list(c[0, :4]) == [7, 3, -3, -2] and not c[0, 4:].any()


def test_q4_matches_exact_rational_rounding():
    rng = np.random.default_rng(41)
    rows = rng.standard_normal((48, 128)).astype(np.float32)
    rows *= rng.choice([1e-20, 1e-3, 1.0, 37.0, 1e20], size=(48, 1)).astype(np.float32)
    codes, maxima = oracle.kv_quantize_rows_q4(rows)
    off = 0
    for r in range(rows.shape[0]):
        assert maxima[r] == np.abs(rows[r]).max()
        d = Fraction(float(np.float32(maxima[r]) * F32_INV7))
        for i in range(128):
            ratio = Fraction(float(rows[r, i])) / d
            exp = max(-7, min(7, _round_half_away(ratio)))
            if codes[r, i] != exp:
                # only where the fp32 quotient rounds across a half-integer
                frac = abs(ratio) - math.floor(abs(ratio))
                assert abs(frac - Fraction(1, 2)) < abs(ratio) * Fraction(1, 2**22), (r, i)
                off += 1
    assert off <= 2


def test_q4_error_bound_range_and_zero_row():
    rng = np.random.default_rng(42)
    rows = (rng.standard_t(3, (200, 128)) * rng.uniform(0.01, 100, (200, 1))).astype(np.float32)
    codes, maxima = oracle.kv_quantize_rows_q4(rows)
    d = (maxima * F32_INV7).astype(np.float64)
    err = np.abs(rows.astype(np.float64) - codes.astype(np.float64) * d[:, None])
    assert np.all(err <= d[:, None] * 0.5 * (1 + 2**-20))
    am = np.abs(rows).argmax(1)
    assert np.all(np.abs(codes[np.arange(200), am]) == 7)
    assert codes.min() >= -7 and codes.max() <= 7
    c, m = oracle.kv_quantize_rows_q4(np.zeros((1, 128), np.float32))
    assert m[0] == 0 and not c.any()


def _q4_cache(n, nkv, seed):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((n, nkv, 128)).astype(np.float32)
    V = rng.standard_normal((n, nkv, 128)).astype(np.float32)
    k4, ks = oracle.kv_quantize_rows_q4(K)
    v4, vs = oracle.kv_quantize_rows_q4(V)
    return K, V, (k4, ks, v4, vs)


def test_q4_one_pass_equals_textbook_softmax():
    for n in (1, 33, 500):
        K, V, (k4, ks, v4, vs) = _q4_cache(n, 2, seed=n)
        cache = oracle.SeqCache(k4, ks, v4, vs)
        q = np.random.default_rng(n + 1).standard_normal(128).astype(np.float32)
        qi, qsc = oracle.quantize_q(q)
        qd = (qi.astype(np.float64).reshape(4, 32) * qsc.astype(np.float64)[:, None]).reshape(128)
        for kh in (0, 1):
            Kd = k4[:, kh].astype(np.float64) * (ks[:, kh] * F32_INV7).astype(np.float64)[:, None]
            Vd = v4[:, kh].astype(np.float64) * (vs[:, kh] * F32_INV7).astype(np.float64)[:, None]
            ref = scipy.special.softmax(Kd @ qd * float(SCALE)) @ Vd
            got = oracle.attn_single_q_q4(q, cache, kh, SCALE)
            assert np.abs(got - ref).max() <= 2e-6 * max(1.0, np.abs(ref).max()), (n, kh)


def test_q4_batch_driver_matches_single_head_calls():
    lens = [70, 5]
    caches = [_q4_cache(n, 2, seed=10 + n)[2] for n in lens]
    q = np.random.default_rng(3).standard_normal((2, 4, 128)).astype(np.float32)
    out = oracle.decode_batch_q4(q, [c[0] for c in caches], [c[1] for c in caches],
                                 [c[2] for c in caches], [c[3] for c in caches], SCALE)
    for b, c in enumerate(caches):
        sc = oracle.SeqCache(*c)
        for h in range(4):
            assert np.array_equal(out[b, h], oracle.attn_single_q_q4(q[b, h], sc, h // 2, SCALE))


def test_q4_is_coarser_than_q8_on_the_same_data():
    # the 256-token experiment of article 9-3 §3 with q4 codes: the output
    # error against fp32 KV grows by roughly the ratio of the steps (127 / 7)
    rng = np.random.default_rng(9)
    n = 256
    K = rng.standard_normal((n, 1, 128)).astype(np.float32)
    V = rng.standard_normal((n, 1, 128)).astype(np.float32)
    q = rng.standard_normal((16, 128)).astype(np.float32)
    k8, ks8 = oracle.kv_quantize_rows(K)
    v8, vs8 = oracle.kv_quantize_rows(V)
    k4, ks4 = oracle.kv_quantize_rows_q4(K)
    v4, vs4 = oracle.kv_quantize_rows_q4(V)
    c8, c4 = oracle.SeqCache(k8, ks8, v8, vs8), oracle.SeqCache(k4, ks4, v4, vs4)
    e8, e4 = [], []
    for h in range(16):
        ref = oracle.attn_ref_f64(q[h], K[:, 0], V[:, 0], float(SCALE))
        e8.append(np.abs(oracle.attn_single_q(q[h], c8, 0, SCALE) - ref).max())
        e4.append(np.abs(oracle.attn_single_q_q4(q[h], c4, 0, SCALE) - ref).max())
    r = np.mean(e4) / np.mean(e8)
    assert 4 < r < 60, r
