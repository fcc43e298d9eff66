"""Helpers shared by the GPU parity tests: run the same seeded inputs through
the CUDA library and through the CPU oracle, and compare."""
import numpy as np

import oracle
from query_decode_attention_gb300 import workloads as W


def out_tolerance(ref: np.ndarray) -> float:
    """fp32 attention outputs: max abs error <= 1e-4 and <= 1e-3 * max|out|."""
    m = float(np.abs(ref).max()) if ref.size else 0.0
    return min(1e-4, 1e-3 * m)


def assert_out_close(got: np.ndarray, ref: np.ndarray, what: str = "", exact=None) -> float:
    """got within the tolerance of the oracle's fp32 one-pass result `ref`.

    `exact` (optional): the oracle's exact-sum result for the same rows
    (oracle.attn_exact_sum: the method's fp32 scores, fp64 sums).  The fp32
    one-pass loop and the kernels' tile-wise loop are two roundings of the same
    computation (article 9-2 §3); over very long sequences the loop's own
    rounding can exceed the tolerance.  Only where it measurably does (ref more
    than half the tolerance from `exact`) is got held to `exact` instead."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    got64 = got.astype(np.float64)
    err = float(np.abs(got64 - ref.astype(np.float64)).max()) if got.size else 0.0
    tol = out_tolerance(ref)
    if err <= tol or exact is None:
        assert err <= tol, f"{what}: max abs err {err:.3e} > tol {tol:.3e}"
        return err
    own = float(np.abs(ref.astype(np.float64) - exact).max())
    err_exact = float(np.abs(got64 - exact).max())
    tol_exact = out_tolerance(exact)
    assert own > tol / 2 and err_exact <= tol_exact, (
        f"{what}: max abs err {err:.3e} > tol {tol:.3e} against the fp32 one pass; "
        f"{err_exact:.3e} against the exact sums (tol {tol_exact:.3e}); the one pass "
        f"itself is {own:.3e} from them")
    return err_exact


def host_inputs(wl: W.Workload, layer: int = 0):
    q = W.host_q(wl, layer)
    Ks, Vs = [], []
    for b in range(wl.B):
        K, V = W.host_kv(wl, b, layer, q=q)
        Ks.append(K)
        Vs.append(V)
    return q, Ks, Vs


def oracle_quantized(Ks, Vs):
    k8s, kss, v8s, vss = [], [], [], []
    for K, V in zip(Ks, Vs):
        k8, ks = oracle.kv_quantize_rows(K)
        v8, vs = oracle.kv_quantize_rows(V)
        k8s.append(k8)
        kss.append(ks)
        v8s.append(v8)
        vss.append(vs)
    return k8s, kss, v8s, vss


def oracle_decode(wl, q, Ks, Vs, sparse=False):
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    return oracle.decode_batch(q, k8s, kss, v8s, vss, wl.scale, kv_bs=wl.kv_bs, sparse=sparse,
                               block=wl.block, topk=wl.topk, probe=wl.probe)
