"""Failure detection on the GPU without a fault: the prefill kernel's waits
are bounded, so a copy that never lands (the test hook withholds one raw
sub-tile) makes the wait run out, the kernel reports KQ8_STATUS_TIMEOUT,
leaves the affected rows unwritten and returns, and the context stays usable
for the next call."""
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


def _case(n, nq=16, nkv=8, seed=31):
    wl = W.custom(1, nq, nkv, [n], seed=seed)
    _, Ks, Vs = host_inputs(wl)
    c = paged.fill_from_host(wl, Ks, Vs, DEV)
    qp = np.random.default_rng(seed).standard_normal((n, nq, 128)).astype(np.float32)
    q_off = torch.tensor([0, n], dtype=torch.int32, device=DEV)
    return wl, Ks, Vs, c, qp, q_off


@pytest.mark.parametrize("withhold", [0, 3])
def test_withheld_copy_times_out_and_the_context_stays_usable(withhold):
    n = 200  # G = 2: CTAs of 2 x 64 new tokens, 2 per KV head; both walks pass sub-tile 3
    wl, Ks, Vs, c, qp, q_off = _case(n)
    q = torch.tensor(qp, device=DEV)
    out = torch.full((n, wl.nq, 128), float("nan"), device=DEV)
    ws = kq8.new_workspace(kq8.kq8_prefill_workspace_bytes(1, wl.nq, wl.nkv, n, n), DEV)
    kq8.kq8_debug_prefill_withhold(out, q, c.cache, c.page_table, c.seq_lens, q_off, n, n,
                                   wl.scale, ws, withhold)
    torch.cuda.synchronize()
    status = kq8.kq8_read_status(ws)
    assert status & kq8.KQ8_STATUS_TIMEOUT, status
    got = out.cpu().numpy()
    # a CTA whose walk reaches the withheld sub-tile writes none of its rows
    assert np.isnan(got).all()
    # the same context runs the intact call and matches the oracle
    out2 = torch.full_like(out, float("nan"))
    kq8.kq8_prefill_attn(out2, q, c.cache, c.page_table, c.seq_lens, q_off, n, n, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    k8s, kss, v8s, vss = oracle_quantized(Ks, Vs)
    ref = oracle.prefill_batch(qp, [n], k8s, kss, v8s, vss, wl.scale)
    assert_out_close(out2.cpu().numpy(), ref, "after a timed-out call")


def test_withhold_hook_rejects_a_negative_index():
    wl, _, _, c, qp, q_off = _case(40)
    q = torch.tensor(qp, device=DEV)
    out = torch.empty_like(q)
    ws = kq8.new_workspace(4096, DEV)
    with pytest.raises(kq8.Kq8Error):
        kq8.kq8_debug_prefill_withhold(out, q, c.cache, c.page_table, c.seq_lens, q_off, 40, 40,
                                       wl.scale, ws, -1)


# ---------------------------------------------------------------------------
# the decode kernel: each warp's bounded wait is decided by the whole warp; a
# CTA whose wait ran out writes nothing, and the chunk merge leaves a row as it
# was when any of its chunks timed out
# ---------------------------------------------------------------------------

def _rows_left_alone(lens, chunk_tiles, num_chunks, withhold):
    """Sequences with a CTA whose first warp walks more than `withhold` tiles:
    warp w of a chunk of L tiles walks tiles w, w + 4, ... (ceil(L / 4) for w = 0)."""
    hit = []
    for n in lens:
        tiles = -(-n // 32)
        chunks = [min(chunk_tiles, tiles - c * chunk_tiles) for c in range(num_chunks)
                  if c * chunk_tiles < tiles]
        hit.append(any(-(-L // 4) > withhold for L in chunks))
    return np.array(hit)


@pytest.mark.parametrize("withhold", [0, 2])
def test_decode_withheld_copy_times_out_and_the_context_stays_usable(withhold):
    lens = [20000, 3099, 100, 0]
    wl = W.custom(len(lens), 32, 8, lens, seed=41)      # G = 4, the serving head ratio
    q, Ks, Vs = host_inputs(wl)
    c = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                           DEV)
    ct, nch = kq8.kq8_decode_plan(wl.B, wl.nq, wl.nkv, wl.max_seq_len)
    hit = _rows_left_alone(lens, ct, nch, withhold)
    assert hit.any()
    out = torch.full((wl.B, wl.nq, 128), float("nan"), device=DEV)
    kq8.kq8_debug_decode_withhold(out, c.q, c.cache, c.page_table, c.seq_lens, wl.max_seq_len,
                                  wl.scale, ws, withhold)
    torch.cuda.synchronize()
    assert kq8.kq8_read_status(ws) & kq8.KQ8_STATUS_TIMEOUT
    got = out.cpu().numpy()
    ref = oracle_decode(wl, q, Ks, Vs)
    for b in range(wl.B):
        if hit[b]:
            assert np.isnan(got[b]).all(), b          # left as it was
        else:
            assert_out_close(got[b], ref[b], f"untouched by the timeout, b={b}")
    # the same workspace and context run the intact call, every row exact
    out2 = torch.full_like(out, float("nan"))
    kq8.kq8_decode_attn(out2, c.q, c.cache, c.page_table, c.seq_lens, wl.max_seq_len, wl.scale, ws)
    assert kq8.kq8_read_status(ws) == 0
    assert_out_close(out2.cpu().numpy(), ref, "after a timed-out decode")


def test_decode_withhold_hook_rejects_a_negative_index():
    wl = W.custom(1, 16, 8, [40], seed=3)
    q, Ks, Vs = host_inputs(wl)
    c = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(1, 16, 8, 40), DEV)
    out = torch.empty((1, 16, 128), device=DEV)
    with pytest.raises(kq8.Kq8Error):
        kq8.kq8_debug_decode_withhold(out, c.q, c.cache, c.page_table, c.seq_lens, 40, wl.scale,
                                      ws, -1)
