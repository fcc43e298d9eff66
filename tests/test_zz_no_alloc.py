"""The allocation-free decode entry point (kq8_decode_attn_noalloc).

It exists for callers that may not allocate device memory -- code running
inside another runtime's allocator or launch path, or serving loops that forbid
device allocation after start-up -- and replaces the caller's workspace with a
fixed scratch array inside the library.  These checks call it through the C ABI
on two calls in a row with different shapes.  Both entry points run the same
kernel with the same split and the same merge order, so each result must equal
kq8_decode_attn's (which takes a caller-allocated workspace) bit for bit -- a
partial left in the shared array by the first call would show in the second --
and match the CPU oracle within the usual tolerance.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from kq8_testlib import assert_out_close, host_inputs, oracle_decode
from query_decode_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from query_decode_attention_gb300 import build  # noqa: E402

build.build()
from query_decode_attention_gb300 import kq8, paged  # noqa: E402

DEV = "cuda:0"


def _both(wl):
    """(no-alloc result, workspace result, oracle result) on the same inputs."""
    q, Ks, Vs = host_inputs(wl)
    case = paged.fill_from_host(wl, Ks, Vs, DEV, q_host=q)
    shape = (wl.B, wl.nq, wl.hd)
    ref = torch.empty(shape, dtype=torch.float32, device=DEV)
    ws = kq8.new_workspace(kq8.kq8_decode_workspace_bytes(wl.B, wl.nq, wl.nkv, wl.max_seq_len),
                           DEV)
    kq8.kq8_decode_attn(ref, case.q, case.cache, case.page_table, case.seq_lens, wl.max_seq_len,
                        wl.scale, ws)
    got = torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)
    kq8.kq8_decode_attn_noalloc(got, case.q, case.cache, case.page_table, case.seq_lens,
                                wl.max_seq_len, wl.scale)
    torch.cuda.synchronize()
    assert kq8.kq8_read_status(ws) == 0
    return got.cpu().numpy(), ref.cpu().numpy(), oracle_decode(wl, q, Ks, Vs)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # first call: several chunks per sequence (the merge path uses the scratch)
    wl1 = W.custom(3, 32, 8, [5000, 17, 2100], seed=21)
    got1, ref1, orc1 = _both(wl1)
    assert np.array_equal(got1, ref1), "noalloc, first call: not bit-identical"
    assert_out_close(got1, orc1, "noalloc vs oracle, first call")
    # second call, other shapes: a stale partial from call one would show here
    wl2 = W.custom(2, 16, 4, [300, 4096], seed=22)
    got2, ref2, orc2 = _both(wl2)
    assert np.array_equal(got2, ref2), "noalloc, second call: not bit-identical"
    assert_out_close(got2, orc2, "noalloc vs oracle, second call")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    B, nq, nkv, n = 1024, 64, 8, 32768
    need = kq8.kq8_decode_workspace_bytes(B, nq, nkv, n)
    assert need > (32 << 20)
    cache = kq8.PagedKVCache(1, nkv, 32, DEV)
    q = torch.zeros((B, nq, 128), device=DEV)
    out = torch.zeros_like(q)
    pt = torch.zeros((B, n // 32), dtype=torch.int32, device=DEV)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    with pytest.raises(kq8.Kq8Error) as e:
        kq8.kq8_decode_attn_noalloc(out, q, cache, pt, sl, n, 0.1)
    assert e.value.code == kq8.KQ8_ERR_WORKSPACE
