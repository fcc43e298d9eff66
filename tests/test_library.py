"""Host-side checks of libkq8 that need no GPU: the library loads, exports
every entry point include/kq8.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from query_decode_attention_gb300 import build
    build.build()
    from query_decode_attention_gb300 import kq8
    return kq8


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kq8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kq8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kq8_append_kv", "kq8_decode_attn", "kq8_sparse_decode_attn",
              "kq8_decode_workspace_bytes", "kq8_sparse_decode_workspace_bytes",
              "kq8_workspace_init", "kq8_read_status", "kq8_strerror", "kq8_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib._build.LIB)
    for n in declared_functions():
        assert hasattr(so, n), n


def test_strerror_and_version(lib):
    assert lib.kq8_version() >= 10000
    assert lib.kq8_strerror(0) == "ok"
    assert "workspace" in lib.kq8_strerror(lib.KQ8_ERR_WORKSPACE)
    assert lib.kq8_strerror(-99) == "unknown error"


def test_workspace_sizes_are_sane(lib):
    small = lib.kq8_decode_workspace_bytes(1, 16, 8, 256)
    assert small >= 256 and small % 256 == 0
    big = lib.kq8_decode_workspace_bytes(64, 32, 8, 32768)
    assert big > small
    assert lib.kq8_decode_workspace_bytes(-1, 16, 8, 256) == 0
    sp = lib.kq8_sparse_decode_workspace_bytes(16, 16, 8, 65536, 32, 32)
    # scores of every block per query head fit
    assert sp >= 16 * 16 * (65536 // 32) * 4
    assert lib.kq8_sparse_decode_workspace_bytes(16, 16, 8, 65536, 48, 32) == 0  # block % 32


def _cache_struct(lib, **kw):
    c = dict(k=16, v=16, kscale=16, vscale=16, num_pages=4, kv_bs=32, num_kv_heads=8,
             head_dim=128)
    c.update(kw)
    return lib.kq8_cache_t(c["k"], c["v"], c["kscale"], c["vscale"], c["num_pages"], c["kv_bs"],
                           c["num_kv_heads"], c["head_dim"])


def _decode(lib, cache, B=1, nq=16, max_seq_len=64, max_pages=2, ws=None, ws_bytes=1 << 20,
            out=256, q=256, pt=256, sl=256):
    so = lib._lib
    return so.kq8_decode_attn(out, q, ctypes.byref(cache), pt, max_pages, sl, max_seq_len, B, nq,
                              0.1, ws, ws_bytes, None)


def test_argument_validation_without_device(lib):
    ok = _cache_struct(lib)
    # fake 256-aligned addresses: validation fails before any launch
    assert _decode(lib, _cache_struct(lib, head_dim=64)) == lib.KQ8_ERR_UNSUPPORTED
    assert _decode(lib, _cache_struct(lib, kv_bs=48)) == lib.KQ8_ERR_UNSUPPORTED
    assert _decode(lib, _cache_struct(lib, k=17)) == lib.KQ8_ERR_INVALID_ARG
    assert _decode(lib, _cache_struct(lib, v=0)) == lib.KQ8_ERR_INVALID_ARG
    assert _decode(lib, ok, nq=12) == lib.KQ8_ERR_UNSUPPORTED          # nq % nkv
    assert _decode(lib, ok, nq=8 * 9) == lib.KQ8_ERR_UNSUPPORTED       # G = 9
    assert _decode(lib, ok, max_seq_len=100, max_pages=2) == lib.KQ8_ERR_INVALID_ARG
    assert _decode(lib, ok, B=-1) == lib.KQ8_ERR_INVALID_ARG
    assert _decode(lib, ok, q=260) == lib.KQ8_ERR_INVALID_ARG          # q not 16-B aligned
    assert _decode(lib, ok, ws=None) == lib.KQ8_ERR_WORKSPACE
    assert _decode(lib, ok, ws=512 + 16) == lib.KQ8_ERR_WORKSPACE      # misaligned
    assert _decode(lib, ok, ws=512, ws_bytes=64) == lib.KQ8_ERR_WORKSPACE
    assert _decode(lib, ok, B=0, ws=512) == lib.KQ8_OK                 # nothing to do
    so = lib._lib
    assert so.kq8_append_kv(ctypes.byref(ok), 256, 256, 256, -1, None, None) == lib.KQ8_ERR_INVALID_ARG
    assert so.kq8_append_kv(ctypes.byref(ok), 256, 256, 256, 0, None, None) == lib.KQ8_OK
    assert so.kq8_append_kv(None, 256, 256, 256, 1, None, None) == lib.KQ8_ERR_INVALID_ARG
    sp = so.kq8_sparse_decode_attn
    args = (256, 256, ctypes.byref(ok), 256, 2, 256, 64, 1, 16, ctypes.c_float(0.1))
    assert sp(*args, 32, 32, 33, None, 512, 1 << 20, None) == lib.KQ8_ERR_UNSUPPORTED  # probe > block
    assert sp(*args, 16, 32, 8, None, 512, 1 << 20, None) == lib.KQ8_ERR_UNSUPPORTED   # block < 32
    assert sp(*args, 32, 0, 8, None, 512, 1 << 20, None) == lib.KQ8_ERR_UNSUPPORTED    # topk 0


def _prefill(lib, cache, B=1, nq=16, total_q=8, max_seq_len=64, max_q_len=8, max_pages=2,
             ws=512, ws_bytes=1 << 20, out=256, q=256, pt=256, sl=256, qo=256):
    return lib._lib.kq8_prefill_attn(out, q, total_q, ctypes.byref(cache), pt, max_pages, sl, qo,
                                     max_seq_len, max_q_len, B, nq, 0.1, ws, ws_bytes, None)


def test_prefill_argument_validation_without_device(lib):
    ok = _cache_struct(lib)
    assert lib.kq8_prefill_workspace_bytes(4, 16, 8, 4096, 512) >= 256
    assert _prefill(lib, _cache_struct(lib, head_dim=64)) == lib.KQ8_ERR_UNSUPPORTED
    assert _prefill(lib, _cache_struct(lib, kv_bs=40)) == lib.KQ8_ERR_UNSUPPORTED
    assert _prefill(lib, ok, nq=12) == lib.KQ8_ERR_UNSUPPORTED         # nq % nkv
    assert _prefill(lib, ok, nq=72) == lib.KQ8_ERR_UNSUPPORTED         # G = 9
    assert _prefill(lib, ok, max_seq_len=100) == lib.KQ8_ERR_INVALID_ARG  # > max_pages * kv_bs
    assert _prefill(lib, ok, max_q_len=65) == lib.KQ8_ERR_INVALID_ARG  # more new than cached
    assert _prefill(lib, ok, total_q=-1) == lib.KQ8_ERR_INVALID_ARG
    assert _prefill(lib, ok, out=264) == lib.KQ8_ERR_INVALID_ARG        # 8-B aligned only
    assert _prefill(lib, ok, qo=None) == lib.KQ8_ERR_INVALID_ARG
    assert _prefill(lib, ok, ws=None) == lib.KQ8_ERR_WORKSPACE
    assert _prefill(lib, ok, ws=512 + 64) == lib.KQ8_ERR_WORKSPACE     # not 256-B aligned
    assert _prefill(lib, ok, ws_bytes=16) == lib.KQ8_ERR_WORKSPACE
    assert _prefill(lib, ok, B=0) == lib.KQ8_OK                        # nothing to do
    assert _prefill(lib, ok, max_q_len=0) == lib.KQ8_OK


def test_product_path_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "query_decode_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "kq8o_" not in text, f


def test_sparse_prefill_argument_validation_without_device(lib):
    ok = _cache_struct(lib)
    so = lib._lib
    assert lib.kq8_sparse_prefill_workspace_bytes(100, 16, 8, 4096, 32, 32) > \
        lib.kq8_sparse_decode_workspace_bytes(100, 16, 8, 4096, 32, 32)
    assert lib.kq8_sparse_prefill_workspace_bytes(100, 16, 8, 4096, 48, 32) == 0   # block % 32

    def call(block=32, topk=4, probe=8, total_q=8, B=1, mq=8, ws=512, ws_bytes=1 << 24):
        return so.kq8_sparse_prefill_attn(256, 256, total_q, ctypes.byref(ok), 256, 2, 256, 256,
                                          64, mq, B, 16, ctypes.c_float(0.1), block, topk, probe,
                                          None, ws, ws_bytes, None)
    assert call(block=16) == lib.KQ8_ERR_UNSUPPORTED
    assert call(probe=33) == lib.KQ8_ERR_UNSUPPORTED
    assert call(topk=0) == lib.KQ8_ERR_UNSUPPORTED
    assert call(mq=65) == lib.KQ8_ERR_INVALID_ARG          # more new tokens than cached
    assert call(total_q=70000) == lib.KQ8_ERR_UNSUPPORTED  # rows > 65535
    assert call(ws=None) == lib.KQ8_ERR_WORKSPACE
    assert call(ws_bytes=1024) == lib.KQ8_ERR_WORKSPACE
    assert call(total_q=0) == lib.KQ8_OK


def test_q4_argument_validation_without_device(lib):
    ok = _cache_struct(lib)
    so = lib._lib
    assert so.kq8_append_kv_q4(ctypes.byref(ok), 256, 256, 256, -1, None, None) == lib.KQ8_ERR_INVALID_ARG
    assert so.kq8_append_kv_q4(ctypes.byref(ok), 256, 256, 256, 0, None, None) == lib.KQ8_OK
    assert so.kq8_append_kv_q4(ctypes.byref(ok), 260, 256, 256, 1, None, None) == lib.KQ8_ERR_INVALID_ARG
    dec = so.kq8_decode_attn_q4
    args = (256, 256, ctypes.byref(ok), 256, 2, 256)
    assert dec(*args, 64, 1, 12, ctypes.c_float(0.1), 512, 1 << 20, None) == lib.KQ8_ERR_UNSUPPORTED
    assert dec(*args, 100, 1, 16, ctypes.c_float(0.1), 512, 1 << 20, None) == lib.KQ8_ERR_INVALID_ARG
    assert dec(*args, 64, 1, 16, ctypes.c_float(0.1), None, 1 << 20, None) == lib.KQ8_ERR_WORKSPACE
    assert dec(*args, 64, 0, 16, ctypes.c_float(0.1), 512, 1 << 20, None) == lib.KQ8_OK


def _prototypes():
    """name -> list of parameter type strings, from include/kq8.h."""
    text = open(os.path.join(ROOT, "include", "kq8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(kq8_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = [p.strip() for p in m.group(2).replace("\n", " ").split(",")]
        if params == ["void"] or params == [""]:
            params = []
        out[m.group(1)] = params
    return out


def _ctype_class(c_param):
    """The ctypes class a C parameter must be marshalled as."""
    if "*" in c_param or c_param.startswith("kq8_stream_t"):
        return "pointer"
    for ctype, cls in (("int32_t", "int32"), ("uint32_t", "uint32"), ("size_t", "size"),
                       ("float", "float"), ("int ", "int32")):
        if c_param.startswith(ctype) or c_param.startswith("const " + ctype):
            return cls
    raise AssertionError(f"unrecognised parameter type: {c_param}")


def _ctypes_class(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "_type_") and isinstance(
            getattr(t, "_type_"), type):
        return "pointer"
    return {ctypes.c_int32: "int32", ctypes.c_uint32: "uint32", ctypes.c_size_t: "size",
            ctypes.c_float: "float"}[t]


def test_binding_argtypes_match_the_header(lib):
    # ctypes marshals by the declared argtypes without checking them against
    # the C prototype: a drift between binding and header passes silently
    protos = _prototypes()
    checked = 0
    for name, params in protos.items():
        fn = getattr(lib._lib, name)
        if fn.argtypes is None:
            continue
        got = [_ctypes_class(t) for t in fn.argtypes]
        want = [_ctype_class(p) for p in params]
        assert got == want, f"{name}: binding {got} vs header {want}"
        checked += 1
    assert checked >= 20, checked
