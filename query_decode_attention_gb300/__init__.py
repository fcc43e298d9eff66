"""GB300-native q8-KV single-query decode attention.

The compute lives in ``libkq8.so`` (hand-written sm_103a CUDA kernels behind a
plain C ABI, declared in ``include/kq8.h``); ``query_decode_attention_gb300.kq8``
is the thin ctypes binding with the same entry-point names.  Importing this
package does not load the library; importing the binding does, and fails
loudly when it has not been built.
"""
__all__ = ["workloads"]
