"""The C-ABI library loads and exports every function include/kvq.h declares (CPU only:
no compute call is made)."""

import ctypes
import os

import certified_quantized_kv_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    if not os.path.exists(kvq.LIB_PATH):
        from certified_quantized_kv_gb300 import build
        build.build()
    return kvq.load_library()


def test_header_symbols_exported():
    names = kvq.header_functions(os.path.join(ROOT, "include", "kvq.h"))
    assert len(names) >= 10, names
    lib = ctypes.CDLL(kvq.LIB_PATH) if _lib() else None
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_null_and_invalid_arguments_without_gpu():
    lib = _lib()
    # argument checks run before any CUDA call
    assert lib.kvq_cache_create(None, None) == kvq.KVQ_ERR_INVALID
    assert b"NULL" in lib.kvq_last_error()
    cfg = kvq.kvq_config(1, 1, 32, 8, 64, 64, 32, 1024, 1, 0.5)       # head_dim 64
    h = ctypes.c_void_p()
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h)) == kvq.KVQ_ERR_INVALID
    assert b"head_dim" in lib.kvq_last_error()
    cfg = kvq.kvq_config(1, 1, 48, 8, 128, 64, 32, 1024, 1, 0.5)      # n_rep = 6
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h)) == kvq.KVQ_ERR_INVALID
    cfg = kvq.kvq_config(1, 1, 32, 8, 128, 64, 32, 1024, 1, 0.5, 8)   # value_bits 8
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h)) == kvq.KVQ_ERR_INVALID
    assert b"value_bits" in lib.kvq_last_error()
    cfg = kvq.kvq_config(1, 1, 32, 8, 128, 64, 32, 1024, 1, 0.5, 4, -1.0)   # v_tol < 0
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h)) == kvq.KVQ_ERR_INVALID
    assert b"v_tol" in lib.kvq_last_error()
    assert lib.kvq_cache_destroy(None) == kvq.KVQ_OK
    assert lib.kvq_append(None, 0, None, None, 1, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_decode_attention(None, 0, None, 0.9, 0.25, None, None, None, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_decode_attention_uncertified(None, 0, None, None, None, None) == kvq.KVQ_ERR_INVALID
    assert b"kvq_decode_attention_uncertified" in lib.kvq_last_error()
    assert lib.kvq_debug_fill_tier2(None, 0, 0) == kvq.KVQ_ERR_INVALID


def test_certificate_layout_matches_header():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    body = text[text.index("typedef struct kvq_certificate"):]
    body = body[: body.index("} kvq_certificate;")]
    fields = [ln.split(";")[0].split()[-1] for ln in body.splitlines()[1:] if ";" in ln]
    assert fields == list(kvq.CERT_DTYPE.names)


def test_resident_blocks_validated_without_gpu():
    lib = _lib()
    cfg = kvq.kvq_config(1, 1, 32, 8, 128, 64, 32, 1024, 1, 0.5, 4, 0.0, -1)   # resident_blocks < 0
    h = ctypes.c_void_p()
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h)) == kvq.KVQ_ERR_INVALID
    assert b"resident_blocks" in lib.kvq_last_error()
    assert lib.kvq_residency_stats(None, 0, None, None, None, 0) == kvq.KVQ_ERR_INVALID


def test_create_without_device_reports_cuda_error():
    """A valid configuration on a machine without a usable GPU fails with KVQ_ERR_CUDA and
    says why (rather than reporting an out-of-memory)."""
    lib = _lib()
    cfg = kvq.kvq_config(1, 1, 4, 1, 128, 64, 32, 1024, 1, 0.5)
    h = ctypes.c_void_p()
    st = lib.kvq_cache_create(ctypes.byref(cfg), ctypes.byref(h))
    if st == kvq.KVQ_OK:   # a GPU is present: nothing to check here
        lib.kvq_cache_destroy(h)
        import pytest
        pytest.skip("a CUDA device is present")
    assert st == kvq.KVQ_ERR_CUDA, (st, lib.kvq_last_error())
    assert b"no usable CUDA device" in lib.kvq_last_error()
