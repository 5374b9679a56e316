"""The allocation-free dense decode entry point against the existing entry point.

kvq_dense_decode_noalloc serves callers that cannot allocate device memory when they
call (their device memory is held by another pool, or they own only fixed buffers).
Its output must match the library's own dense path -- kvq_decode_attention with
tau_cov = 1, which returns dense attention for every head -- within the tolerance of
the other parity tests, on two calls in a row that share the fixed scratch array.
This file is collected last so that a run stopping at the first failure has already
run every other test.
"""

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _reference(q, K, V):
    """Dense output of the existing entry point (rung 4 via tau_cov = 1)."""
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N)
    try:
        cache.append(0, K, V)
        out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cache.decode(0, q, 1.0, 0.25, out)
        torch.cuda.synchronize()
    finally:
        cache.close()
    return out


def test_noalloc_dense_matches_existing_entry_point_twice():
    cases = [W.c1(ctx=64 * 37 + 19, Hq=8, Hkv=2, batch=2), W.c1(seed=5, ctx=64 * 90, Hq=32, Hkv=8)]
    for q, K, V in cases:          # two calls in a row, the second reusing the scratch
        q, K, V = q.cuda().contiguous(), K.cuda().contiguous(), V.cuda().contiguous()
        ref = _reference(q, K, V)
        out = torch.full_like(ref, float("nan"))
        kvq.dense_decode_noalloc(q, K, V, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.allclose(out.float(), ref.float(), atol=ATOL, rtol=RTOL), \
            (out.float() - ref.float()).abs().max().item()


def test_noalloc_rejects_oversize_and_host_buffers():
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, 1, 64, 128, dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(kvq.KvqError) as e:
        kvq.dense_decode_noalloc(q.cpu(), k, k, out)
    assert e.value.status == kvq.KVQ_ERR_INVALID
    lib = kvq.load_library()
    # 64 groups x 2048 chunks of partials cannot fit in the fixed scratch
    st = lib.kvq_dense_decode_noalloc(q.data_ptr(), k.data_ptr(), k.data_ptr(), 8, 32, 8,
                                      2048 * 1024, out.data_ptr(), None)
    assert st == kvq.KVQ_ERR_CAPACITY
    assert b"8 MiB" in lib.kvq_last_error()
