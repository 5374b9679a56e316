"""The allocation-free dense decode entry point, through the C ABI.

kvq_dense_decode_noalloc serves callers that cannot allocate device memory when they
call: their device memory is held by another framework's pool, they own only fixed
buffers, or a step must not fail on allocation.  Its output must match the library's
existing dense path -- kvq_decode_attention with tau_cov = 1, which returns dense
attention for every head -- within the tolerance of the other parity tests, and the
oracle's dense attention element by element, on two calls in a row that share the fixed
scratch array.  This file is collected last so that a run stopping at the first failure
has already run every other test; it passes alone in a fresh process too (its first
test makes the first call on the device, which sets the scratch array up).
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import oracle as O  # noqa: E402
import workloads as W  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2          # the parity tests' output tolerance
CAP_TOKENS = 507904              # B * Hkv = 8: the largest context the 8 MiB scratch takes


def _existing_entry_point(q, K, V):
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


def _check_against_oracle(out, q, K, V):
    """Element by element against oracle.dense_attention (float64): max-abs 2e-3 where
    the exact outputs lie within +-2, 2e-3 + 1e-2 |x| beyond."""
    q, K, V, out = q.cpu().numpy(), K.cpu().numpy(), V.cpu().numpy(), out.cpu().float().numpy()
    B, Hq, _ = q.shape
    n_rep = Hq // K.shape[1]
    worst = 0.0
    for b in range(B):
        for h in range(Hq):
            ref = O.dense_attention(q[b, h], K[b, h // n_rep], V[b, h // n_rep])
            err = np.abs(out[b, h] - ref)
            if np.max(np.abs(ref)) <= 2.0:
                assert err.max() <= ATOL, (b, h, err.max())
            assert np.all(err <= ATOL + RTOL * np.abs(ref)), (b, h, err.max())
            worst = max(worst, float(err.max()))
    return worst


def _call(q, K, V):
    out = torch.full_like(q, float("nan"))
    kvq.dense_decode_noalloc(q, K, V, out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    return out


def test_noalloc_first_call_on_the_device():
    """The first call sets the scratch array up on the device and returns KVQ_OK."""
    q, K, V = W.c1(ctx=64 * 5 + 3, Hq=4, Hkv=1)
    q, K, V = q.cuda(), K.cuda(), V.cuda()
    out = torch.empty_like(q)
    lib = kvq.load_library()
    st = lib.kvq_dense_decode_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), 1, 4, 1,
                                      K.shape[2], out.data_ptr(), None)
    assert st == kvq.KVQ_OK, lib.kvq_last_error()
    torch.cuda.synchronize()
    _check_against_oracle(out, q, K, V)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (8, 8), (6, 2), (12, 4)])
def test_noalloc_dense_matches_existing_entry_point_twice(Hq, Hkv):
    """Two calls in a row (the second reuses the scratch the first left behind), each
    against the existing entry point and against the oracle."""
    cases = [W.c1(ctx=64 * 37 + 19, Hq=Hq, Hkv=Hkv, batch=2),
             W.c1(seed=5, ctx=64 * 90, Hq=Hq, Hkv=Hkv)]
    for q, K, V in cases:
        q, K, V = q.cuda().contiguous(), K.cuda().contiguous(), V.cuda().contiguous()
        ref = _existing_entry_point(q, K, V)
        out = _call(q, K, V)
        assert torch.allclose(out.float(), ref.float(), atol=ATOL, rtol=RTOL), \
            (out.float() - ref.float()).abs().max().item()
        _check_against_oracle(out, q, K, V)


def test_noalloc_on_a_side_stream():
    q, K, V = W.c1(seed=9, ctx=64 * 21 + 7, Hq=8, Hkv=2)
    q, K, V = q.cuda(), K.cuda(), V.cuda()
    out = torch.full_like(q, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        kvq.dense_decode_noalloc(q, K, V, out)
    side.synchronize()
    _check_against_oracle(out, q, K, V)


def test_noalloc_capacity_edge():
    """B * Hkv = 8 groups: 507904 tokens fit the scratch (checked against the oracle on
    one group), 507905 do not and are refused before anything is launched."""
    lib = kvq.load_library()
    q = torch.zeros(1, 32, 128, dtype=torch.float16, device="cuda")
    small = torch.zeros(1, 8, 64, 128, dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    st = lib.kvq_dense_decode_noalloc(q.data_ptr(), small.data_ptr(), small.data_ptr(), 1, 32, 8,
                                      CAP_TOKENS + 1, out.data_ptr(), None)
    assert st == kvq.KVQ_ERR_CAPACITY
    assert b"8 MiB" in lib.kvq_last_error()
    q, K, V = W.c1(device="cuda", seed=11, ctx=CAP_TOKENS, Hq=32, Hkv=8)
    out = _call(q.contiguous(), K.contiguous(), V.contiguous())
    _check_against_oracle(out[:, :4], q[:, :4], K[:, :1], V[:, :1])   # group 0
    del K, V
    torch.cuda.empty_cache()


def test_noalloc_rejects_bad_buffers():
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, 1, 64, 128, dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(ValueError):                      # tensors on two devices
        kvq.dense_decode_noalloc(q.cpu(), k, k, out)
    with pytest.raises(kvq.KvqError) as e:               # host memory, caught by the C ABI
        kvq.dense_decode_noalloc(q.cpu(), k.cpu(), k.cpu(), out.cpu())
    assert e.value.status == kvq.KVQ_ERR_INVALID
    lib = kvq.load_library()
    # 64 groups x 2048 chunks of partials cannot fit in the fixed scratch
    st = lib.kvq_dense_decode_noalloc(q.data_ptr(), k.data_ptr(), k.data_ptr(), 8, 32, 8,
                                      2048 * 1024, out.data_ptr(), None)
    assert st == kvq.KVQ_ERR_CAPACITY
    assert b"8 MiB" in lib.kvq_last_error()
