"""Debug modes of the library: device-side bounds checks and an injected failure of the
append's tier-2 mirror copy (both without faulting the GPU).

KVQ_DEBUG_BOUNDS makes every kernel check the indices it addresses tier 1, tier 2 and
the scratch with; a violation is recorded in a device word (the access is skipped) and
the call returns KVQ_ERR_INVALID naming the kernel.  On valid inputs the word stays
clear: every call returns KVQ_OK and the results are bit-identical to the unchecked run.

KVQ_DEBUG_FAIL_MIRROR makes kvq_append report the mirror copy as failed (the copy is not
issued): the call returns KVQ_ERR_CUDA with the copy named in the error text, the cache
keeps its length, and both that cache (once the tokens are appended again) and a fresh
one decode as the oracle does.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import workloads as W  # noqa: E402
from _parity import compare_decode, compare_tier1, gpu_run, oracle_run  # noqa: E402


def _decode_all(debug, q, K, V, tau=0.95, eps=0.25, chunks=None, value_bits=4, resident=0):
    """Appends in chunks, then a certified, an uncertified and a forced rung-4 decode."""
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N, value_bits=value_bits, resident_blocks=resident)
    res = []
    try:
        cache.set_debug(debug)
        pos = 0
        for n in (chunks or [N]):
            cache.append(0, K[:, :, pos:pos + n].contiguous(), V[:, :, pos:pos + n].contiguous())
            pos += n
        qd = q.contiguous()
        for call in range(4):
            out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
            cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
            if call < 2:   # twice: with residency the second call serves blocks from HBM
                cache.decode(0, qd, tau, eps, out, cert)
            elif call == 2:
                cache.decode_uncertified(0, qd, out, cert)
            else:
                cache.set_debug(debug | kvq.DEBUG_FORCE_DENSE)
                cache.decode(0, qd, tau, eps, out, cert)
                cache.set_debug(debug)
            torch.cuda.synchronize()
            res.append((out.cpu(), cert.cpu()))
    finally:
        cache.close()
    return res


@pytest.mark.parametrize("ctx,chunks,value_bits,resident", [
    (64 * 40 + 13, [100, 1, 64 * 40 + 13 - 101], 4, 0),
    (64 * 300, None, 4, 0),
    (64 * 21 + 5, [64 * 10, 64 * 11 + 5], 16, 0),
    (64 * 33, None, 4, 1 << 12),
])
def test_bounds_checks_stay_clear_on_valid_inputs(ctx, chunks, value_bits, resident):
    q, K, V = W.c3_layer(0, device="cuda", ctx=ctx, Hq=8, Hkv=2, batch=2)
    plain = _decode_all(0, q, K, V, chunks=chunks, value_bits=value_bits, resident=resident)
    checked = _decode_all(kvq.DEBUG_BOUNDS, q, K, V, chunks=chunks, value_bits=value_bits,
                          resident=resident)
    for (o0, c0), (o1, c1) in zip(plain, checked):
        assert torch.equal(o0, o1) and torch.equal(c0, c1)


def test_injected_mirror_failure():
    q, K, V = W.c1(ctx=64 * 12 + 9, Hq=8, Hkv=2)
    Kd, Vd = K.cuda(), V.cuda()
    cache = kvq.Cache(1, 1, 8, 2, max_ctx=2048)
    try:
        cache.append(0, Kd[:, :, :64 * 5].contiguous(), Vd[:, :, :64 * 5].contiguous())
        for lo, hi in ((64 * 5, 64 * 5 + 10), (64 * 5, 64 * 12 + 9)):   # partial-block and full-block paths
            cache.set_debug(kvq.DEBUG_FAIL_MIRROR)
            with pytest.raises(kvq.KvqError) as e:
                cache.append(0, Kd[:, :, lo:hi].contiguous(), Vd[:, :, lo:hi].contiguous())
            assert e.value.status == kvq.KVQ_ERR_CUDA
            assert "mirror" in str(e.value) and "injected" in str(e.value)
            assert cache.length(0) == 64 * 5
        # the process and the cache stay usable: append the rest again and decode
        cache.set_debug(0)
        cache.append(0, Kd[:, :, 64 * 5:].contiguous(), Vd[:, :, 64 * 5:].contiguous())
        assert cache.length(0) == K.shape[2]
        out = torch.empty(1, 8, 128, dtype=torch.float16, device="cuda")
        cert = torch.empty(8 * 32, dtype=torch.uint8, device="cuda")
        cache.decode(0, q.cuda(), 0.995, 0.25, out, cert)
        torch.cuda.synchronize()
        got = out.cpu()
    finally:
        cache.close()
    t1, r = oracle_run(q, K, V, 0.995, 0.25)
    assert np.max(np.abs(got.float().numpy() - r.out64)) <= 2e-3
    # a fresh cache matches the oracle throughout
    g = gpu_run(q, K, V, 0.995, 0.25)
    compare_tier1(g["t1"], t1)
    compare_decode(g, t1, r, 0.995, 0.25, 4)
