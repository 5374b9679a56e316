"""FP16-values configuration (value_bits = 16: FP16 values resident in VRAM, keys-only
tier 2) against the oracle with value_fp16, element by element.  Tolerances are those
of tests/_parity.py.
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
from _parity import (OUT_ATOL, OUT_RTOL, compare_decode, compare_tier1, gpu_run,  # noqa: E402
                     oracle_run)


def _check(q, K, V, tau, eps, **kw):
    g = gpu_run(q, K, V, tau, eps, value_bits=16, **kw)
    t1, r = oracle_run(q, K, V, tau, eps, value_bits=16)
    compare_tier1(g["t1"], t1, value_bits=16)
    st = compare_decode(g, t1, r, tau, eps, q.shape[1] // K.shape[1])
    c = g["cert"]
    assert np.all(c["e_val"] == 0.0) and np.all(c["n_val_promoted"] == 0)
    return g, r, st


@pytest.mark.parametrize("ctx", [37, 64, 64 * 16 + 1, 64 * 33 + 63, 64 * 700 + 5])
def test_fp16_values_ragged(ctx):
    q, K, V = W.tiny(seed=50 + ctx % 5, ctx=ctx, Hq=8, Hkv=2, kscale=3.0)
    _check(q, K, V, 0.95, 0.25, chunks=None)


def test_fp16_values_chunked_appends():
    q, K, V = W.tiny(seed=51, ctx=64 * 12 + 37, Hq=4, Hkv=1, kscale=2.0)
    _check(q, K, V, 0.9, 0.25, chunks=[1, 63, 64, 100, 1, 540, 36])


def test_fp16_values_c1_shape_and_rungs():
    q, K, V = W.c1()
    _check(q, K, V, 0.995, 0.25)
    # a tight budget drives heads up the ladder (rung 2 has no values to page in)
    g, r, _ = _check(q, K, V, 0.9, 0.02)
    assert np.any(r.level > 0)


def test_fp16_values_dense_rungs():
    q, K, V = W.tiny(seed=52, ctx=64 * 20 + 3, Hq=8, Hkv=2, kscale=3.0)
    nb = K.shape[2] // 64
    g, r, _ = _check(q, K, V, 1.0, 0.25)                 # tau = 1: rung 4 everywhere
    assert np.all(g["cert"]["level"] == 4)
    # a dense group pages in its keys only (values are read from VRAM)
    assert np.all(g["cert"]["promoted_bytes"] == nb * 64 * 128 * 2)
    g = gpu_run(q, K, V, 0.9, 0.25, debug=kvq.DEBUG_FORCE_RANK_FAIL, value_bits=16)
    assert np.all(g["cert"]["rank_ok"] == 0) and np.all(g["cert"]["level"] == 4)
    for h in range(8):
        dense = O.dense_attention(q[0, h].numpy(), K[0, h // 4].numpy(), V[0, h // 4].numpy())
        assert np.allclose(g["out"][0, h].float().numpy(), dense, atol=OUT_ATOL, rtol=OUT_RTOL)


def test_fp16_values_uncertified():
    q, K, V = W.tiny(seed=53, ctx=64 * 30 + 17, Hq=8, Hkv=2, kscale=3.0)
    cache = kvq.Cache(1, 1, 8, 2, max_ctx=K.shape[2], value_bits=16)
    try:
        cache.append(0, K.cuda(), V.cuda())
        out = torch.empty(1, 8, 128, dtype=torch.float16, device="cuda")
        cert = torch.empty(8 * 32, dtype=torch.uint8, device="cuda")
        cache.decode_uncertified(0, q.cuda(), out, cert)
        torch.cuda.synchronize()
        c = kvq.certificates(cert).reshape(1, 8)
    finally:
        cache.close()
    qn, Kn, Vn = q.numpy(), K.numpy(), V.numpy()
    u = O.uncertified_decode_layer(qn, Kn, Vn, O.quantize_layer(Kn, Vn),
                                   O.OracleConfig(n_rep=4, value_fp16=True))
    err = np.abs(out.cpu().float().numpy() - u.out64)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(u.out64))
    assert np.all(c["e_val"] == 0.0)
    np.testing.assert_allclose(c["e_key"], u.e_key, rtol=1e-4, atol=1e-6)
