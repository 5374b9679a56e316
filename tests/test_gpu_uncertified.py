"""The uncertified INT8/INT4 baseline (kvq_decode_attention_uncertified) against the
oracle, element by element: output within the output tolerance, the reported bounds
within the bound tolerance, the certificate's fixed fields exact.
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
from _parity import BOUND_ATOL, BOUND_RTOL, OUT_ATOL, OUT_RTOL  # noqa: E402


def _run(q, K, V, debug=0, host_io=False, then_certified=None):
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=max(N, 1))
    try:
        cache.set_debug(debug)
        cache.append(0, K.cuda().contiguous(), V.cuda().contiguous())
        if host_io:
            out = torch.empty(B, Hq, D, dtype=torch.float16).pin_memory()
            cert = torch.empty(B * Hq * 32, dtype=torch.uint8).pin_memory()
            cache.decode_uncertified(0, q.contiguous(), out, cert)
        else:
            out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
            cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
            cache.decode_uncertified(0, q.cuda().contiguous(), out, cert)
        torch.cuda.synchronize()
        res = (out.cpu(), kvq.certificates(cert).reshape(B, Hq))
        if then_certified is not None:
            tau, eps = then_certified
            out2 = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
            cert2 = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
            cache.decode(0, q.cuda().contiguous(), tau, eps, out2, cert2)
            torch.cuda.synchronize()
            res = res + (out2.cpu(), kvq.certificates(cert2).reshape(B, Hq))
        return res
    finally:
        cache.close()


def _compare(out, cert, q, K, V):
    qn, Kn, Vn = q.numpy(), K.numpy(), V.numpy()
    r = O.uncertified_decode_layer(qn, Kn, Vn, O.quantize_layer(Kn, Vn))
    err = np.abs(out.float().numpy() - r.out64)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(r.out64)), f"output off by {err.max():.3e}"
    for name in ("e_key", "e_val"):
        g, o = cert[name].astype(np.float64), getattr(r, name)
        assert np.all(np.abs(g - o) <= BOUND_RTOL * np.abs(o) + BOUND_ATOL), name
    assert np.all(cert["level"] == 0) and np.all(cert["rank_ok"] == 1)
    assert np.all(cert["k_star"] == 0) and np.all(cert["promoted_bytes"] == 0)
    assert np.all(cert["n_val_promoted"] == 0)
    return r


@pytest.mark.parametrize("ctx", [37, 64, 64 * 16 + 1, 64 * 33 + 63, 64 * 300 + 5])
def test_uncertified_ragged(ctx):
    q, K, V = W.tiny(seed=40 + ctx % 7, ctx=ctx, Hq=8, Hkv=2, kscale=3.0)
    out, cert = _run(q, K, V)
    _compare(out, cert, q, K, V)


def test_uncertified_c1_shape():
    q, K, V = W.c1()
    out, cert = _run(q, K, V)
    _compare(out, cert, q, K, V)


@pytest.mark.parametrize("n_rep", [1, 3])
def test_uncertified_gqa_widths(n_rep):
    q, K, V = W.tiny(seed=7, ctx=64 * 20 + 9, Hq=2 * n_rep, Hkv=2, kscale=2.0)
    out, cert = _run(q, K, V)
    _compare(out, cert, q, K, V)


def test_uncertified_ignores_forced_rungs_and_host_buffers_agree():
    q, K, V = W.tiny(seed=8, ctx=64 * 12 + 3, Hq=8, Hkv=2, kscale=3.0)
    out0, cert0 = _run(q, K, V)
    out1, cert1 = _run(q, K, V, debug=kvq.DEBUG_FORCE_DENSE | kvq.DEBUG_FORCE_RANK_FAIL)
    out2, cert2 = _run(q, K, V, host_io=True)
    assert torch.equal(out0, out1) and np.array_equal(cert0, cert1)
    assert torch.equal(out0, out2) and np.array_equal(cert0, cert2)


def test_certified_call_after_uncertified_is_unaffected():
    """The uncertified call leaves no flag or queue state that changes the next
    certified call."""
    q, K, V = W.c1(ctx=64 * 40 + 11, Hq=8, Hkv=2)
    _, _, out_c, cert_c = _run(q, K, V, then_certified=(0.995, 0.25))
    cache = kvq.Cache(1, 1, 8, 2, max_ctx=K.shape[2])
    try:
        cache.append(0, K.cuda(), V.cuda())
        out = torch.empty(1, 8, 128, dtype=torch.float16, device="cuda")
        cert = torch.empty(8 * 32, dtype=torch.uint8, device="cuda")
        cache.decode(0, q.cuda(), 0.995, 0.25, out, cert)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), out_c)
        assert np.array_equal(kvq.certificates(cert).reshape(1, 8), cert_c)
    finally:
        cache.close()
