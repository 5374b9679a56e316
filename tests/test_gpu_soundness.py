"""Soundness of the GPU certificate itself: on thousands of random and adversarial heads
the CUDA path's output is within its own E_key + E_val of float64 dense attention over
the FP16 originals ("Runtime-Certified Bounded-Error Quantized Attention", Method §2),
and heads at rungs 3-4 return dense attention (Contributions, deterministic recovery).

Allowance beyond the bound: the fp16 rounding of the returned output (2^-11 of its
largest magnitude) plus 1e-5 for fp32 arithmetic.
"""

import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import workloads as W  # noqa: E402


def _dense64(q, K, V, n_rep):
    """float64 softmax(q K^T / sqrt(D)) V per (sequence, query head)."""
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            k = K[b, h // n_rep].astype(np.float64)
            s = k @ q[b, h].astype(np.float64) / math.sqrt(D)
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ V[b, h // n_rep].astype(np.float64)
    return out


def _adversarial_keys(rng, q0, n_tok, s0=2.0 ** -5):
    """Keys just below a half INT8 step, signed against q, so INT8 rounding moves every
    score by close to its bound Delta; one anchor row per block pins the scales to s0."""
    D = q0.shape[-1]
    sg = np.sign(q0.astype(np.float64))
    sg[sg == 0] = 1
    K = np.clip(rng.standard_normal((n_tok, D)), -3.9, 3.9)
    n = rng.integers(0, 120, size=(n_tok, 1))
    adv = sg * (n + 7.0 / 16.0) * s0
    K = np.where(rng.random((n_tok, 1)) < 0.7, adv, K)
    K[::64] = -sg * 127 * s0
    return K.astype(np.float16)


def _run(q, K, V, tau, eps):
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N)
    try:
        cache.append(0, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
        out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
        cache.decode(0, torch.from_numpy(q).cuda(), tau, eps, out, cert)
        torch.cuda.synchronize()
        return out.cpu().float().numpy(), kvq.certificates(cert).reshape(B, Hq)
    finally:
        cache.close()


def _check(q, K, V, tau, eps, n_rep):
    out, c = _run(q, K, V, tau, eps)
    ref = _dense64(q, K, V, n_rep)
    n_cert = 0
    worst = 0.0
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            err = float(np.max(np.abs(out[b, h] - ref[b, h])))
            allow = 2.0 ** -11 * float(np.max(np.abs(ref[b, h]))) + 1e-5
            if c["level"][b, h] >= 3:
                assert c["e_key"][b, h] == 0 and c["e_val"][b, h] == 0
                assert err <= allow + 1e-3, f"dense rung off by {err}"
            else:
                bound = float(c["e_key"][b, h]) + float(c["e_val"][b, h])
                assert err <= bound + allow, f"(b={b}, h={h}) error {err} > bound {bound}"
                n_cert += 1
                if bound > 0:
                    worst = max(worst, err / bound)
    return n_cert, worst


def test_soundness_random_heads():
    rng = np.random.default_rng(60)
    n_cert = 0
    for trial in range(24):
        ctx = int(rng.integers(64, 2200))
        ks = float(rng.choice([0.5, 1.0, 3.0, 8.0]))
        q, K, V = W.tiny(seed=600 + trial, ctx=ctx, Hq=8, Hkv=2, batch=8, kscale=ks)
        q = (q.float() * float(rng.uniform(0.3, 3.0))).half()
        tau = float(rng.choice([0.5, 0.9, 0.99]))
        n, _ = _check(q.numpy(), K.numpy(), V.numpy(), tau, math.inf, 4)
        n_cert += n
    assert n_cert >= 1200   # heads whose ranking check failed went to a dense rung


def test_soundness_adversarial_heads():
    rng = np.random.default_rng(61)
    n_cert, worst = 0, 0.0
    for trial in range(16):
        nb = int(rng.integers(1, 12))
        n_tok = nb * 64 + int(rng.integers(0, 64))
        B, Hkv, n_rep = 4, 2, 4
        q = rng.standard_normal((B, Hkv * n_rep, 128)).astype(np.float16)
        K = np.zeros((B, Hkv, n_tok, 128), np.float16)
        for b in range(B):
            for g in range(Hkv):
                q[b, g * n_rep + 1:(g + 1) * n_rep] = q[b, g * n_rep]   # one query per group
                K[b, g] = _adversarial_keys(rng, q[b, g * n_rep], n_tok)
        V = rng.standard_normal((B, Hkv, n_tok, 128)).astype(np.float16)
        n, w = _check(q, K, V, 0.5, math.inf, n_rep)
        n_cert += n
        worst = max(worst, w)
    assert n_cert >= 300
    assert worst > 0.0
