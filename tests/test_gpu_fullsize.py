"""Full-size workloads on the GPU, checked against the oracle on sampled KV groups.

The CUDA path decodes a whole 128K-token layer of the Llama-3.1-8B-shaped cache (and
the 32K x 4 low-rank workload) in the same launch configuration as bench.py; the
oracle then recomputes sampled (sequence, KV head) groups one by one.  Rung 4 depends
on every head of a sequence, so the sampled comparison asserts it did not fire.
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
from _parity import compare_decode  # noqa: E402


def _run_full(q, K, V, tau, eps, value_bits=4):
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N, value_bits=value_bits)
    try:
        cache.append(0, K.contiguous(), V.contiguous())
        out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
        lvl = torch.empty(B, dtype=torch.int32, device="cuda")
        cache.decode(0, q.contiguous(), tau, eps, out, cert, lvl)
        torch.cuda.synchronize()
        t1 = {k: v.cpu() for k, v in cache.export_tier1(0).items()}
        st = {k: v.cpu() for k, v in cache.export_decode_state(N // 64).items()}
    finally:
        cache.close()
    return out.cpu(), kvq.certificates(cert).reshape(B, Hq), lvl.cpu().numpy(), t1, st


def _check_groups(q, K, V, tau, eps, groups, value_bits=4):
    out, cert, lvl, t1g, st = _run_full(q, K, V, tau, eps, value_bits)
    assert np.all(lvl < 4), "rung 4 fired; sampled comparison does not apply"
    n_rep = q.shape[1] // K.shape[1]
    qc, Kc, Vc = q.cpu(), K.cpu(), V.cpu()
    for b, g in groups:
        hs = slice(g * n_rep, (g + 1) * n_rep)
        qs = qc[b:b + 1, hs].numpy()
        Ks, Vs = Kc[b:b + 1, g:g + 1].numpy(), Vc[b:b + 1, g:g + 1].numpy()
        t1 = O.quantize_layer(Ks, Vs)
        v4 = value_bits != 16
        for name in ("kc", "vc", "eta") if v4 else ("kc",):
            assert np.array_equal(t1g[name][b, g].numpy(), getattr(t1, name)[0, 0]), name
        for name in ("ks", "vs", "vo") if v4 else ("ks",):
            assert np.array_equal(t1g[name][b, g].numpy().view(np.uint16), getattr(t1, name)[0, 0].view(np.uint16)), name
        if not v4:
            assert np.all(t1g["eta"][b, g].numpy() == 0.0)
        r = O.decode_layer(qs, Ks, Vs, t1, tau, eps, O.OracleConfig(n_rep=n_rep, value_fp16=not v4))
        g_res = dict(out=out[b:b + 1, hs], cert=cert[b:b + 1, hs],
                     level=np.array([cert['level'][b, hs].max()]),   # rung over the sampled heads
                     nb=Ks.shape[2] // 64,
                     state={k: v[b:b + 1, hs] if v.shape[1] == q.shape[1] else v[b:b + 1, g:g + 1]
                            for k, v in st.items()})
        stats = compare_decode(g_res, t1, r, tau, eps, n_rep)
        assert stats["strict"] + stats["excluded"] == n_rep


def test_c3_layer_128k_sampled_groups():
    q, K, V = W.c3_layer(0, device="cuda")
    _check_groups(q, K, V, 0.995, 0.25, [(0, 0), (0, 5)])


def test_c2_lowrank_32k_b4_sampled_groups():
    q, K, V = W.c2(device="cuda")
    _check_groups(q, K, V, 0.995, 0.25, [(0, 3), (3, 7)])


def test_c3_layer_128k_fp16_values_sampled_groups():
    q, K, V = W.c3_layer(0, device="cuda")
    _check_groups(q, K, V, 0.995, 0.25, [(0, 2), (0, 6)], value_bits=16)


def test_c3_layer_128k_uncertified_sampled_groups():
    from _parity import BOUND_ATOL, BOUND_RTOL, OUT_ATOL, OUT_RTOL
    q, K, V = W.c3_layer(0, device="cuda")
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N)
    try:
        cache.append(0, K.contiguous(), V.contiguous())
        out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
        cache.decode_uncertified(0, q.contiguous(), out, cert)
        torch.cuda.synchronize()
        c = kvq.certificates(cert).reshape(B, Hq)
    finally:
        cache.close()
    n_rep = Hq // Hkv
    qc, Kc, Vc = q.cpu(), K.cpu(), V.cpu()
    for g in (1, 4):
        hs = slice(g * n_rep, (g + 1) * n_rep)
        Ks, Vs = Kc[0:1, g:g + 1].numpy(), Vc[0:1, g:g + 1].numpy()
        u = O.uncertified_decode_layer(qc[0:1, hs].numpy(), Ks, Vs, O.quantize_layer(Ks, Vs))
        err = np.abs(out[0, hs].cpu().float().numpy() - u.out64[0])
        assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(u.out64[0]))
        for name in ("e_key", "e_val"):
            gv, ov = c[name][0, hs].astype(np.float64), getattr(u, name)[0]
            assert np.all(np.abs(gv - ov) <= BOUND_RTOL * np.abs(ov) + BOUND_ATOL), name


def test_c4_planted_needle_64k_b8_rung4():
    """The planted-needle workload at full size (B = 8, 64K tokens, 32 query / 8 KV heads):
    INT8 rounding reverses the top block of every KV group, so every ranking check fails,
    every sequence takes rung 4 and every head returns dense attention over the FP16
    originals with E_key = E_val = 0.  Sampled heads are compared with the oracle's dense
    attention in float64."""
    from _parity import OUT_ATOL, OUT_RTOL
    q, K, V, info = W.c4(device="cuda")
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N)
    try:
        cache.append(0, K.half().contiguous(), V.half().contiguous())
        qh = q.half().contiguous()
        out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
        lvl = torch.empty(B, dtype=torch.int32, device="cuda")
        cache.decode(0, qh, 0.995, 0.25, out, cert, lvl)
        torch.cuda.synchronize()
    finally:
        cache.close()
    c = kvq.certificates(cert).reshape(B, Hq)
    assert np.all(lvl.cpu().numpy() == 4)
    assert np.all(c["level"] == 4) and np.all(c["e_key"] == 0) and np.all(c["e_val"] == 0)
    n_rep = Hq // Hkv
    for b, h in [(0, 0), (3, 13), (7, 31)]:
        g = h // n_rep
        o = O.dense_attention(qh[b, h].cpu().numpy(), K[b, g].half().cpu().numpy(), V[b, g].half().cpu().numpy())
        err = np.abs(out[b, h].cpu().float().numpy() - o)
        assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(o)), (b, h, float(err.max()))


def test_max_context_2m_tokens():
    """The largest cache a sequence may hold (max_ctx = 2,097,152 tokens: 32,768 blocks,
    the selection keeps one key per block in shared memory), one KV group of four query
    heads, plus a ragged partial block: the whole group is compared with the oracle."""
    N = (1 << 21)
    q, K, V = W.c3_layer(0, device="cuda", ctx=N, Hq=4, Hkv=1)
    # leave the last 37 tokens for a second append: the partial block at maximum size
    out, cert, lvl, t1g, st = None, None, None, None, None
    cache = kvq.Cache(1, 1, 4, 1, max_ctx=N)
    try:
        cache.append(0, K[:, :, :N - 37].contiguous(), V[:, :, :N - 37].contiguous())
        cache.append(0, K[:, :, N - 37:].contiguous(), V[:, :, N - 37:].contiguous())
        assert cache.length(0) == N
        o = torch.empty(1, 4, 128, dtype=torch.float16, device="cuda")
        c = torch.empty(4 * 32, dtype=torch.uint8, device="cuda")
        lv = torch.empty(1, dtype=torch.int32, device="cuda")
        cache.decode(0, q, 0.995, 0.25, o, c, lv)
        torch.cuda.synchronize()
        out, cert, lvl = o.cpu(), kvq.certificates(c).reshape(1, 4), lv.cpu().numpy()
        t1g = {k: v.cpu() for k, v in cache.export_tier1(0).items()}
        st = {k: v.cpu() for k, v in cache.export_decode_state(N // 64).items()}
    finally:
        cache.close()
    qc, Kc, Vc = q.cpu(), K.cpu(), V.cpu()
    del K, V
    t1 = O.quantize_layer(Kc.numpy(), Vc.numpy())
    for name in ("kc", "vc", "eta"):
        assert np.array_equal(t1g[name].numpy(), getattr(t1, name)), name
    r = O.decode_layer(qc.numpy(), Kc.numpy(), Vc.numpy(), t1, 0.995, 0.25, O.OracleConfig(n_rep=4))
    g_res = dict(out=out, cert=cert, level=lvl, nb=N // 64, state=st)
    # 32,768 blocks of nearly equal mass: blocks within the 1e-6 band of the boundary
    # block swap between the fp32 and fp64 selections, which changes the group's union,
    # so the group's levels and bounds are not compared strictly (min_strict 0); every
    # head's output still is
    stats = compare_decode(g_res, t1, r, 0.995, 0.25, 4, min_strict=0.0)
    assert stats["strict"] + stats["excluded"] == 4 and stats["out_compared"] == 4, stats

