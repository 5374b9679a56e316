"""CUDA path (through the C ABI) against the oracle, element by element.

Sizes span several 64-token blocks, 16-block work chunks and a ragged partial block.
Tolerances are defined in tests/_parity.py.
"""

import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import oracle as O  # noqa: E402
import workloads as W  # noqa: E402
from _parity import (compare_decode, compare_tier1, gpu_run, oracle_run)  # noqa: E402


def _check(q, K, V, tau, eps, chunks=None, **kw):
    g = gpu_run(q, K, V, tau, eps, chunks=chunks, **kw)
    t1, r = oracle_run(q, K, V, tau, eps, rank_positions=kw.get("rank_positions", 1),
                       l4=kw.get("l4", 0.5), v_tol=kw.get("v_tol", 0.0))
    compare_tier1(g["t1"], t1)
    st = compare_decode(g, t1, r, tau, eps, q.shape[1] // K.shape[1])
    return g, r, st


# ---------------------------------------------------------------------------------
# Method §1: quantise-and-append, bit-exact, any append pattern
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("chunks", [None, [1, 63, 64, 100, 1, 576], [64] * 12 + [37], [7] * 115])
def test_tier1_bit_exact(chunks):
    q, K, V = W.tiny(seed=3, ctx=805, Hq=8, Hkv=2, batch=2, kscale=3.0)
    g = gpu_run(q, K, V, 0.9, 0.25, chunks=chunks)
    t1, _ = oracle_run(q, K, V, 0.9, 0.25)
    compare_tier1(g["t1"], t1)


def test_tier1_edge_values():
    """Zero channels, constant groups, huge and tiny magnitudes, exact ties."""
    q, K, V = W.tiny(seed=4, ctx=64 * 4, Hq=4, Hkv=1)
    K = K.float(); V = V.float()
    K[:, :, :64, 3] = 0.0
    K[:, :, 64:128, :] *= 3000.0
    K[:, :, 128:192, :] *= 1e-4
    V[:, :, :64, :32] = 1.5
    V[:, :, 64:128, 32:64] *= 2000.0
    V[:, :, 192:, :] = torch.round(V[:, :, 192:, :] * 4) / 4
    g = gpu_run(q, K.half(), V.half(), 0.9, 0.25)
    t1, r = oracle_run(q, K.half(), V.half(), 0.9, 0.25)
    compare_tier1(g["t1"], t1)
    # the decode over the same cache: the x3000 block dominates every head (its block
    # log-mass is ~7000) with Delta ~ 250, so a softmax reference that added Delta to the
    # block log-mass would make every weight underflow; the oracle certifies every head at
    # rung 2 (the x2000 values of that block are paged in)
    st = compare_decode(g, t1, r, 0.9, 0.25, 4, min_strict=1.0)
    assert np.all(r.level == 2) and np.all(g["cert"]["level"] == 2), (r.level, g["cert"]["level"])
    assert np.all(np.isfinite(g["cert"]["e_key"])) and np.all(np.isfinite(g["cert"]["e_val"]))


def test_tier1_exact_ties():
    """Keys and values at exact half steps of their scales (code ties, resolved to even on
    both sides), next to values just off them: the quantiser's codes, scales and eta stay
    bit-exact with the oracle, including the rare path that divides exactly."""
    gen = torch.Generator().manual_seed(21)
    n_blk, D = 6, 128
    N = 64 * n_blk + 7
    s0, v0 = 2.0 ** -5, 2.0 ** -3
    K = torch.zeros(1, 2, N, D, dtype=torch.float64)
    V = torch.zeros(1, 2, N, D, dtype=torch.float64)
    for b in range(n_blk):
        rows = slice(64 * b, 64 * b + 64)
        n = torch.randint(-126, 126, (64, D), generator=gen).double()
        K[0, :, rows] = (n + 0.5) * s0                       # K / s = n + 1/2 exactly
        K[0, :, 64 * b] = 127 * s0                            # pins every channel scale to s0
        m = torch.randint(0, 15, (64, D), generator=gen).double()
        V[0, :, rows] = (m + 0.5) * v0
        V[0, :, rows, 0::32] = 0.0                            # group min 0 ...
        V[0, :, rows, 1::32] = 15 * v0                        # ... and max 15 v0: scale v0
        if b % 2:                                             # just off the ties: +- 2^-11 v0
            V[0, :, rows, 2::5] += v0 * 2.0 ** -11 * torch.sign(torch.randn(64, 26, generator=gen)).double()[:, :1]
    K[0, :, 64 * n_blk:] = torch.randn(2, 7, D, generator=gen).double()
    V[0, :, 64 * n_blk:] = torch.randn(2, 7, D, generator=gen).double()
    q = torch.randn(1, 8, D, generator=gen).half()
    g = gpu_run(q, K.half(), V.half(), 0.9, 0.25, chunks=[100, N - 100])
    t1, _ = oracle_run(q, K.half(), V.half(), 0.9, 0.25)
    compare_tier1(g["t1"], t1)
    assert np.any(t1.kc % 2 == 0) and np.any(t1.kc % 2 != 0)


@pytest.mark.parametrize("kscale", [60.0, 200.0])
def test_decode_large_delta(kscale):
    """Keys scaled x60 and x200 (Delta ~ 7 and ~ 25 per block, peaked attention): the
    softmax reference sits at the largest INT8 block log-mass, not Delta above it, so the
    INT4-path weight products stay normal binary16 numbers; every head strictly compared."""
    q, K, V = W.tiny(seed=13, ctx=64 * 24 + 5, Hq=8, Hkv=2, batch=2, kscale=kscale)
    g, r, st = _check(q, K, V, 0.95, 0.25)
    assert float(np.max(r.delta)) > (20.0 if kscale > 100 else 5.0)


# ---------------------------------------------------------------------------------
# Method §2-§3: decode parity
# ---------------------------------------------------------------------------------

def test_decode_c1_shape():
    q, K, V = W.c1()                       # 4096 tokens, 32 q heads / 8 KV heads
    g, r, st = _check(q, K, V, 0.995, 0.25)
    assert st["strict"] >= 24, st


# 256 / 257 full blocks: either side of the point where the block selection ranks every
# block exactly instead of narrowing them down by histogram levels first
@pytest.mark.parametrize("ctx", [64 * 16, 64 * 16 + 1, 64 * 33 + 63, 37, 64, 64 * 256 + 7, 64 * 257,
                                 64 * 700 + 5, 64 * 2100])
def test_decode_ragged(ctx):
    q, K, V = W.tiny(seed=5, ctx=ctx, Hq=8, Hkv=2, batch=2, kscale=3.0)
    _check(q, K, V, 0.95, 0.25, chunks=[ctx // 3, ctx - ctx // 3])


@pytest.mark.parametrize("n_rep", [1, 2, 3])
def test_decode_gqa_widths(n_rep):
    q, K, V = W.tiny(seed=6, ctx=64 * 20 + 9, Hq=2 * n_rep, Hkv=2, kscale=3.0)
    _check(q, K, V, 0.95, 0.25)


def test_ladder_rungs_parity():
    """Value groups with an 8x range push heads to rung 2; a tight eps adds rung 1."""
    q, K, V = W.tiny(seed=7, ctx=64 * 40 + 11, Hq=8, Hkv=2, kscale=6.0)
    V = V.float()
    V[:, :, :, :32] *= 8
    V = V.half()
    for tau, eps in [(0.995, 0.25), (0.8, 0.25), (0.5, 0.3), (0.9, 0.05)]:
        g, r, st = _check(q, K, V, tau, eps)
        assert st["strict"] > 0


def test_rung_levels_seen():
    q, K, V = W.c3_layer(0, ctx=8192, Hq=8, Hkv=2)
    g, r, st = _check(q, K, V, 0.995, 0.25)
    assert (r.planned >= 1).any(), "workload did not reach rungs 1-2"


def test_tau_one_is_dense():
    q, K, V = W.tiny(seed=8, ctx=64 * 10 + 3, Hq=8, Hkv=2, kscale=3.0)
    g = gpu_run(q, K, V, 1.0, 0.25)
    assert np.all(g["cert"]["level"] == 4) and np.all(g["cert"]["e_key"] == 0)
    for h in range(8):
        dense = O.dense_attention(q[0, h].numpy(), K[0, h // 4].numpy(), V[0, h // 4].numpy())
        assert np.allclose(g["out"][0, h].float().numpy(), dense, atol=2e-3, rtol=1e-2)


def test_forced_rank_failure_goes_dense():
    q, K, V = W.tiny(seed=9, ctx=64 * 10 + 3, Hq=8, Hkv=2, kscale=3.0)
    g = gpu_run(q, K, V, 0.95, 0.25, debug=kvq.DEBUG_FORCE_RANK_FAIL)
    assert np.all(g["cert"]["rank_ok"] == 0)
    assert np.all(g["cert"]["level"] == 4) and np.all(g["level"] == 4)
    for h in range(8):
        dense = O.dense_attention(q[0, h].numpy(), K[0, h // 4].numpy(), V[0, h // 4].numpy())
        assert np.allclose(g["out"][0, h].float().numpy(), dense, atol=2e-3, rtol=1e-2)


def test_planted_block_fires_rank_check():
    q, K, V, info = W.c4(batch=2, ctx=8192, Hq=8, Hkv=2)
    g, r, st = _check(q, K, V, 0.995, 0.25)
    assert np.all(g["cert"]["rank_ok"] == 0)
    assert np.all(g["level"] == 4)


def test_eps_special_cases():
    q, K, V = W.tiny(seed=10, ctx=64 * 12 + 5, Hq=8, Hkv=2, kscale=3.0)
    g, r, st = _check(q, K, V, 0.9, math.inf)
    c = g["cert"]
    assert np.all((c["level"] == 0) | (c["rank_ok"] == 0))
    g0, r0, st0 = _check(q, K, V, 0.9, 0.0)
    c0 = g0["cert"]
    assert np.all((c0["level"] >= 3) | ((c0["e_key"] == 0) & (c0["e_val"] == 0)))


def test_host_buffers_match_device_buffers():
    q, K, V = W.tiny(seed=11, ctx=64 * 9 + 1, Hq=8, Hkv=2, kscale=3.0)
    gd = gpu_run(q, K, V, 0.95, 0.25)
    gh = gpu_run(q, K, V, 0.95, 0.25, host_io=True)
    assert torch.equal(gd["out"], gh["out"])
    assert np.array_equal(gd["cert"], gh["cert"]) and np.array_equal(gd["level"], gh["level"])


def test_pageable_host_buffers_are_ready_on_return():
    """Pageable host outputs hold the results when the call returns (no synchronise by
    the caller); page-locked ones are copied in stream order and match after one."""
    q, K, V = W.tiny(seed=12, ctx=64 * 7 + 5, Hq=8, Hkv=2, kscale=3.0)
    B, Hq, D = q.shape
    cache = kvq.Cache(1, B, Hq, K.shape[1], max_ctx=K.shape[2])
    try:
        cache.append(0, K.cuda().contiguous(), V.cuda().contiguous())
        out_d = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        cert_d = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
        cache.decode(0, q.cuda().contiguous(), 0.95, 0.25, out_d, cert_d)
        torch.cuda.synchronize()
        ref_out, ref_cert = out_d.cpu(), kvq.certificates(cert_d)
        out_h = torch.full((B, Hq, D), float("nan"), dtype=torch.float16)   # pageable
        cert_h = torch.zeros(B * Hq * 32, dtype=torch.uint8)
        cache.decode(0, q.contiguous(), 0.95, 0.25, out_h, cert_h)
        assert torch.equal(out_h, ref_out)
        assert np.array_equal(kvq.certificates(cert_h), ref_cert)
        out_p = torch.full((B, Hq, D), float("nan"), dtype=torch.float16).pin_memory()
        cert_p = torch.zeros(B * Hq * 32, dtype=torch.uint8).pin_memory()
        cache.decode(0, q.contiguous().pin_memory(), 0.95, 0.25, out_p, cert_p)
        torch.cuda.synchronize()
        assert torch.equal(out_p, ref_out)
        assert np.array_equal(kvq.certificates(cert_p), ref_cert)
    finally:
        cache.close()


def test_deterministic_repeat():
    q, K, V = W.c1(ctx=64 * 50 + 7, Hq=8, Hkv=2)
    g = gpu_run(q, K, V, 0.995, 0.25, repeat=3)
    o0, c0, l0 = g["runs"][0]
    for o, c, l in g["runs"][1:]:
        assert torch.equal(o, o0) and np.array_equal(c, c0) and np.array_equal(l, l0)


def test_rank_positions_two():
    q, K, V = W.tiny(seed=12, ctx=64 * 30 + 2, Hq=8, Hkv=2, kscale=4.0)
    _check(q, K, V, 0.9, 0.25, rank_positions=2)


# ---------------------------------------------------------------------------------
# C-ABI error behaviour
# ---------------------------------------------------------------------------------

def test_errors():
    cache = kvq.Cache(1, 1, 4, 1, max_ctx=128)
    try:
        q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
        out = torch.empty_like(q)
        with pytest.raises(kvq.KvqError) as e:
            cache.decode(0, q, 0.9, 0.25, out)       # empty layer
        assert e.value.status == kvq.KVQ_ERR_INVALID
        k = torch.zeros(1, 1, 100, 128, dtype=torch.float16, device="cuda")
        cache.append(0, k, k)
        with pytest.raises(kvq.KvqError) as e:
            cache.append(0, k, k)                    # 200 > max_ctx
        assert e.value.status == kvq.KVQ_ERR_CAPACITY
        assert cache.length(0) == 100
        for tau, eps in [(0.0, 0.25), (1.5, 0.25), (0.9, -1.0), (0.9, float("nan"))]:
            with pytest.raises(kvq.KvqError) as e:
                cache.decode(0, q, tau, eps, out)
            assert e.value.status == kvq.KVQ_ERR_INVALID
        with pytest.raises(kvq.KvqError):
            cache.decode(1, q, 0.9, 0.25, out)       # layer out of range
        cache.decode(0, q, 0.9, 0.25, out)           # still usable
    finally:
        cache.close()
    with pytest.raises(kvq.KvqError) as e:
        kvq.Cache(1, 1, 6, 1, max_ctx=128)           # n_rep = 6 unsupported
    assert e.value.status == kvq.KVQ_ERR_INVALID


def _offset_view(shape, dtype, byte_offset):
    """A contiguous CUDA tensor of `shape` that starts `byte_offset` bytes into an
    allocation (torch's CUDA allocations start 256-byte aligned)."""
    es = torch.empty(0, dtype=dtype).element_size()
    assert byte_offset % es == 0
    n = math.prod(shape)
    raw = torch.zeros(n * es + 256, dtype=torch.uint8, device="cuda")
    return raw[byte_offset:byte_offset + n * es].view(dtype).view(shape)


def test_unaligned_device_buffers_are_rejected():
    """The kernels read and write device buffers in place with vector accesses; buffers
    that are not aligned for them are refused before anything is enqueued, and the cache
    stays usable."""
    cache = kvq.Cache(1, 1, 4, 1, max_ctx=256)
    try:
        k = torch.randn(1, 1, 100, 128, device="cuda").half()
        kb = _offset_view((1, 1, 100, 128), torch.float16, 2)
        kb.copy_(k)
        assert kb.data_ptr() % 16 == 2
        with pytest.raises(kvq.KvqError) as e:
            cache.append(0, kb, k)
        assert e.value.status == kvq.KVQ_ERR_INVALID and "aligned" in str(e.value)
        assert cache.length(0) == 0
        cache.append(0, k, k)
        q = torch.randn(1, 4, 128, device="cuda").half()
        out = torch.empty_like(q)
        qb = _offset_view((1, 4, 128), torch.float16, 8)
        qb.copy_(q)
        ob = _offset_view((1, 4, 128), torch.float16, 6)
        for qq, oo in [(qb, out), (q, ob)]:
            with pytest.raises(kvq.KvqError) as e:
                cache.decode(0, qq, 0.9, 0.25, oo)
            assert e.value.status == kvq.KVQ_ERR_INVALID
            with pytest.raises(kvq.KvqError) as e:
                cache.decode_uncertified(0, qq, oo)
            assert e.value.status == kvq.KVQ_ERR_INVALID
        cert_bad = _offset_view((4 * 32,), torch.uint8, 4)
        with pytest.raises(kvq.KvqError) as e:
            cache.decode(0, q, 0.9, 0.25, out, cert=cert_bad)
        assert e.value.status == kvq.KVQ_ERR_INVALID
        # an int32 tensor is always 4-byte aligned, so the misaligned ladder-level buffer
        # goes to the C entry point directly
        lvl_bad = _offset_view((8,), torch.uint8, 2)
        st = cache.lib.kvq_decode_attention(cache.handle, 0, q.data_ptr(), 0.9, 0.25, out.data_ptr(),
                                            None, lvl_bad.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == kvq.KVQ_ERR_INVALID
        # the binding refuses wrong dtypes and shapes before the C call
        with pytest.raises(ValueError):
            cache.decode(0, q.float(), 0.9, 0.25, out)
        with pytest.raises(ValueError):
            cache.decode(0, q[:, :2].contiguous(), 0.9, 0.25, out)
        with pytest.raises(ValueError):
            cache.append(0, k.float(), k.float())
        torch.cuda.synchronize()
        cache.decode(0, q, 0.9, 0.25, out)           # still usable
        ref = torch.empty_like(q)
        cache.decode(0, qb.clone(), 0.9, 0.25, ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    finally:
        cache.close()
    q = torch.randn(1, 4, 128, device="cuda").half()
    k = torch.randn(1, 1, 64, 128, device="cuda").half()
    out = torch.empty_like(q)
    qb = _offset_view((1, 4, 128), torch.float16, 2)
    with pytest.raises(kvq.KvqError) as e:
        kvq.dense_decode_noalloc(qb, k, k, out)
    assert e.value.status == kvq.KVQ_ERR_INVALID


# ---------------------------------------------------------------------------------
# value tolerance v_tol (Results: structured reasoning)
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("v_tol", [0.1, 0.03])
def test_value_tolerance(v_tol):
    q, K, V = W.c5_point(64 * 120 + 9, 2, Hq=8, Hkv=2)
    g, r, st = _check(q, K, V, 0.99, 0.5, v_tol=v_tol)
    c = g["cert"]
    ok = c["level"] < 3
    assert np.all(c["e_val"][ok] <= v_tol * (1 + 1e-4))
    assert np.any(c["level"] == 2)


def test_tier1_passes_never_read_tier2():
    """The scoring pass, the selection, the INT8/INT4 pass and its combine use tier 1 only
    (the bounds' inputs come without FP16 data, Method §2): the uncertified call gives
    bit-identical outputs and bounds after tier 2 is overwritten with NaN, while a dense
    call (tau_cov = 1, every block read from tier 2) then returns NaN."""
    q, K, V = W.tiny(seed=80, ctx=64 * 40 + 5, Hq=8, Hkv=2, batch=2, kscale=3.0)
    cache = kvq.Cache(1, 2, 8, 2, max_ctx=64 * 41)
    try:
        cache.append(0, K.cuda().contiguous(), V.cuda().contiguous())
        qd = q.cuda().contiguous()
        runs = []
        for poison in (False, True):
            if poison:
                cache.debug_fill_tier2(0, 0x7E00)   # binary16 NaN
            out = torch.empty(2, 8, 128, dtype=torch.float16, device="cuda")
            cert = torch.empty(2 * 8 * 32, dtype=torch.uint8, device="cuda")
            cache.decode_uncertified(0, qd, out, cert)
            torch.cuda.synchronize()
            runs.append((out.cpu(), cert.cpu()))
        assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1])
        assert torch.isfinite(runs[1][0].float()).all()
        out = torch.empty(2, 8, 128, dtype=torch.float16, device="cuda")
        cache.decode(0, qd, 1.0, 0.25, out)
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all()
    finally:
        cache.close()


def test_token_by_token_appends_feed_tier2():
    """One token per append (the serving loop): tokens that stay in the partial block are
    mirrored to tier 2 from the partial-block buffer without a join; blocks they later
    complete are paged in correctly (tau = 1 reads every full block from tier 2), and the
    certified path matches the oracle."""
    q, K, V = W.tiny(seed=70, ctx=64 * 3 + 29, Hq=8, Hkv=2, kscale=3.0)
    N = K.shape[2]
    g = gpu_run(q, K, V, 1.0, 0.25, chunks=[1] * N)
    for h in range(8):
        dense = O.dense_attention(q[0, h].numpy(), K[0, h // 4].numpy(), V[0, h // 4].numpy())
        assert np.allclose(g["out"][0, h].float().numpy(), dense, atol=2e-3, rtol=1e-2)
    _check(q, K, V, 0.9, 0.25, chunks=[1] * 100 + [5] * 20 + [N - 200])

