"""Cross-step residency of FP16 tier-2 blocks (kvq_config.resident_blocks).

Not a step of the paper's method: an option of this library that keeps FP16 blocks
paged in by one decode call in HBM for later calls.  The resident copies are
bit-identical to tier 2, so every output and certificate must equal those of a cache
without residency (bit for bit) and match the oracle; the byte counters must account
for every FP16 block the call pages in, split into HBM hits and host-link reads.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import workloads as W  # noqa: E402
from _parity import compare_decode, oracle_run  # noqa: E402

BLOCK_BYTES = 16384


def _calls(K, V, queries, tau, eps, resident_blocks, value_bits=4, uncertified_between=False):
    """Decode each query in turn on one cache; per call: out, cert, residency stats."""
    B, Hkv, N, D = K.shape
    Hq = queries[0].shape[1]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=N, value_bits=value_bits, resident_blocks=resident_blocks)
    res = []
    try:
        cache.append(0, K.cuda().contiguous(), V.cuda().contiguous())
        for q in queries:
            out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
            cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
            lvl = torch.empty(B, dtype=torch.int32, device="cuda")
            cache.decode(0, q.cuda().contiguous(), tau, eps, out, cert, lvl)
            torch.cuda.synchronize()
            st = cache.residency_stats(0, reset=True)
            if uncertified_between:   # pages nothing in, so it must leave the slots alone
                cache.decode_uncertified(0, q.cuda().contiguous(), torch.empty_like(out))
                torch.cuda.synchronize()
                assert cache.residency_stats(0, reset=True)["host_bytes"] == 0
            c = kvq.certificates(cert).reshape(B, Hq)
            res.append(dict(out=out.cpu(), cert=c, level=lvl.cpu().numpy(), stats=st,
                            paged=int(c["promoted_bytes"][:, ::Hq // Hkv].sum())))
    finally:
        cache.close()
    return res


def _same(a, b):
    assert torch.equal(a["out"], b["out"]), "output differs from the cache without residency"
    assert a["cert"].tobytes() == b["cert"].tobytes(), "certificate differs"
    assert np.array_equal(a["level"], b["level"])


def _oracle_check(q, K, V, tau, eps, run, value_bits=4):
    t1, r = oracle_run(q, K, V, tau, eps, value_bits=value_bits)
    g = dict(out=run["out"], cert=run["cert"], level=run["level"], state=None, nb=K.shape[2] // 64)
    compare_decode(g, t1, r, tau, eps, q.shape[1] // K.shape[1], check_sets=False)


@pytest.mark.parametrize("make", ["c1", "c5"])
def test_repeat_call_served_from_hbm(make):
    """Capacity above the working set: the second call reads nothing over the host link."""
    q, K, V = W.c1() if make == "c1" else W.c5_point(ctx=4096, batch=1)
    tau, eps = 0.995, 0.25
    base = _calls(K, V, [q, q], tau, eps, 0)
    res = _calls(K, V, [q, q], tau, eps, 2 * 8 * 64)
    for a, b in zip(res, base):
        _same(a, b)
    first, second = res[0]["stats"], res[1]["stats"]
    assert res[0]["paged"] > 0
    # every distinct block misses once in the first call and takes a slot; a value block
    # a dense rung reads again in the same call is already a hit
    assert first["resident_bytes"] + first["host_bytes"] == res[0]["paged"]
    assert first["host_bytes"] == first["slots_in_use"] * BLOCK_BYTES
    assert second == dict(resident_bytes=res[1]["paged"], host_bytes=0,
                          slots_in_use=first["slots_in_use"])
    _oracle_check(q, K, V, tau, eps, res[1])


@pytest.mark.parametrize("make", ["c5", "c2"])
def test_capacity_below_working_set(make):
    """With S slots every later identical call finds the same S blocks resident: exactly
    S hits when no dense rung runs (no block is read twice in one call), at most 2 S when
    one does (a value block of rung 2 is read again by the dense rung)."""
    q, K, V = W.c5_point(ctx=4096, batch=1) if make == "c5" else W.c2(batch=1, ctx=64 * 96)
    S = 50 if make == "c5" else 16   # c2 pages in about 40 key blocks
    res = _calls(K, V, [q, q, q], 0.995, 0.25, S)
    base = _calls(K, V, [q], 0.995, 0.25, 0)
    dense = int(base[0]["level"].max()) >= 3
    assert res[0]["paged"] > S * BLOCK_BYTES
    for r in res:
        _same(r, base[0])
        assert r["stats"]["resident_bytes"] + r["stats"]["host_bytes"] == r["paged"]
        assert r["stats"]["slots_in_use"] == S
    for r in res[1:]:
        hit = r["stats"]["resident_bytes"]
        if dense:
            assert S * BLOCK_BYTES <= hit <= 2 * S * BLOCK_BYTES
        else:
            assert hit == S * BLOCK_BYTES


def test_changing_queries_and_eviction():
    """Different queries select different blocks; slots a call does not use are freed."""
    q1, K, V = W.c2(batch=1, ctx=64 * 96)
    gen = torch.Generator().manual_seed(12)
    q2 = torch.randn(q1.shape, generator=gen).half()
    qs = [q1, q2, q1]
    tau, eps = 0.995, 0.25
    res = _calls(K, V, qs, tau, eps, 4096)
    base = _calls(K, V, qs, tau, eps, 0)
    for a, b in zip(res, base):
        _same(a, b)
        st = a["stats"]
        assert st["resident_bytes"] + st["host_bytes"] == a["paged"]
        # capacity exceeds every call's working set: what a call used stays, the rest is freed
        assert 0 < st["slots_in_use"] <= a["paged"] // BLOCK_BYTES
    for q, r in zip(qs, res):
        _oracle_check(q, K, V, tau, eps, r)


def test_dense_rungs_and_uncertified_calls():
    """tau_cov = 1 pages every key and value block in (rung 4); uncertified calls in
    between leave the slots untouched."""
    q, K, V = W.tiny(seed=21, ctx=64 * 40 + 17, Hq=8, Hkv=2, batch=2, kscale=3.0)
    res = _calls(K, V, [q, q], 1.0, 0.25, 2 * 2 * 2 * 40, uncertified_between=True)
    base = _calls(K, V, [q], 1.0, 0.25, 0)
    _same(res[0], base[0])
    _same(res[1], base[0])
    assert res[0]["paged"] == 2 * 2 * 2 * 40 * BLOCK_BYTES
    assert res[1]["stats"] == dict(resident_bytes=res[1]["paged"], host_bytes=0, slots_in_use=320)
    _oracle_check(q, K, V, 1.0, 0.25, res[1])


def test_fp16_values_configuration():
    """value_bits 16: only keys live in tier 2, so only keys are made resident."""
    q, K, V = W.c1()
    res = _calls(K, V, [q, q], 0.995, 0.25, 512, value_bits=16)
    base = _calls(K, V, [q, q], 0.995, 0.25, 0, value_bits=16)
    for a, b in zip(res, base):
        _same(a, b)
    assert res[1]["stats"]["host_bytes"] == 0
    _oracle_check(q, K, V, 0.995, 0.25, res[1], value_bits=16)


def test_serving_loop_with_appends():
    """Decode steps interleaved with appends (some completing a block, some not): blocks
    completed after a slot table was filled must be paged in from tier 2, and every step
    must equal the cache without residency bit for bit."""
    q0, K, V = W.c1(ctx=64 * 20 + 50, Hq=8, Hkv=2, batch=2)
    gen = torch.Generator().manual_seed(31)
    steps = [(int(n), torch.randn(q0.shape, generator=gen).half()) for n in (1, 13, 64, 2, 70)]
    B, Hkv, N0, D = K.shape
    extra = sum(n for n, _ in steps)
    Kx = torch.randn(B, Hkv, extra, D, generator=gen).half()
    Vx = torch.randn(B, Hkv, extra, D, generator=gen).half()

    def run(slots):
        cache = kvq.Cache(1, B, q0.shape[1], Hkv, max_ctx=N0 + extra, resident_blocks=slots)
        outs, pos = [], 0
        try:
            cache.append(0, K.cuda().contiguous(), V.cuda().contiguous())
            for n, q in steps:
                cache.append(0, Kx[:, :, pos:pos + n].cuda().contiguous(), Vx[:, :, pos:pos + n].cuda().contiguous())
                pos += n
                out = torch.empty(B, q.shape[1], D, dtype=torch.float16, device="cuda")
                cert = torch.empty(B * q.shape[1] * 32, dtype=torch.uint8, device="cuda")
                cache.decode(0, q.cuda().contiguous(), 0.995, 0.25, out, cert)
                torch.cuda.synchronize()
                outs.append((out.cpu(), kvq.certificates(cert).tobytes(), cache.residency_stats(0, reset=True)))
        finally:
            cache.close()
        return outs

    base, res = run(0), run(4096)
    for (ob, cb, _), (orr, cr, st) in zip(base, res):
        assert torch.equal(ob, orr) and cb == cr
    assert res[-1][2]["resident_bytes"] > 0
    # the final state against the oracle
    pos = extra
    Kf = torch.cat([K, Kx], dim=2)
    Vf = torch.cat([V, Vx], dim=2)
    c = kvq.certificates(res[-1][1]).reshape(B, q0.shape[1])
    _oracle_check(steps[-1][1], Kf, Vf, 0.995, 0.25,
                  dict(out=res[-1][0], cert=c, level=c["level"].max(axis=1)))


@pytest.mark.parametrize("ctx", [37, 64, 64 * 3 + 5])
def test_short_layers(ctx):
    """Layers with no or few full blocks: the eviction pass and the slot table must cope
    with nothing (or almost nothing) to page in."""
    q, K, V = W.tiny(seed=40 + ctx, ctx=ctx, Hq=8, Hkv=2, batch=2, kscale=3.0)
    base = _calls(K, V, [q, q], 0.995, 0.25, 0)
    res = _calls(K, V, [q, q], 0.995, 0.25, 16, uncertified_between=True)
    for a, b in zip(res, base):
        _same(a, b)
        assert a["stats"]["resident_bytes"] + a["stats"]["host_bytes"] == a["paged"]
    _oracle_check(q, K, V, 0.995, 0.25, res[1])
