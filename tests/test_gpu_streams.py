"""Decode calls on caller streams: a non-default stream, and two caches decoding at the
same time on two streams (each cache owns its scratch, work queues and counters).  The
results must equal those of the same calls made one after another on the default
stream, bit for bit."""

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import workloads as W  # noqa: E402


def _cache(q, K, V, **kw):
    B, Hq = q.shape[0], q.shape[1]
    Hkv, N = K.shape[1], K.shape[2]
    c = kvq.Cache(1, B, Hq, Hkv, max_ctx=N, **kw)
    c.append(0, K.cuda().contiguous(), V.cuda().contiguous())
    torch.cuda.synchronize()
    return c


def _decode(cache, q, stream=None, tau=0.995):
    B, Hq, D = q.shape
    out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
    lvl = torch.empty(B, dtype=torch.int32, device="cuda")
    cache.decode(0, q, tau, 0.25, out, cert, lvl, stream=stream)
    return out, cert, lvl


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.cpu(), y.cpu())


def test_non_default_stream_matches_default():
    q, K, V = W.c5_point(ctx=64 * 48 + 21, batch=2, Hq=8, Hkv=2)
    qd = q.cuda().contiguous()
    c = _cache(q, K, V)
    try:
        ref = _decode(c, qd)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            got = _decode(c, qd, stream=s)
        s.synchronize()
        _same(ref, got)
        # the uncertified path on the same stream
        out_ref = torch.empty_like(ref[0])
        c.decode_uncertified(0, qd, out_ref)
        torch.cuda.synchronize()
        out = torch.empty_like(ref[0])
        with torch.cuda.stream(s):
            c.decode_uncertified(0, qd, out, stream=s)
        s.synchronize()
        assert torch.equal(out, out_ref)
    finally:
        c.close()


def test_two_caches_on_two_streams_at_once():
    qa, Ka, Va = W.c1(seed=7, ctx=64 * 40 + 9, Hq=8, Hkv=2, batch=2)
    qb, Kb, Vb = W.c5_point(ctx=64 * 56 + 3, batch=1, Hq=8, Hkv=2)
    qa, qb = qa.cuda().contiguous(), qb.cuda().contiguous()
    ca, cb = _cache(qa.cpu(), Ka, Va), _cache(qb.cpu(), Kb, Vb, resident_blocks=64)
    try:
        ref_a, ref_b = [], []
        for _ in range(3):
            ref_a.append(_decode(ca, qa))
            ref_b.append(_decode(cb, qb))
        torch.cuda.synchronize()
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        for s in (sa, sb):
            s.wait_stream(torch.cuda.current_stream())
        got_a, got_b = [], []
        for _ in range(3):   # interleaved launches: the two caches' kernels overlap
            with torch.cuda.stream(sa):
                got_a.append(_decode(ca, qa, stream=sa))
            with torch.cuda.stream(sb):
                got_b.append(_decode(cb, qb, stream=sb))
        torch.cuda.synchronize()
        for r, g in zip(ref_a + ref_b, got_a + got_b):
            _same(r, g)
    finally:
        ca.close()
        cb.close()
