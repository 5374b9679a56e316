"""Helpers that run the CUDA path (through the C ABI) and the oracle on the same inputs
and compare them.  Imported by the GPU tests only.

Tolerances (stated once, used everywhere):
  * codes, scales, eta, value ranges: bit-exact;
  * selected block sets and ladder decisions: exact, excluding blocks whose cumulative
    covered mass lies within SEL_BAND of tau_cov (and blocks whose mass is within
    SEL_BAND of the boundary block's), and heads whose deciding quantity is within
    relative DECIDE_REL of its threshold;
  * outputs: max-abs |gpu - oracle| <= OUT_ATOL (2e-3) for every head whose oracle
    outputs lie within +-OUT_STRICT_RANGE, and |gpu - oracle| <= OUT_ATOL + OUT_RTOL |oracle|
    beyond (the returned output is binary16, whose rounding alone is 2^-11 relative and
    exceeds 2e-3 above |x| = 4);
  * bounds: |gpu - oracle| <= BOUND_RTOL |oracle| + BOUND_ATOL;
  * coverage: at least MIN_STRICT_FRAC of the heads of every call are compared strictly
    (level, ranking-check outcome and bounds), unless a test states a lower share and why.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import certified_quantized_kv_gb300 as kvq
import oracle as O

SEL_BAND = 1e-6
DECIDE_REL = 1e-4
OUT_ATOL = 2e-3
OUT_RTOL = 1e-2
OUT_STRICT_RANGE = 2.0
MIN_STRICT_FRAC = 0.5
BOUND_RTOL = 1e-4
BOUND_ATOL = 1e-6


def gpu_run(q, K, V, tau, eps, chunks=None, debug=0, rank_positions=1, l4=0.5, max_ctx=None,
            host_io=False, repeat=1, value_bits=4, v_tol=0.0):
    """Append K, V (CPU fp16 tensors [B, Hkv, N, D]) in `chunks` and decode once."""
    B, Hq, D = q.shape
    Hkv, N = K.shape[1], K.shape[2]
    cache = kvq.Cache(1, B, Hq, Hkv, max_ctx=max_ctx or max(N, 1), rank_positions=rank_positions,
                      l4_head_fraction=l4, value_bits=value_bits, v_tol=v_tol)
    try:
        cache.set_debug(debug)
        Kd, Vd = K.cuda(), V.cuda()
        pos = 0
        for n in (chunks or [N]):
            if n == 0:
                continue
            cache.append(0, Kd[:, :, pos:pos + n].contiguous(), Vd[:, :, pos:pos + n].contiguous())
            pos += n
        assert pos == N
        outs = []
        for _ in range(repeat):
            if host_io:
                out = torch.empty(B, Hq, D, dtype=torch.float16).pin_memory()
                cert = torch.empty(B * Hq * 32, dtype=torch.uint8).pin_memory()
                lvl = torch.empty(B, dtype=torch.int32).pin_memory()
                cache.decode(0, q.contiguous(), tau, eps, out, cert, lvl)
            else:
                out = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
                cert = torch.empty(B * Hq * 32, dtype=torch.uint8, device="cuda")
                lvl = torch.empty(B, dtype=torch.int32, device="cuda")
                cache.decode(0, q.cuda().contiguous(), tau, eps, out, cert, lvl)
            torch.cuda.synchronize()
            outs.append((out.cpu(), kvq.certificates(cert).reshape(B, Hq), lvl.cpu().numpy()))
        t1 = {k: v.cpu() for k, v in cache.export_tier1(0).items()}
        nb = N // 64
        st = None
        if tau < 1.0 and not (debug & kvq.DEBUG_FORCE_DENSE):
            st = {k: v.cpu() for k, v in cache.export_decode_state(nb).items()}
        torch.cuda.synchronize()
    finally:
        cache.close()
    out, cert, lvl = outs[-1]
    return dict(out=out, cert=cert, level=lvl, t1=t1, state=st, nb=nb, runs=outs)


def oracle_run(q, K, V, tau, eps, rank_positions=1, l4=0.5, value_bits=4, v_tol=0.0):
    qn, Kn, Vn = q.numpy(), K.numpy(), V.numpy()
    t1 = O.quantize_layer(Kn, Vn)
    cfg = O.OracleConfig(n_rep=q.shape[1] // K.shape[1], rank_positions=rank_positions,
                         l4_head_fraction=l4, value_fp16=value_bits == 16,
                         v_tol=v_tol if v_tol > 0 else math.inf)
    return t1, O.decode_layer(qn, Kn, Vn, t1, tau, eps, cfg)


def compare_tier1(g, t1, value_bits=4):
    assert np.array_equal(g["kc"].numpy(), t1.kc), "INT8 key codes differ"
    assert np.array_equal(g["ks"].numpy().view(np.uint16), t1.ks.view(np.uint16)), "key scales differ"
    if value_bits == 16:   # FP16 values: no INT4 codes exist, eta is zero
        assert np.all(g["eta"].numpy() == 0.0), "eta must be zero with FP16 values"
        assert np.array_equal(g["vmin"].numpy(), t1.vmin) and np.array_equal(g["vmax"].numpy(), t1.vmax)
        return
    assert np.array_equal(g["vc"].numpy(), t1.vc), "INT4 value codes differ"
    assert np.array_equal(g["vs"].numpy().view(np.uint16), t1.vs.view(np.uint16)), "value scales differ"
    assert np.array_equal(g["vo"].numpy().view(np.uint16), t1.vo.view(np.uint16)), "value offsets differ"
    assert np.array_equal(g["eta"].numpy().view(np.uint32), t1.eta.view(np.uint32)), "eta differs"
    assert np.array_equal(g["vmin"].numpy(), t1.vmin) and np.array_equal(g["vmax"].numpy(), t1.vmax)


def ambiguous_blocks(r: O.DecodeResult, b: int, h: int, tau: float, band: float = SEL_BAND) -> set:
    """Blocks whose membership in S_h is decided within `band` of the coverage threshold."""
    sel, cum = r.sel[b][h], r.cum[b][h]
    mass = r.mass[b, h]
    amb = set()
    if mass.size == 0:
        return amb
    order = sorted(range(mass.size), key=lambda i: (-mass[i], i))
    k = len(sel)
    before_last = cum[-2] if k >= 2 else (cum[0] - mass[sel[0]] if k == 1 else None)
    if k > 0:
        after_last = cum[-1]
        if abs(after_last - tau) <= band or (before_last is not None and abs(before_last - tau) <= band):
            amb.add(sel[-1])
            if k < mass.size:
                amb.add(order[k])
    # blocks nearly tied with the boundary block may swap order across it
    m_b = mass[sel[-1]] if k > 0 else mass[order[0]]
    amb |= {i for i in range(mass.size) if abs(mass[i] - m_b) <= band}
    if k < mass.size:
        m_n = mass[order[k]]
        amb |= {i for i in range(mass.size) if abs(mass[i] - m_n) <= band}
    return amb


def marginal_head(r: O.DecodeResult, b: int, h: int, eps: float) -> bool:
    """Head whose rung is decided within DECIDE_REL of a threshold."""
    def near(x, t):
        if not math.isfinite(t):
            return False
        if t == 0:   # an exact zero bound (nothing left in INT8) is exact on both sides
            return 0 < abs(x) <= 1e-30
        return abs(x - t) <= DECIDE_REL * abs(t)
    e0 = r.e_key0[b, h] + r.e_val0[b, h]
    if near(e0, eps) or near(r.e_key0[b, h], eps / 2):
        return True
    if r.round1[b, h] and near(r.e_key[b, h] + r.e_val[b, h], eps):
        return True
    sel = r.sel[b][h]
    if len(sel) > 1:
        for arr in (r.lse8[b, h], r.lse16[b, h]):
            v = np.sort(arr[sel])[::-1]
            if v[0] - v[1] <= DECIDE_REL:
                return True
    return False


def compare_decode(g, t1, r: O.DecodeResult, tau, eps, n_rep, check_sets=True,
                   min_strict=MIN_STRICT_FRAC):
    """Compare one decode call; returns a dict of counters for reporting."""
    out_g = g["out"].float().numpy()
    cert = g["cert"]
    B, Hq, _ = out_g.shape
    Hkv = Hq // n_rep
    nb = g["nb"]
    stats = dict(heads=0, strict=0, excluded=0, out_compared=0, set_mismatch_groups=0,
                 max_out_err=0.0, max_out_err_unit_range=0.0, max_bound_rel=0.0)
    assert np.all(np.isfinite(out_g)), "non-finite output"
    group_exact = np.ones((B, Hkv), bool)
    if check_sets and g["state"] is not None and nb > 0:
        sel_g = g["state"]["sel"].numpy().astype(bool)
        for b in range(B):
            for h in range(Hq):
                want = np.zeros(nb, bool)
                want[r.sel[b][h]] = True
                amb = ambiguous_blocks(r, b, h, tau)
                diff = np.nonzero(sel_g[b, h] != want)[0]
                bad = [int(i) for i in diff if int(i) not in amb]
                assert not bad, f"selected set of (b={b}, h={h}) differs on blocks {bad[:10]}"
                if diff.size:
                    group_exact[b, h // n_rep] = False
                assert cert["k_star"][b, h] == len(r.sel[b][h]) or diff.size, "k_star differs"
        kp0 = g["state"]["kprom0"].numpy().astype(bool)
        for b in range(B):
            for gg in range(Hkv):
                if group_exact[b, gg]:
                    assert np.array_equal(kp0[b, gg], r.kprom0[b, gg]), "union of selections differs"
    stats["set_mismatch_groups"] = int((~group_exact).sum())
    for b in range(B):
        for h in range(Hq):
            stats["heads"] += 1
            gg = h // n_rep
            marg = marginal_head(r, b, h, eps) or not group_exact[b, gg]
            lv_g, lv_o = int(cert["level"][b, h]), int(r.level[b, h])
            if marg:
                stats["excluded"] += 1
            else:
                assert lv_g == lv_o, f"ladder level of (b={b}, h={h}): gpu {lv_g} oracle {lv_o}"
                assert int(cert["rank_ok"][b, h]) == int(r.rank_ok[b, h])
            if lv_g != lv_o:
                continue
            ref = r.out64[b, h]
            err = np.abs(out_g[b, h] - ref)
            stats["out_compared"] += 1
            stats["max_out_err"] = max(stats["max_out_err"], float(err.max()))
            if np.max(np.abs(ref)) <= OUT_STRICT_RANGE:
                stats["max_out_err_unit_range"] = max(stats["max_out_err_unit_range"], float(err.max()))
                assert err.max() <= OUT_ATOL, \
                    f"output of (b={b}, h={h}) off by {err.max():.3e} > {OUT_ATOL} (level {lv_o})"
            assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), \
                f"output of (b={b}, h={h}) off by {err.max():.3e} (level {lv_o})"
            if not marg:
                stats["strict"] += 1
                for name, o_val in (("e_key", r.e_key[b, h]), ("e_val", r.e_val[b, h])):
                    gv = float(cert[name][b, h])
                    d = abs(gv - o_val)
                    assert d <= BOUND_RTOL * abs(o_val) + BOUND_ATOL, \
                        f"{name} of (b={b}, h={h}): gpu {gv} oracle {o_val}"
                    if o_val != 0:
                        stats["max_bound_rel"] = max(stats["max_bound_rel"], d / abs(o_val))
                if group_exact[b, gg]:
                    assert int(cert["promoted_bytes"][b, h]) == int(r.promoted_bytes[b, h])
                    assert int(cert["n_val_promoted"][b, h]) == int(r.n_val_promoted[b, h])
    # per-sequence ladder level where no head of the sequence was excluded
    for b in range(B):
        if all(not marginal_head(r, b, h, eps) and group_exact[b, h // n_rep] for h in range(Hq)):
            assert int(g["level"][b]) == int(r.ladder_level[b])
    assert stats["strict"] >= min_strict * stats["heads"], \
        f"only {stats['strict']} of {stats['heads']} heads compared strictly: {stats}"
    return stats
