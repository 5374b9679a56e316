"""Pins of the oracle against what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a hand-worked
example, a closed form, brute force with exact or high-precision arithmetic, or an
invariant that a dropped term, wrong sign or transposed operand would break.
Page cited: "Runtime-Certified Bounded-Error Quantized Attention" (gist.science
technical summary), Method §1-§3 and Contributions ("deterministic recovery").
"""

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.numpy()


def _case(seed=0, ctx=200, Hq=4, Hkv=1, batch=1, kscale=1.0):
    q, K, V = W.tiny(seed=seed, ctx=ctx, Hq=Hq, Hkv=Hkv, batch=batch, kscale=kscale)
    return _np(q), _np(K), _np(V)


# ---------------------------------------------------------------------------------
# binary16 round-up, pinned by brute force over every fp16 value
# ---------------------------------------------------------------------------------

def test_f16_round_up_brute_force():
    allh = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)   # +0 .. max finite
    allf = allh.astype(np.float32)
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.uniform(0, 70000, 2000), rng.uniform(0, 1e-3, 2000),
        rng.uniform(0, 1e-6, 500), allf[::97], allf[::89] * np.float32(1.0000001)]).astype(np.float32)
    xs = xs[xs <= allf[-1]]
    got = O.f16_round_up(xs).astype(np.float32)
    want = allf[np.searchsorted(allf, xs, side="left")]
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------------
# Method §1 quantisers: hand-worked golden example
# ---------------------------------------------------------------------------------

def _load_golden():
    keys, value = [], None
    with open(os.path.join(GOLDEN, "quant_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, rest = line.split(None, 1)
            parts = [p.split() for p in rest.split("|")]
            if head == "key":
                ch = int(parts[0][0])
                keys.append((ch, [float(x) for x in parts[0][1:]], [int(x) for x in parts[1]],
                             float(parts[2][0])))
            elif head == "value":
                value = ([float(x) for x in parts[0]], [int(x) for x in parts[1]],
                         (float(parts[2][0]), float(parts[2][1])), float(parts[3][0]))
    return keys, value


def test_golden_key_quantisation():
    keys, _ = _load_golden()
    kb = np.zeros((64, 128), np.float16)
    for ch, vals, _, _ in keys:
        kb[: len(vals), ch] = vals
    codes, scales = O.quantize_key_block(kb)
    for ch, vals, want_codes, want_scale in keys:
        assert float(scales[ch]) == want_scale
        assert list(codes[: len(want_codes), ch]) == want_codes
        assert np.all(codes[len(want_codes):, ch] == 0)


def test_golden_value_quantisation():
    _, (vals, codes_w, (s_w, o_w), eta_w) = _load_golden()
    vb = np.zeros((64, 128), np.float16)
    vb[0, :32] = vals[2]
    vb[0, 0] = vals[0]
    vb[0, 1] = vals[1]
    codes, s, o, eta = O.quantize_value_block(vb)
    assert float(s[0, 0]) == s_w and float(o[0, 0]) == o_w
    assert codes[0, 0] == codes_w[0] and codes[0, 1] == codes_w[1]
    assert np.all(codes[0, 2:32] == codes_w[2])
    # every other group is constant zero: s = 0, code 0, exact
    assert np.all(s[1:] == 0) and np.all(s[0, 1:] == 0) and np.all(codes[1:] == 0)
    assert float(eta) == eta_w


# ---------------------------------------------------------------------------------
# Method §1 quantisers: invariants on random and adversarial blocks
# ---------------------------------------------------------------------------------

def test_key_quantiser_invariants():
    rng = np.random.default_rng(2)
    for trial in range(20):
        scale = 10.0 ** rng.uniform(-3, 2)
        kb = (rng.standard_normal((3, 64, 128)) * scale).astype(np.float16)
        kb[0, :, 5] = 0
        codes, s = O.quantize_key_block(kb)
        assert codes.dtype == np.int8 and codes.min() >= -127 and codes.max() <= 127
        k = kb.astype(np.float64)
        s64 = s.astype(np.float64)[:, None, :]
        a = np.abs(k).max(axis=1)
        assert np.all(s.astype(np.float64) >= a / 127)          # rounded up
        khat = O.dequantize_keys(codes, s)
        assert np.all(np.abs(k - khat) <= s64 * (0.5 + 2.0 ** -17))
        assert np.all(s[0, 5] == 0) and np.all(codes[0, :, 5] == 0)
        # the fp32 product s*code is exact
        assert np.array_equal(khat, (s.astype(np.float32)[:, None, :] * codes.astype(np.float32)).astype(np.float64))


def test_key_grid_roundtrip():
    rng = np.random.default_rng(3)
    s = np.float16(2.0 ** -6)
    codes = rng.integers(-126, 127, (64, 128)).astype(np.int8)
    codes[0, :] = 127                               # pin the max so the scale is exactly s
    kb = (codes.astype(np.float64) * float(s)).astype(np.float16)
    c2, s2 = O.quantize_key_block(kb)
    assert np.all(s2 == s) and np.array_equal(c2, codes)


def test_value_quantiser_invariants():
    rng = np.random.default_rng(4)
    for trial in range(20):
        scale = 10.0 ** rng.uniform(-2, 2)
        vb = (rng.standard_normal((2, 64, 128)) * scale + rng.uniform(-5, 5)).astype(np.float16)
        codes, s, o, eta = O.quantize_value_block(vb)
        assert codes.max() <= 15
        v = vb.astype(np.float64).reshape(2, 64, 4, 32)
        mn = v.min(axis=-1)
        assert np.array_equal(o.astype(np.float64), mn)               # offset = group min, exact
        c = codes.reshape(2, 64, 4, 32)
        assert np.all(c[v == mn[..., None]] == 0)                     # the min encodes as 0
        vhat = O.dequantize_values(codes, s, o).reshape(2, 64, 4, 32)
        err = np.abs(v - vhat)
        assert np.all(err <= s.astype(np.float64)[..., None] * 0.5 * (1 + 2.0 ** -10) + 1e-7 * np.abs(v).max())
        # eta is the fp32 max error, recomputed exactly with rationals on a sample
        for bi in range(2):
            e_exact = max(abs(Fraction(float(x)) - Fraction(float(np.float32(y))))
                          for x, y in zip(vb[bi].astype(np.float32).ravel()[::7],
                                          vhat[bi].ravel()[::7]))
            assert float(eta[bi]) >= float(np.float32(float(e_exact))) * (1 - 2 ** -23)
        e32 = np.abs(vb.astype(np.float32) - vhat.reshape(2, 64, 128).astype(np.float32)).reshape(2, -1).max(1)
        assert np.array_equal(eta, e32)


# ---------------------------------------------------------------------------------
# A1 dense attention: high-precision brute force and closed forms
# ---------------------------------------------------------------------------------

def _mp_attention(q, K, V):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    D = len(q)
    s = [mpmath.fsum(mpmath.mpf(float(q[c])) * mpmath.mpf(float(K[t, c])) for c in range(D)) / mpmath.sqrt(D)
         for t in range(K.shape[0])]
    m = max(s)
    e = [mpmath.exp(x - m) for x in s]
    z = mpmath.fsum(e)
    return np.array([float(mpmath.fsum(e[t] * mpmath.mpf(float(V[t, c])) for t in range(len(e))) / z)
                     for c in range(V.shape[1])])


def test_dense_attention_brute_force():
    rng = np.random.default_rng(5)
    for n in (1, 3, 7):
        q = rng.standard_normal(8).astype(np.float16)
        K = (rng.standard_normal((n, 8)) * 3).astype(np.float16)
        V = rng.standard_normal((n, 8)).astype(np.float16)
        assert np.allclose(O.dense_attention(q, K, V), _mp_attention(q, K, V), rtol=0, atol=1e-13)


def test_dense_attention_closed_forms():
    rng = np.random.default_rng(6)
    q = rng.standard_normal(128).astype(np.float16)
    V = rng.standard_normal((50, 128)).astype(np.float16)
    K = np.tile(rng.standard_normal(128).astype(np.float16), (50, 1))
    assert np.allclose(O.dense_attention(q, K, V), V.astype(np.float64).mean(0), atol=1e-14)
    K2 = np.zeros((50, 128), np.float16)
    K2[17] = (np.sign(q.astype(np.float32)) * 60).astype(np.float16)   # one key dominates
    assert np.allclose(O.dense_attention(q, K2, V), V[17].astype(np.float64), atol=1e-12)


# ---------------------------------------------------------------------------------
# Contributions "deterministic recovery": tau_cov = 1 returns exact dense output
# ---------------------------------------------------------------------------------

def test_tau_one_is_dense():
    q, K, V = _case(seed=7, ctx=300, Hq=8, Hkv=2)
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 1.0, 0.25, O.OracleConfig(n_rep=4))
    assert np.all(r.level == 4) and np.all(r.e_key == 0) and np.all(r.e_val == 0)
    for h in range(8):
        dense = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
        assert np.array_equal(r.out[0, h], dense.astype(np.float16))


# ---------------------------------------------------------------------------------
# A5/A7 soundness: measured error <= E_key + E_val on random and adversarial heads
# ---------------------------------------------------------------------------------

def _group_inputs(q, K, V, t1, g=0, b=0):
    D = q.shape[-1]
    nb = K.shape[2] // 64
    v_hat = O.dequantize_values(t1.vc[b, g], t1.vs[b, g], t1.vo[b, g])
    R = float(np.max(t1.vmax[b, g].astype(np.float64) - t1.vmin[b, g].astype(np.float64)))
    return nb, v_hat, R


def _check_sound(q, K, V, rng, n_masks=3):
    t1 = O.quantize_layer(K, V)
    nb, v_hat, R = _group_inputs(q, K, V, t1)
    worst = 0.0
    for h in range(q.shape[1]):
        qh = q[0, h]
        s_ex = K[0, 0].astype(np.float64) @ qh.astype(np.float64) / math.sqrt(q.shape[-1])
        s_hat = O.int8_scores(qh, t1.kc[0, 0], t1.ks[0, 0])
        delta = O.score_perturbation(qh, t1.ks[0, 0])
        # |s - s_hat| <= Delta for every INT8 token (A5)
        assert np.all(np.abs(s_ex[: nb * 64].reshape(nb, 64) - s_hat) <= delta[:, None])
        dense = O.dense_attention(qh, K[0, 0], V[0, 0])
        for _ in range(n_masks):
            kp = rng.random(nb) < rng.random()
            vp = rng.random(nb) < rng.random()
            r = O.mixed_attention(s_ex, s_hat, V[0, 0], v_hat, delta, t1.eta[0, 0], R, kp, vp)
            err = np.max(np.abs(r.out - dense))
            assert err <= r.e_key + r.e_val + 1e-9, (err, r.e_key, r.e_val)
            if r.e_key + r.e_val > 0:
                worst = max(worst, err / (r.e_key + r.e_val))
            if kp.all():
                assert r.e_key == 0
            if vp.all():
                assert r.e_val == 0
    return worst


def test_soundness_random_heads():
    rng = np.random.default_rng(8)
    n_heads = 0
    for seed in range(40):
        ctx = int(rng.integers(64, 700))
        ks = float(rng.choice([0.5, 1.0, 3.0, 8.0]))
        q, K, V = _case(seed=100 + seed, ctx=ctx, Hq=64, Hkv=1, kscale=ks)
        q = q.astype(np.float32)
        q *= rng.uniform(0.2, 3.0, size=(1, 64, 1)).astype(np.float32)
        _check_sound(q.astype(np.float16), K, V, rng, n_masks=4)
        n_heads += 64
    assert n_heads >= 2500
    # 2560 heads x 4 promotion masks = 10240 certified (head, mask) cases


def _adversarial_keys(q, nb, rng, s0=2.0 ** -5):
    """Keys just below a half step, signed so INT8 rounding lowers q.k (as in the c4 needle)."""
    D = q.shape[-1]
    sg = np.sign(q.astype(np.float64)); sg[sg == 0] = 1
    K = np.zeros((nb * 64, D))
    for b in range(nb):
        rows = np.clip(rng.standard_normal((64, D)), -3.9, 3.9)
        n = rng.integers(0, 120, size=(64, 1))
        adv = sg * (n + 7.0 / 16.0) * s0
        mask = rng.random((64, 1)) < 0.7
        rows = np.where(mask, adv, rows)
        rows[0] = -sg * 127 * s0            # anchor: channel scales are exactly s0
        K[b * 64:(b + 1) * 64] = rows
    return K.astype(np.float16)


def test_soundness_adversarial_heads():
    rng = np.random.default_rng(9)
    worst = 0.0
    for trial in range(12):
        nb = int(rng.integers(1, 6))
        q = rng.standard_normal((1, 4, 128)).astype(np.float16)
        q[0, 1:] = q[0, 0]
        K = _adversarial_keys(q[0, 0], nb, rng)[None, None]
        V = rng.standard_normal((1, 1, nb * 64, 128)).astype(np.float16)
        worst = max(worst, _check_sound(q, K, V, rng, n_masks=3))
        # the bound is not vacuous on these heads: the key error reaches a good part of Delta
        t1 = O.quantize_layer(K, V)
        qh = q[0, 0]
        s_ex = K[0, 0].astype(np.float64) @ qh.astype(np.float64) / math.sqrt(128)
        s_hat = O.int8_scores(qh, t1.kc[0, 0], t1.ks[0, 0])
        delta = O.score_perturbation(qh, t1.ks[0, 0])
        ratio = np.max((s_ex[: nb * 64].reshape(nb, 64) - s_hat) / delta[:, None])
        assert ratio > 0.8
    assert worst > 0


# ---------------------------------------------------------------------------------
# Total-variation lemma behind E_key, closed form on two tokens
# ---------------------------------------------------------------------------------

def test_tv_lemma_brute_force():
    """One INT8 block (64 equal scores s1) plus one exact partial-block token (s0).

    The true scores are s1 + delta_t with |delta_t| <= Delta.  Brute force over the
    split of the 64 tokens into two groups shifted by d1 and d2 (grids over
    [-Delta, Delta]) gives the worst total variation; it must not exceed the oracle's
    E_key / R = S / A, and for small Delta must reach at least a third of it (not vacuous).
    """
    for s0, s1, Dl in [(0.0, 0.0, 0.1), (2.0, -1.0, 0.3), (-3.0, 1.0, 0.05), (0.0, 5.0, 1.0)]:
        w0, w1 = math.exp(s0), math.exp(s1)
        Z = w0 + 64 * w1
        grid = np.linspace(-Dl, Dl, 41)
        worst = 0.0
        for k in range(0, 65, 4):
            for d1 in grid:
                for d2 in grid:
                    wa, wb = k * w1 * math.exp(d1), (64 - k) * w1 * math.exp(d2)
                    z = w0 + wa + wb
                    tv = 0.5 * (abs(w0 / z - w0 / Z) + abs(wa / z - k * w1 / Z) + abs(wb / z - (64 - k) * w1 / Z))
                    worst = max(worst, tv)
        s_exact = np.full(65, s1); s_exact[64] = s0
        s_hat = np.full((1, 64), s1)
        V = np.zeros((65, 128), np.float16); V[:64, 0] = 1.0          # value range R = 1
        v_hat = V[:64].astype(np.float64)[None]
        r = O.mixed_attention(s_exact, s_hat, V, v_hat, np.array([Dl]), np.zeros(1, np.float32), 1.0,
                              np.array([False]), np.array([False]))
        p1 = 64 * w1 / Z
        assert abs(r.S - p1 * math.expm1(Dl)) < 1e-15
        assert abs(r.A - ((1 - p1) + p1 * math.exp(-Dl))) < 1e-15
        # closed form of the certificate for this head: R = 1, one INT8 block of mass p1
        e_cf = p1 * math.expm1(Dl) / ((1 - p1) + p1 * math.exp(-Dl))
        assert abs(r.e_key - e_cf) <= 1e-14 * e_cf
        assert worst <= r.e_key + 1e-15
        if Dl <= 0.3:                 # first-order tight for small perturbations
            assert worst >= r.e_key / 3


def test_e_key_monotone_in_promotion():
    """Promoting more key blocks never raises S/A (the point of rung 1)."""
    rng = np.random.default_rng(10)
    q, K, V = _case(seed=11, ctx=64 * 12, Hq=4, Hkv=1, kscale=4.0)
    t1 = O.quantize_layer(K, V)
    nb, v_hat, R = _group_inputs(q, K, V, t1)
    qh = q[0, 2]
    s_ex = K[0, 0].astype(np.float64) @ qh.astype(np.float64) / math.sqrt(128)
    s_hat = O.int8_scores(qh, t1.kc[0, 0], t1.ks[0, 0])
    delta = O.score_perturbation(qh, t1.ks[0, 0])
    order = rng.permutation(nb)
    kp = np.zeros(nb, bool)
    prev = math.inf
    for b in order:
        r = O.mixed_attention(s_ex, s_hat, V[0, 0], v_hat, delta, t1.eta[0, 0], R, kp, np.zeros(nb, bool))
        assert r.S / r.A <= prev * (1 + 1e-12)
        prev = r.S / r.A
        kp[b] = True


# ---------------------------------------------------------------------------------
# A6 selection: brute force over subsets
# ---------------------------------------------------------------------------------

def test_selection_brute_force():
    rng = np.random.default_rng(12)
    for trial in range(300):
        nb = int(rng.integers(1, 11))
        lse8 = rng.standard_normal(nb) * rng.uniform(0.1, 4)
        if rng.random() < 0.3:
            lse8[rng.integers(0, nb)] = lse8[0]                     # exact ties
        tail = rng.standard_normal() if rng.random() < 0.5 else -math.inf
        tau = float(rng.choice([0.5, 0.9, 0.99, 0.995, rng.random()]))
        chosen, mass, tail_mass, cum = O.select_top_k_star(lse8, tail, tau)
        assert abs(mass.sum() + tail_mass - 1) < 1e-12
        best_k = None
        for k in range(nb + 1):
            covers = [c for c in itertools.combinations(range(nb), k)
                      if tail_mass + sum(mass[list(c)]) >= tau]
            if covers:
                best_k = k
                best_mass = max(sum(mass[list(c)]) for c in covers)
                break
        if best_k is None:          # tau above the total due to rounding: take every block
            assert len(chosen) == nb
            continue
        assert len(chosen) == best_k
        assert abs(sum(mass[chosen]) - best_mass) < 1e-12
        if chosen:                   # order: descending mass, ties to the lower index
            keys = [(-mass[b], b) for b in chosen]
            assert keys == sorted(keys)
            assert all(mass[b] <= mass[chosen[-1]] or b in chosen for b in range(nb))


# ---------------------------------------------------------------------------------
# A8 ladder special cases
# ---------------------------------------------------------------------------------

def test_eps_infinite_and_zero():
    q, K, V = _case(seed=13, ctx=64 * 9 + 17, Hq=8, Hkv=2, kscale=3.0)
    t1 = O.quantize_layer(K, V)
    cfg = O.OracleConfig(n_rep=4)
    r = O.decode_layer(q, K, V, t1, 0.9, math.inf, cfg)
    for h in range(8):
        assert r.level[0, h] == (0 if r.rank_ok[0, h] else 3) or r.level[0, h] == 4
    r0 = O.decode_layer(q, K, V, t1, 0.9, 0.0, cfg)
    for h in range(8):
        assert r0.level[0, h] >= 3 or (r0.e_key[0, h] == 0 and r0.e_val[0, h] == 0)


def test_ladder_output_within_certificate():
    """Every returned head is within its certificate of exact attention (or exactly dense)."""
    for seed, ks, eps in [(14, 1.0, 0.25), (15, 4.0, 0.1), (16, 8.0, 0.05), (17, 2.0, 0.02)]:
        q, K, V = _case(seed=seed, ctx=64 * 10 + 5, Hq=8, Hkv=2, kscale=ks)
        V[0, 1, 64:128] *= 8
        t1 = O.quantize_layer(K, V)
        r = O.decode_layer(q, K, V, t1, 0.9, eps, O.OracleConfig(n_rep=4))
        for h in range(8):
            dense = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
            err = np.max(np.abs(r.out64[0, h] - dense))
            if r.level[0, h] >= 3:
                assert err == 0
            else:
                assert r.e_key[0, h] + r.e_val[0, h] <= eps
                assert err <= r.e_key[0, h] + r.e_val[0, h] + 1e-9


def test_ladder_rungs_fire():
    """Large value ranges force rung 2; a tight eps with peaked keys forces rung 1."""
    q, K, V = _case(seed=18, ctx=64 * 16, Hq=4, Hkv=1, kscale=6.0)
    V = V.astype(np.float32)
    V[0, 0, :, :32] *= 8
    V = V.astype(np.float16)
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 0.8, 0.25, O.OracleConfig(n_rep=4))
    assert np.any(r.planned[0] == 2)
    assert np.all(r.vprom1[0, 0] >= r.kprom0[0, 0] * 0)      # shapes line up
    r1 = O.decode_layer(q, K, V, t1, 0.5, 0.3, O.OracleConfig(n_rep=4))
    assert np.any(r1.planned[0] >= 1)


def test_l4_when_half_the_heads_fail():
    q, K, V, info = W.c4(batch=1, ctx=4096, Hq=8, Hkv=2)
    q, K, V = _np(q), _np(K), _np(V)
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 0.995, 0.25, O.OracleConfig(n_rep=4))
    assert np.all(r.rank_ok == 0), r.rank_ok          # every planted head fails the check
    assert np.all(r.level == 4)
    assert np.all(r.ladder_level == 4)
    for h in range(8):
        dense = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
        assert np.array_equal(r.out[0, h], dense.astype(np.float16))


def test_c4_planted_flips_ranking():
    """The c4 construction: FP16 ranks the planted block first, INT8 the decoy."""
    q, K, V, info = W.c4(batch=2, ctx=8192, Hq=8, Hkv=2)
    q, K, V = _np(q), _np(K), _np(V)
    t1 = O.quantize_layer(K, V)
    for (b, g, pb, db) in info:
        qh = q[b, g * 4]
        s_ex = K[b, g].astype(np.float64) @ qh.astype(np.float64) / math.sqrt(128)
        nb = K.shape[2] // 64
        lse16 = O.block_logsumexp(s_ex[: nb * 64].reshape(nb, 64))
        lse8 = O.block_logsumexp(O.int8_scores(qh, t1.kc[b, g], t1.ks[b, g]))
        assert int(np.argmax(lse16)) == pb and int(np.argmax(lse8)) == db
        assert 0.02 < lse16[pb] - lse16[db] < 0.08
        assert np.all(t1.ks[b, g, pb] == np.float16(1 / 32))


# ---------------------------------------------------------------------------------
# P7 / P8
# ---------------------------------------------------------------------------------

def test_gqa_equals_mha_with_repeated_kv_when_dense():
    q, K, V = _case(seed=19, ctx=64 * 3 + 9, Hq=8, Hkv=2)
    t1 = O.quantize_layer(K, V)
    rg = O.decode_layer(q, K, V, t1, 1.0, 0.25, O.OracleConfig(n_rep=4))
    Km = np.repeat(K, 4, axis=1); Vm = np.repeat(V, 4, axis=1)
    rm = O.decode_layer(q, Km, Vm, O.quantize_layer(Km, Vm), 1.0, 0.25, O.OracleConfig(n_rep=1))
    assert np.array_equal(rg.out, rm.out)


def test_identical_heads_identical_results():
    q, K, V = _case(seed=20, ctx=64 * 7 + 3, Hq=4, Hkv=1, kscale=3.0)
    q[0, 1:] = q[0, 0]
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 0.95, 0.2, O.OracleConfig(n_rep=4))
    for h in range(1, 4):
        assert np.array_equal(r.out[0, h], r.out[0, 0])
        assert r.level[0, h] == r.level[0, 0] and r.e_key[0, h] == r.e_key[0, 0]


def test_single_block_fully_promoted_is_exact():
    q, K, V = _case(seed=21, ctx=64, Hq=4, Hkv=1)
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 0.9999999, math.inf, O.OracleConfig(n_rep=4))
    for h in range(4):
        assert r.k_star[0, h] == 1 and r.e_key[0, h] == 0
        dense = O.dense_attention(q[0, h], K[0, 0], V[0, 0])
        # keys exact; values INT4 -> error within E_val, and E_val > 0
        assert np.max(np.abs(r.out64[0, h] - dense)) <= r.e_val[0, h] + 1e-12


def test_partial_block_only_is_exact():
    q, K, V = _case(seed=22, ctx=37, Hq=4, Hkv=1)
    t1 = O.quantize_layer(K, V)
    r = O.decode_layer(q, K, V, t1, 0.995, 0.0, O.OracleConfig(n_rep=4))
    for h in range(4):
        assert r.level[0, h] == 0 and r.e_key[0, h] == 0 and r.e_val[0, h] == 0
        dense = O.dense_attention(q[0, h], K[0, 0], V[0, 0])
        assert np.allclose(r.out64[0, h], dense, atol=1e-14)


def test_c2_mass_concentrated():
    q, K, V = W.c2(batch=1, ctx=4096, Hq=8, Hkv=2)
    q, K = _np(q).astype(np.float64), _np(K).astype(np.float64)
    gen = torch.Generator().manual_seed(1)
    fr = []
    for h in range(8):
        s = K[0, h // 4] @ q[0, h] / math.sqrt(128)
        p = np.exp(s - s.max()); p /= p.sum()
        blk = p.reshape(-1, 64).sum(1)
        top = np.sort(blk)[::-1]
        fr.append(top[: max(1, int(round(0.05 * len(blk))))].sum())
    del gen
    assert min(fr) >= 0.99, fr


# ---------------------------------------------------------------------------------
# uncertified INT8/INT4 baseline (Experiments: the plain quantized comparison)
# ---------------------------------------------------------------------------------

def test_uncertified_is_softmax_attention_over_reconstructions():
    """Brute force: textbook softmax attention over the explicitly reconstructed cache
    (s * code keys, s * code + o values on full blocks, FP16 on the partial block)."""
    for seed, ctx, Hq, Hkv in ((0, 200, 4, 1), (5, 321, 8, 2), (9, 64, 4, 1), (11, 40, 4, 1)):
        q, K, V = _case(seed=seed, ctx=ctx, Hq=Hq, Hkv=Hkv, kscale=2.0)
        t1 = O.quantize_layer(K, V)
        res = O.uncertified_decode_layer(q, K, V, t1)
        nb = ctx // 64
        for g in range(Hkv):
            Kr = K[0, g].astype(np.float64).copy()
            Vr = V[0, g].astype(np.float64).copy()
            for b in range(nb):
                Kr[64 * b:64 * b + 64] = O.dequantize_keys(t1.kc[0, g, b], t1.ks[0, g, b])
                Vr[64 * b:64 * b + 64] = O.dequantize_values(t1.vc[0, g, b], t1.vs[0, g, b],
                                                             t1.vo[0, g, b])
            for h in range(g * (Hq // Hkv), (g + 1) * (Hq // Hkv)):
                qh = q[0, h].astype(np.float64)
                s = Kr @ qh / math.sqrt(128)
                p = np.exp(s - s.max()); p /= p.sum()
                np.testing.assert_allclose(res.out64[0, h], p @ Vr, rtol=1e-11, atol=1e-12)


def test_uncertified_grid_aligned_cache_is_exact():
    """Keys on their INT8 grid and values on their INT4 grid reconstruct exactly, so the
    uncertified output equals dense attention and E_val = 0."""
    rng = np.random.default_rng(21)
    nb, D = 3, 128
    s0 = 2.0 ** -4
    codes = rng.integers(-126, 127, (nb * 64, D))
    codes[::64] = 127                                  # every block's scale is exactly s0
    K = (codes * s0).astype(np.float16)[None, None]
    vcode = rng.integers(0, 16, (nb * 64, D))
    vcode[:, ::32] = 0
    vcode[:, 1::32] = 15                               # each group spans 0..15 steps
    V = (vcode * 2.0 ** -3 - 1.0).astype(np.float16)[None, None]
    q = rng.standard_normal((1, 4, D)).astype(np.float16)
    t1 = O.quantize_layer(K, V)
    res = O.uncertified_decode_layer(q, K, V, t1)
    for h in range(4):
        ref = O.dense_attention(q[0, h], K[0, 0], V[0, 0])
        np.testing.assert_allclose(res.out64[0, h], ref, rtol=1e-12, atol=1e-13)
    assert np.all(res.e_val == 0.0)


def test_uncertified_bound_is_sound():
    """The reported (unenforced) bound still covers the uncertified output's error."""
    rng = np.random.default_rng(13)
    for seed in range(6):
        q, K, V = _case(seed=300 + seed, ctx=int(rng.integers(64, 600)), Hq=16, Hkv=1,
                        kscale=float(rng.choice([1.0, 4.0])))
        t1 = O.quantize_layer(K, V)
        res = O.uncertified_decode_layer(q, K, V, t1)
        for h in range(16):
            ref = O.dense_attention(q[0, h], K[0, 0], V[0, 0])
            err = np.max(np.abs(res.out64[0, h] - ref))
            assert err <= res.e_key[0, h] + res.e_val[0, h] + 1e-9


# ---------------------------------------------------------------------------------
# FP16-values configuration (Results: the ablation that replaces INT4 values by FP16)
# ---------------------------------------------------------------------------------

def _grid_keys(rng, n, D=128, s0=2.0 ** -5):
    codes = rng.integers(-126, 127, (n, D))
    codes[::64] = 127                                  # every block's scales are exactly s0
    return (codes * s0).astype(np.float16)


def test_fp16_values_on_grid_keys_equal_dense():
    """Keys on their INT8 grid reconstruct exactly and the values are the FP16 originals,
    so every certified head returns dense attention (the INT4 path would not: the values
    here are off the INT4 grid) and E_val = 0."""
    rng = np.random.default_rng(31)
    for ctx in (64 * 5, 64 * 7 + 19):
        K = _grid_keys(rng, ctx)[None, None]
        V = rng.standard_normal((1, 1, ctx, 128)).astype(np.float16)
        q = (rng.standard_normal((1, 4, 128)) * 0.3).astype(np.float16)
        t1 = O.quantize_layer(K, V)
        cfg = O.OracleConfig(n_rep=4, value_fp16=True)
        r = O.decode_layer(q, K, V, t1, 0.9, float("inf"), cfg)
        u = O.uncertified_decode_layer(q, K, V, t1, cfg)
        assert np.all(r.e_val == 0.0) and np.all(u.e_val == 0.0)
        assert np.all(r.level == 0) and np.all(r.n_val_promoted == 0)
        for h in range(4):
            ref = O.dense_attention(q[0, h], K[0, 0], V[0, 0])
            np.testing.assert_allclose(r.out64[0, h], ref, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(u.out64[0, h], ref, rtol=1e-12, atol=1e-13)
        # the INT4 configuration differs on the same inputs
        r4 = O.decode_layer(q, K, V, t1, 0.9, float("inf"), O.OracleConfig(n_rep=4))
        assert np.max(np.abs(r4.out64 - r.out64)) > 1e-4


def test_fp16_values_bound_sound_and_no_value_pages():
    rng = np.random.default_rng(32)
    for seed in range(5):
        q, K, V = _case(seed=400 + seed, ctx=int(rng.integers(64, 900)), Hq=8, Hkv=2, kscale=4.0)
        t1 = O.quantize_layer(K, V)
        cfg = O.OracleConfig(n_rep=4, value_fp16=True)
        r = O.decode_layer(q, K, V, t1, 0.9, 0.05, cfg)
        nb = K.shape[2] // 64
        assert np.all(r.e_val == 0.0) and np.all(r.n_val_promoted == 0)
        assert np.all(r.vprom1 == (nb > 0))            # every block counts as FP16-valued
        for h in range(8):
            ref = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
            err = np.max(np.abs(r.out64[0, h] - ref))
            assert err <= r.e_key[0, h] + 1e-9
            if r.level[0, h] >= 3:
                assert err <= 1e-12
        for g in range(2):
            heads = range(4 * g, 4 * g + 4)
            k_blocks = int(r.kprom1[0, g].sum())
            dense = any(r.level[0, h] >= 3 for h in heads)
            want = (nb if dense else k_blocks) * 64 * 128 * 2   # dense: the other keys
            assert int(r.promoted_bytes[0, 4 * g]) == want


# ---------------------------------------------------------------------------------
# value tolerance v_tol (Results: tightening it closes the value-sensitive gap)
# ---------------------------------------------------------------------------------

def test_v_tol_budget_holds_and_tightening_pages_in_more_values():
    q, K, V = W.c5_point(64 * 40 + 7, 1, Hq=8, Hkv=2)
    q, K, V = q.numpy(), K.numpy(), V.numpy()
    t1 = O.quantize_layer(K, V)
    prev_v, prev_bytes = -1, -1
    for v_tol in (math.inf, 0.2, 0.1, 0.05, 0.02):
        cfg = O.OracleConfig(n_rep=4, v_tol=v_tol)
        r = O.decode_layer(q, K, V, t1, 0.99, 0.5, cfg)
        ok = r.level < 3
        assert np.all(r.e_val[ok] <= v_tol) and np.all(r.e_key[ok] + r.e_val[ok] <= 0.5)
        nv = int(r.vprom1.sum())
        assert nv >= prev_v                         # a tighter budget never pages in less
        assert int(r.promoted_bytes.sum()) >= prev_bytes
        prev_v, prev_bytes = nv, int(r.promoted_bytes.sum())
        for h in np.nonzero(ok[0])[0]:
            ref = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
            assert np.max(np.abs(r.out64[0, h] - ref)) <= r.e_key[0, h] + r.e_val[0, h] + 1e-9
    assert prev_v > 0
    # an infinite v_tol is the plain eps rule
    a = O.decode_layer(q, K, V, t1, 0.99, 0.5, O.OracleConfig(n_rep=4))
    b = O.decode_layer(q, K, V, t1, 0.99, 0.5, O.OracleConfig(n_rep=4, v_tol=math.inf))
    assert np.array_equal(a.level, b.level) and np.array_equal(a.out64, b.out64)



# ---------------------------------------------------------------------------------
# A4 value ranges: every cached token counts, the partial FP16 block included
# ---------------------------------------------------------------------------------

def test_value_range_includes_partial_block():
    """Method §2 computes E_key from the range of the exact values; the range is taken
    over every cached token, so an extreme value in the partial (not yet quantised)
    block sets it, and E_key scales with it."""
    rng = np.random.default_rng(41)
    ctx = 64 * 3 + 10
    V = rng.standard_normal((1, 1, ctx, 128)).astype(np.float16)
    V[0, 0, 64 * 3 + 4, 7] = 50.0          # in the partial block
    V[0, 0, 64 * 3 + 9, 9] = -40.0
    K = rng.standard_normal((1, 1, ctx, 128)).astype(np.float16)
    t1 = O.quantize_layer(K, V)
    full = V[0, 0].astype(np.float32)
    assert np.array_equal(t1.vmax[0, 0], full.max(axis=0)) and np.array_equal(t1.vmin[0, 0], full.min(axis=0))
    assert t1.vmax[0, 0, 7] == 50.0 and t1.vmin[0, 0, 9] == -40.0
    # a single token: the range is zero and so is E_key, whatever the key error
    t_one = O.quantize_layer(K[:, :, :1], V[:, :, :1])
    assert np.all(t_one.vmax == t_one.vmin)
    # E_key is linear in R: the same head with the outliers removed from the partial block
    V2 = V.copy()
    V2[0, 0, 64 * 3 + 4, 7] = 0.0
    V2[0, 0, 64 * 3 + 9, 9] = 0.0
    q = rng.standard_normal((1, 1, 128)).astype(np.float16)   # one head: one selection
    r1 = O.decode_layer(q, K, V, t1, 0.3, math.inf, O.OracleConfig(n_rep=1))
    t2 = O.quantize_layer(K, V2)
    r2 = O.decode_layer(q, K, V2, t2, 0.3, math.inf, O.OracleConfig(n_rep=1))
    R1 = float(np.max(t1.vmax[0, 0].astype(np.float64) - t1.vmin[0, 0]))
    R2 = float(np.max(t2.vmax[0, 0].astype(np.float64) - t2.vmin[0, 0]))
    assert R1 >= 50.0 and R2 < 15.0
    assert not r1.kprom0.all()              # INT8 blocks remain: E_key > 0
    assert r2.e_key0[0, 0] > 0                # (round-0 bounds, before any rung)
    assert abs(r1.e_key0[0, 0] / r2.e_key0[0, 0] - R1 / R2) <= 1e-12 * R1 / R2
