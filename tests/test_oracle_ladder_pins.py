"""Pins of the oracle's fallback-ladder planner (CPU only).

"Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary),
Method §3: the four-rung ladder -- rung 1 widens the set of blocks scored with FP16
keys, rung 2 pages in FP16 values, rung 3 recomputes one head densely, rung 4 the whole
layer -- behind the ranking-consistency check.  The oracle's reading (its
``plan_ladder``, ``ranking_consistent`` and the rung-4 rule of ``decode_layer``):

  * rung 1 when E_key > eps/2: the fewest INT8 blocks whose removal brings the
    projected E_key = (S - removed) / A * R to eps/2 or below, taken in descending
    contribution mass_b (e^Delta_b - 1), ties to the lower block index;
  * rung 2 when the projected E_key + E_val > eps (or E_val > v_tol): the fewest
    INT4-value blocks whose removal brings the projected E_val to
    min(eps - projected E_key, v_tol), in descending mass_b * eta_b;
  * the ranking check compares the first R positions of the selected blocks ordered
    by INT8 and by FP16 block log-mass;
  * rung 4 when at least l4_head_fraction * Hq heads of a sequence are at rung 3.

These tests check the planner against brute force rather than against itself: every
subset of the candidate blocks is enumerated (at most ten blocks), its projected bound
is summed token by token from the mixed softmax, and the planner's answer must be a
smallest subset that meets the target and the prefix of the descending order.  The
ranking check and the rung-4 count are pinned on hand-built orders and on a planted
construction with a known number of failing heads.
"""

import itertools
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

BLK = 64
REL_GUARD = 1e-9     # skip draws whose deciding sums lie this close to a threshold


def _random_head(rng, nb, n_tail):
    """Synthetic inputs of mixed_attention for one head with nb full blocks."""
    N = nb * BLK + n_tail
    D = 8
    s_exact = rng.standard_normal(N) * rng.uniform(0.5, 3.0)
    # per-block perturbation bounds with a wide spread, INT8 scores within them
    delta = rng.uniform(0.0, 1.0, nb) ** 2 * rng.uniform(0.05, 2.0)
    delta[rng.random(nb) < 0.15] = 0.0                      # some blocks exact already
    noise = rng.uniform(-1, 1, (nb, BLK)) * delta[:, None]
    s_hat = s_exact[: nb * BLK].reshape(nb, BLK) + noise
    V = rng.standard_normal((N, D)).astype(np.float16)
    v_hat = V[: nb * BLK].astype(np.float64).reshape(nb, BLK, D) + rng.uniform(-0.05, 0.05, (nb, BLK, D))
    eta = (rng.uniform(0.0, 1.0, nb) ** 2 * rng.uniform(0.01, 1.0)).astype(np.float32)
    eta[rng.random(nb) < 0.15] = 0.0
    R = float(rng.uniform(1.0, 10.0))
    kprom = rng.random(nb) < rng.uniform(0.0, 0.5)
    vprom = rng.random(nb) < rng.uniform(0.0, 0.4)
    return s_exact, s_hat, V, v_hat, delta, eta, R, kprom, vprom


def _token_terms(s_exact, s_hat, delta, eta, kprom):
    """Token-level pieces of the certificate, from the definitions: the mixed softmax
    p_hat over s' (FP16 score on FP16-key blocks and the partial block, INT8 score
    elsewhere), and per block the summed key term p_t (e^Delta_t - 1), the summed
    e^-Delta_t term and the summed value term p_t eta_b."""
    nb = s_hat.shape[0]
    N = s_exact.shape[0]
    s = np.array(s_exact, dtype=np.float64)
    d_t = np.zeros(N)
    for b in range(nb):
        if not kprom[b]:
            s[b * BLK:(b + 1) * BLK] = s_hat[b]
            d_t[b * BLK:(b + 1) * BLK] = delta[b]
    w = np.array([math.exp(x - s.max()) for x in s])
    p = w / math.fsum(w)
    key = [math.fsum(p[t] * math.expm1(d_t[t]) for t in range(b * BLK, (b + 1) * BLK)) for b in range(nb)]
    a_all = math.fsum(p[t] * math.exp(-d_t[t]) for t in range(N))
    val = [math.fsum(p[t] * float(eta[b]) for t in range(b * BLK, (b + 1) * BLK)) for b in range(nb)]
    return np.array(key), a_all, np.array(val)


def _smallest_cover(cands, contrib, total, target):
    """Brute force: the least k such that some k-subset X of cands has
    total - sum_X contrib <= target; returns (k, best sums for every k)."""
    best = []
    k_min = None
    for k in range(len(cands) + 1):
        m = max((math.fsum(contrib[list(X)]) for X in itertools.combinations(cands, k)), default=0.0)
        best.append(m)
        if k_min is None and total - m <= target:
            k_min = k
    return k_min, best


def _is_descending_prefix(chosen, cands, contrib):
    order = sorted(cands, key=lambda b: (-contrib[b], b))
    return list(chosen) == order[: len(chosen)]


def test_plan_ladder_brute_force():
    """Rungs 1 and 2: smallest covering subsets, descending prefixes, branch rules."""
    rng = np.random.default_rng(2024)
    seen = dict(level0=0, rung1=0, rung2=0, rung2_after_1=0, vtol=0)
    checked = 0
    for trial in range(900):
        nb = int(rng.integers(1, 11))
        n_tail = int(rng.choice([0, 0, 5, 40]))
        s_exact, s_hat, V, v_hat, delta, eta, R, kprom, vprom = _random_head(rng, nb, n_tail)
        res = O.mixed_attention(s_exact, s_hat, V, v_hat, delta, eta, R, kprom, vprom)
        key, a_all, val = _token_terms(s_exact, s_hat, delta, eta, kprom)
        S = math.fsum(key)
        E_key = S / a_all * R
        E_val = math.fsum(val[b] for b in range(nb) if not vprom[b])
        # the oracle's certificate is the same quantity (checked elsewhere); here it fixes
        # the thresholds, so eps is drawn around the bound to reach every branch
        assert abs(res.e_key - E_key) <= 1e-9 * max(1.0, E_key)
        assert abs(res.e_val - E_val) <= 1e-9 * max(1.0, E_val)
        tot = E_key + E_val
        eps = float(rng.choice([0.3, 0.7, 1.0, 1.5, 3.0])) * tot if tot > 0 else 0.1
        v_tol = math.inf if rng.random() < 0.7 else float(rng.uniform(0.2, 1.0)) * max(E_val, 1e-12)
        level, add_k, add_v = O.plan_ladder(res, kprom, vprom, delta, eta, R, eps, v_tol)

        if tot <= eps * (1 - REL_GUARD) and E_val <= v_tol * (1 - REL_GUARD):
            assert (level, add_k, add_v) == (0, [], [])
            seen["level0"] += 1
            checked += 1
            continue
        if abs(tot - eps) <= REL_GUARD * eps or abs(E_key - eps / 2) <= REL_GUARD * eps:
            continue
        assert level in (1, 2)

        # ---- rung 1 ----
        cand_k = [b for b in range(nb) if not kprom[b] and key[b] > 0]
        target_k = eps / 2 * a_all / R            # (S - removed) <= target_k
        if E_key > eps / 2:
            k_min, best = _smallest_cover(cand_k, key, S, target_k)
            if any(abs(S - m - target_k) <= REL_GUARD * max(target_k, 1e-300) for m in best):
                continue
            assert _is_descending_prefix(add_k, cand_k, key), (add_k, cand_k)
            if k_min is None:                     # no subset reaches eps/2: every candidate
                assert sorted(add_k) == sorted(cand_k)
            else:
                assert len(add_k) == k_min, (len(add_k), k_min)
                assert S - math.fsum(key[add_k]) <= target_k * (1 + 1e-12)
                seen["rung1"] += 1
            S_proj = S - math.fsum(key[add_k])
        else:
            assert add_k == []
            S_proj = S
        ek_proj = S_proj / a_all * R

        # ---- rung 2 ----
        cand_v = [b for b in range(nb) if not vprom[b] and val[b] > 0]
        rung2 = ek_proj + E_val > eps or E_val > v_tol
        if abs(ek_proj + E_val - eps) <= REL_GUARD * eps:
            continue
        if not rung2:
            assert level == 1 and add_v == []
            checked += 1
            continue
        assert level == 2
        target_v = min(eps - ek_proj, v_tol)      # E_val - removed <= target_v
        k_min, best = _smallest_cover(cand_v, val, E_val, target_v)
        if any(abs(E_val - m - target_v) <= REL_GUARD * max(abs(target_v), 1e-300) for m in best):
            continue
        assert _is_descending_prefix(add_v, cand_v, val), (add_v, cand_v)
        if k_min is None:
            assert sorted(add_v) == sorted(cand_v)
        else:
            assert len(add_v) == k_min, (len(add_v), k_min)
            assert E_val - math.fsum(val[add_v]) <= target_v + 1e-12 * max(1.0, E_val)
        seen["rung2"] += 1
        seen["rung2_after_1"] += bool(add_k)
        seen["vtol"] += v_tol < math.inf
        checked += 1
    # every branch was exercised many times
    assert checked >= 500, checked
    for k, n in seen.items():
        assert n >= 15, seen


def test_rung1_stops_at_half_eps_not_eps():
    """A hand-sized head: three INT8 blocks whose key terms are 0.5, 0.3 and 0.2 of
    S = 1 (E_key = 1 with A = R = 1) and a value term E_val = 0.1.  Rung 1 removes blocks
    until the projected E_key <= eps/2:
      eps = 1.02 -> target 0.51: the 0.5-block alone (a stop at eps would also take one);
      eps = 0.99 -> target 0.495: two blocks (a stop at eps would take one);
      eps = 0.3  -> target 0.15: all three (a stop at eps would take two).
    Each time the projected E_key + E_val is within eps, so the head stays at rung 1."""
    S, A, R = 1.0, 1.0, 1.0
    pm = np.array([0.5, 0.3, 0.2]) / math.expm1(0.5)
    eta = np.full(3, 0.1 / pm.sum(), np.float32)
    ev = float(np.sum(pm * eta.astype(np.float64)))
    res = O.MixedResult(out=np.zeros(1), e_key=S / A * R, e_val=ev, S=S, A=A, pmass=pm, tail_mass=0.0)
    no = np.zeros(3, bool)
    delta = np.full(3, 0.5)
    assert O.plan_ladder(res, no, no, delta, eta, R, 1.02) == (1, [0], [])
    assert O.plan_ladder(res, no, no, delta, eta, R, 0.99) == (1, [0, 1], [])
    assert O.plan_ladder(res, no, no, delta, eta, R, 0.3) == (1, [0, 1, 2], [])
    # certified as it stands: nothing is planned
    assert O.plan_ladder(res, no, no, delta, eta, R, 1.2) == (0, [], [])
    # blocks with FP16 keys already are not candidates; zero key terms never are
    kp = np.array([True, False, False])
    assert O.plan_ladder(res, kp, no, delta, eta, R, 0.99)[1] == [1, 2]
    assert O.plan_ladder(res, no, no, np.array([0.5, 0.0, 0.5]), eta, R, 0.3)[1] == [0, 2]


def test_rung2_budget_after_rung1():
    """Rung 2 plans against eps minus the projected (not the measured) E_key, and its
    value budget is also bounded by v_tol."""
    pm = np.array([0.4, 0.3, 0.2, 0.1])
    eta = np.array([1.0, 1.0, 1.0, 1.0], np.float32)            # value terms 0.4 .. 0.1
    delta = np.array([math.log(2.0), 0.0, 0.0, 0.0])              # key term of block 0: 0.4
    S, A, R = 0.4, 1.0, 1.0
    res = O.MixedResult(out=np.zeros(1), e_key=0.4, e_val=1.0, S=S, A=A, pmass=pm, tail_mass=0.0)
    no = np.zeros(4, bool)
    # eps = 0.6: E_key 0.4 > 0.3 -> rung 1 takes block 0 (projected E_key 0); rung 2 then
    # needs E_val <= 0.6: remove 0.4 -> 0.6, one block
    assert O.plan_ladder(res, no, no, delta, eta, R, 0.6) == (2, [0], [0])
    # the same with v_tol = 0.35: E_val must reach 0.35: 1.0 - 0.4 - 0.3 = 0.3, two blocks
    assert O.plan_ladder(res, no, no, delta, eta, R, 0.6, 0.35) == (2, [0], [0, 1])
    # eps = 2: certified at level 0 unless v_tol binds
    assert O.plan_ladder(res, no, no, delta, eta, R, 2.0) == (0, [], [])
    assert O.plan_ladder(res, no, no, delta, eta, R, 2.0, 0.5) == (2, [], [0, 1])
    # eps = 0.9: E_key 0.4 <= 0.45, no rung 1; E_val must reach 0.5: two blocks (0.4 + 0.3)
    assert O.plan_ladder(res, no, no, delta, eta, R, 0.9) == (2, [], [0, 1])


# ---------------------------------------------------------------------------------
# ranking-consistency check at R > 1 (hand-built orders)
# ---------------------------------------------------------------------------------

def test_ranking_consistent_positions():
    sel = [0, 1, 2, 3, 4, 5]
    lse8 = np.array([1.0, 5.0, 3.0, 6.0, 2.0, 0.0])    # order 3, 1, 2, 4, 0, 5
    lse16 = np.array([1.5, 5.5, 2.0, 6.5, 3.0, 0.0])   # order 3, 1, 4, 2, 0, 5
    assert O.ranking_consistent(sel, lse8, lse16, 1)
    assert O.ranking_consistent(sel, lse8, lse16, 2)
    assert not O.ranking_consistent(sel, lse8, lse16, 3)
    assert not O.ranking_consistent(sel, lse8, lse16, 6)
    # only the selected blocks count: without block 4 the first five positions agree
    assert O.ranking_consistent([0, 1, 2, 3, 5], lse8, lse16, 5)
    # the top-1 agrees but the second differs
    lse16b = np.array([1.5, 2.5, 5.0, 6.5, 3.0, 0.0])  # order 3, 2, 4, 1, 0, 5
    assert O.ranking_consistent(sel, lse8, lse16b, 1)
    assert not O.ranking_consistent(sel, lse8, lse16b, 2)
    # exact ties go to the lower block index on both sides
    t8 = np.array([4.0, 4.0, 1.0])
    assert O.ranking_consistent([0, 1, 2], t8, np.array([4.0, 3.0, 1.0]), 2)
    assert not O.ranking_consistent([0, 1, 2], t8, np.array([3.0, 4.0, 1.0]), 1)
    assert O.ranking_consistent([1, 2], t8, np.array([0.0, 4.0, 4.0]), 1)
    # fewer selected blocks than positions: the whole order is compared
    assert O.ranking_consistent([2, 5], lse8, lse16, 3)
    assert not O.ranking_consistent([2, 4], lse8, lse16, 3)
    # one selected block (or none) is always consistent
    assert O.ranking_consistent([3], lse8, -lse16, 2)
    assert O.ranking_consistent([], lse8, lse16, 2)


# ---------------------------------------------------------------------------------
# rung 4: at least l4_head_fraction * Hq heads of a sequence at rung 3
# ---------------------------------------------------------------------------------

def _three_failing_heads():
    """The planted-needle construction on 2 KV heads x 4 query heads, with the planted
    query kept on heads 0-2 of group 0 only; every other head gets a fresh Gaussian
    query.  Exactly three heads then fail the ranking check."""
    q, K, V, info = W.c4(batch=1, ctx=4096, Hq=8, Hkv=2)
    q, K, V = q.numpy().copy(), K.numpy(), V.numpy()
    rng = np.random.default_rng(77)
    for h in (3, 4, 5, 6, 7):
        q[0, h] = rng.standard_normal(128).astype(np.float16)
    return q, K, V


@pytest.fixture(scope="module")
def planted3():
    q, K, V = _three_failing_heads()
    return q, K, V, O.quantize_layer(K, V)


def test_rung4_threshold_is_inclusive(planted3):
    q, K, V, t1 = planted3
    base = O.decode_layer(q, K, V, t1, 0.995, 0.25, O.OracleConfig(n_rep=4, l4_head_fraction=0.5))
    assert list(base.rank_ok[0]) == [0, 0, 0, 1, 1, 1, 1, 1]
    assert list(base.level[0, :3]) == [3, 3, 3] and np.all(base.level[0, 3:] < 3)
    assert int(base.ladder_level[0]) == 3
    for rho, want_l4 in ((3 / 8, True), (2 / 8, True), (0.5, False), (3 / 8 + 1e-6, False),
                         (3 / 8 - 1e-6, True), (1.0, False)):
        r = O.decode_layer(q, K, V, t1, 0.995, 0.25, O.OracleConfig(n_rep=4, l4_head_fraction=rho))
        if want_l4:
            assert np.all(r.level[0] == 4) and int(r.ladder_level[0]) == 4, rho
            for h in range(8):
                dense = O.dense_attention(q[0, h], K[0, h // 4], V[0, h // 4])
                assert np.array_equal(r.out[0, h], dense.astype(np.float16))
        else:
            assert np.array_equal(r.level, base.level), rho
            assert np.array_equal(r.out, base.out)
