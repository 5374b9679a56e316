"""Oracle for certified quantized-KV decode attention (plain numpy, CPU).

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the library.  It shares no code, table or
helper with the CUDA path.

Source: "Runtime-Certified Bounded-Error Quantized Attention", gist.science technical
summary (Japanese and French editions).  Section names used below:
  Method §1  tiered storage (INT8 keys per channel, INT4 values per group,
             scale/offset metadata, per-block error annotations; FP16 originals
             in pinned system RAM; fallback to exact dense attention)
  Method §2  two-term error decomposition: E_key (total variation between exact
             and approximate softmax, bounded through the per-token score
             perturbation Delta) and E_val (attention-mass-weighted sum of the
             per-block reconstruction errors eta_b); both computed online from
             quantisation scales, query norms and value ranges
  Method §3  adaptive top-K* selection covering tau_cov of the INT8-estimated
             mass; ranking-consistency check; the four-rung fallback ladder
  Contributions "deterministic recovery": O_dense is returned when the bound
             cannot be met.

The pages give no formulas.  Where they are silent, each function states the reading
(A1..A8) it implements.  The pages print no worked example or bound value, so agreement
with the paper's own numbers is parity unpinned; the functions are pinned instead by
invariants, closed forms and brute force in tests/test_oracle_pins.py, and the ladder
planner (plan_ladder, ranking_consistent, the rung-4 rule) by subset enumeration and
hand-built orders in tests/test_oracle_ladder_pins.py.

Arithmetic.  Quantisation uses IEEE binary32 operations (numpy float32 ops are
correctly rounded) and binary16 storage, spelled out step by step because they fix
integer codes and fp16 scales.  Everything after quantisation is float64.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 64            # tokens per block (the unit of promotion and of eta_b)
VALUE_GROUP = 32      # consecutive channels sharing one INT4 scale/offset
KEY_QMAX = 127        # symmetric INT8 key codes in [-127, 127]
VALUE_QMAX = 15       # asymmetric INT4 value codes in [0, 15]
KAPPA = 0.5 + 2.0 ** -8   # Delta = KAPPA * (1/sqrt(D)) * sum_c |q_c| s_c


@dataclass
class OracleConfig:
    """Knobs of the certified path that the pages leave open (our readings)."""
    n_rep: int = 4                 # query heads per KV head; head h uses KV head h // n_rep
    rank_positions: int = 1        # ranking check compares the top-R positions of S_h
    l4_head_fraction: float = 0.5  # L4 when >= this fraction of a sequence's heads reach L3
    kappa: float = KAPPA
    # FP16-values configuration (the pages' ablation that replaces the INT4 values with
    # FP16 values, Results: structured reasoning): values stay FP16 in VRAM, so every
    # block counts as value-promoted from the start, E_val = 0, rung 2 has nothing to
    # page in and tier 2 holds (and pages in) keys only.
    value_fp16: bool = False
    # Value tolerance v_tol (Results: tightening it closes the value-sensitive gap).  Our
    # reading: a budget on E_val alone, on top of E_key + E_val <= eps; a head is
    # certified only if both hold, and rung 2 pages in values until the projected E_val
    # is within min(v_tol, eps - E_key).  Infinite by default (no separate budget).
    v_tol: float = math.inf


# --------------------------------------------------------------------------------------
# binary16 rounding (IEEE 754): the one rounding mode numpy does not offer directly
# --------------------------------------------------------------------------------------

def f16_round_up(x) -> np.ndarray:
    """Smallest binary16 value >= x, for finite float32 x >= 0.

    Rounding the stored scale *up* keeps |K / s| <= 127 (and (v - o) / s <= 15), so a
    code never has to be clamped by more than one fp32 rounding.
    """
    x = np.asarray(x, dtype=np.float32)
    h = x.astype(np.float16)                       # round to nearest, ties to even
    below = h.astype(np.float32) < x
    h = np.where(below, np.nextafter(h, np.float16(np.inf)), h)
    return h.astype(np.float16)


# --------------------------------------------------------------------------------------
# Method §1: tier-1 quantisation
# --------------------------------------------------------------------------------------

def quantize_key_block(kb: np.ndarray):
    """Per-channel symmetric INT8 keys for one block (Method §1, "INT8 keys per channel").

    Reading A2: one fp16 scale per (block, channel).
      a    = max_t |K[t, c]|                    (exact in fp32)
      s    = round_up_f16(a / 127)              (IEEE fp32 divide)
      code = 0 if s == 0 else clamp(rint(K / s), -127, 127)   (fp32 divide, ties to even)
    kb: float16 [..., 64, D].  Returns (codes int8 [..., 64, D], scales float16 [..., D]).
    """
    k32 = kb.astype(np.float32)
    a = np.max(np.abs(k32), axis=-2)
    s = f16_round_up(a / np.float32(KEY_QMAX))
    s32 = s.astype(np.float32)[..., None, :]
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    r = k32 / safe
    code = np.where(s32 > 0, np.clip(np.rint(r), -KEY_QMAX, KEY_QMAX), np.float32(0.0))
    return code.astype(np.int8), s


def dequantize_keys(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """k_hat = s * code, exact in fp32 (11-bit x 8-bit product), returned as float64."""
    return scales.astype(np.float64)[..., None, :] * codes.astype(np.float64)


def quantize_value_block(vb: np.ndarray):
    """Per-group asymmetric INT4 values for one block (Method §1, "INT4 values per group").

    Reading A3: a group is 32 consecutive channels of one token.
      mn, mx = min, max of the group            (exact in fp32)
      o      = mn                               (an fp16 value, stored exactly)
      s      = round_up_f16((mx - mn) / 15)     (fp32 subtract and divide)
      code   = 0 if s == 0 else clamp(rint((v - o) / s), 0, 15)
      v_hat  = s * code + o                     (fp32; the product is exact)
      eta_b  = max over the block of |v - v_hat| (fp32)   -- the per-block error annotation
    vb: float16 [..., 64, D].  Returns codes uint8 [..., 64, D] (one code per channel,
    unpacked), scales float16 [..., 64, D/32], offsets float16 [..., 64, D/32],
    eta float32 [...].
    """
    lead = vb.shape[:-2]
    T, D = vb.shape[-2:]
    G = D // VALUE_GROUP
    v32 = vb.astype(np.float32).reshape(*lead, T, G, VALUE_GROUP)
    mn = v32.min(axis=-1)
    mx = v32.max(axis=-1)
    o = mn.astype(np.float16)
    s = f16_round_up((mx - mn) / np.float32(VALUE_QMAX))
    s32 = s.astype(np.float32)[..., None]
    o32 = o.astype(np.float32)[..., None]
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    r = (v32 - o32) / safe
    code = np.where(s32 > 0, np.clip(np.rint(r), 0, VALUE_QMAX), np.float32(0.0))
    vhat = s32 * code + o32
    err = np.abs(v32 - vhat)
    eta = err.reshape(*lead, T * D).max(axis=-1).astype(np.float32)
    return code.reshape(*lead, T, D).astype(np.uint8), s, o, eta


def dequantize_values(codes: np.ndarray, scales: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """v_hat = s * code + o in fp32 (as the quantiser computed it), returned as float64."""
    lead = codes.shape[:-2]
    T, D = codes.shape[-2:]
    G = D // VALUE_GROUP
    c32 = codes.astype(np.float32).reshape(*lead, T, G, VALUE_GROUP)
    vhat = scales.astype(np.float32)[..., None] * c32 + offsets.astype(np.float32)[..., None]
    return vhat.reshape(*lead, T, D).astype(np.float64)


@dataclass
class Tier1:
    """Tier-1 (VRAM) contents of one layer, in canonical unpacked layout."""
    kc: np.ndarray     # int8    [B, Hkv, nb, 64, D]
    ks: np.ndarray     # float16 [B, Hkv, nb, D]
    vc: np.ndarray     # uint8   [B, Hkv, nb, 64, D]   (codes 0..15)
    vs: np.ndarray     # float16 [B, Hkv, nb, 64, D/32]
    vo: np.ndarray     # float16 [B, Hkv, nb, 64, D/32]
    eta: np.ndarray    # float32 [B, Hkv, nb]
    vmin: np.ndarray   # float32 [B, Hkv, D]   over every cached token
    vmax: np.ndarray   # float32 [B, Hkv, D]


def quantize_layer(K: np.ndarray, V: np.ndarray) -> Tier1:
    """Quantise every full 64-token block of a layer; track value ranges (Method §1, §2).

    K, V: float16 [B, Hkv, N, D] (the FP16 originals, i.e. tier 2).  The last N mod 64
    tokens form the partial block, which stays FP16 until it fills (reading A2).
    Reading A4: the value range used by E_key is the per-channel min/max over every
    cached token, partial block included.
    """
    B, H, N, D = K.shape
    nb = N // BLOCK
    kb = K[:, :, : nb * BLOCK].reshape(B, H, nb, BLOCK, D)
    vb = V[:, :, : nb * BLOCK].reshape(B, H, nb, BLOCK, D)
    kc, ks = quantize_key_block(kb)
    vc, vs, vo, eta = quantize_value_block(vb)
    if N > 0:
        v32 = V.astype(np.float32)
        vmin, vmax = v32.min(axis=2), v32.max(axis=2)
    else:
        vmin = np.full((B, H, D), np.inf, np.float32)
        vmax = np.full((B, H, D), -np.inf, np.float32)
    return Tier1(kc, ks, vc, vs, vo, eta, vmin, vmax)


# --------------------------------------------------------------------------------------
# Dense exact attention (Method §1 fallback; Contributions "deterministic recovery")
# --------------------------------------------------------------------------------------

def softmax(x: np.ndarray) -> np.ndarray:
    m = np.max(x)
    e = np.exp(x - m)
    return e / e.sum()


def logsumexp(x: np.ndarray) -> float:
    if x.size == 0:
        return -math.inf
    m = float(np.max(x))
    if m == -math.inf:
        return -math.inf
    return m + math.log(float(np.exp(x - m).sum()))


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """O_dense = softmax(q . K^T / sqrt(D)) V over the FP16 originals, in float64.

    Reading A1: scale 1/sqrt(D); q [D], K and V [N, D].
    """
    D = q.shape[-1]
    s = K.astype(np.float64) @ q.astype(np.float64) / math.sqrt(D)
    return softmax(s) @ V.astype(np.float64)


# --------------------------------------------------------------------------------------
# Method §3 light INT8 scoring pass and Method §2 runtime quantities
# --------------------------------------------------------------------------------------

def int8_scores(q: np.ndarray, kc: np.ndarray, ks: np.ndarray) -> np.ndarray:
    """s_hat[b, t] = (1/sqrt(D)) sum_c q_c * (s_{b,c} * code_{b,t,c}) for every full block."""
    D = q.shape[-1]
    return dequantize_keys(kc, ks) @ q.astype(np.float64) / math.sqrt(D)


def block_logsumexp(scores: np.ndarray) -> np.ndarray:
    """Per-block log of the summed exponentials: scores [nb, 64] -> [nb]."""
    if scores.shape[0] == 0:
        return np.zeros(0)
    m = scores.max(axis=1)
    return m + np.log(np.exp(scores - m[:, None]).sum(axis=1))


def score_perturbation(q: np.ndarray, ks: np.ndarray, kappa: float = KAPPA) -> np.ndarray:
    """Delta_b, the bound on |s_t - s_hat_t| for every token of INT8 block b (Method §2).

    Reading A5 (Hoelder with the scale-weighted l1 norm of the query):
      |s_t - s_hat_t| = (1/sqrt(D)) |sum_c q_c (K_tc - k_hat_tc)|
                     <= (1/sqrt(D)) sum_c |q_c| s_bc (1/2 + 2^-17),
    and kappa = 1/2 + 2^-8 leaves slack for fp rounding of the computed scores.
    """
    D = q.shape[-1]
    return kappa * (ks.astype(np.float64) @ np.abs(q.astype(np.float64))) / math.sqrt(D)


def select_top_k_star(lse8: np.ndarray, tail_lse: float, tau_cov: float):
    """Adaptive top-K* (Method §3): the fewest blocks whose estimated mass covers tau_cov.

    Reading A6: mass_b = exp(lse8_b - LSE), LSE over every token (INT8 scores for full
    blocks, exact scores for the FP16 partial block, whose mass counts as covered).
    Blocks are taken in descending mass (ties: lower block index first) until
    tail_mass + sum >= tau_cov.  Returns (selected block ids in that order, mass [nb],
    tail_mass, cumulative covered mass after each selected block).
    """
    nb = lse8.shape[0]
    LSE = logsumexp(np.concatenate([lse8, [tail_lse]]))
    mass = np.exp(lse8 - LSE)
    tail_mass = math.exp(tail_lse - LSE) if tail_lse > -math.inf else 0.0
    order = sorted(range(nb), key=lambda b: (-mass[b], b))
    covered = tail_mass
    chosen, cum = [], []
    for b in order:
        if covered >= tau_cov:
            break
        chosen.append(b)
        covered += mass[b]
        cum.append(covered)
    return chosen, mass, tail_mass, cum


@dataclass
class MixedResult:
    out: np.ndarray          # [D] float64
    e_key: float
    e_val: float
    S: float                 # sum_t p_hat_t (e^Delta_t - 1)
    A: float                 # sum_t p_hat_t e^-Delta_t
    pmass: np.ndarray        # [nb] p_hat mass of each full block
    tail_mass: float


def mixed_attention(s_exact: np.ndarray, s_hat: np.ndarray, V: np.ndarray, v_hat: np.ndarray,
                    delta: np.ndarray, eta: np.ndarray, R: float,
                    kprom: np.ndarray, vprom: np.ndarray) -> MixedResult:
    """Mixed-precision attention and its certificate (Method §2, §3).

    s_exact [N]    q.k/sqrt(D) with the FP16 keys       (used on promoted blocks and
                   the partial block)
    s_hat [nb, 64] INT8 scores                          (used on the other blocks)
    V [N, D]       FP16 values;  v_hat [nb, 64, D] INT4 reconstructions
    delta [nb]     per-block score perturbation bound;  eta [nb]  reconstruction error
    R              max_c (vmax_c - vmin_c)
    kprom, vprom   bool [nb]: blocks whose FP16 keys / values are paged in

    Reading A7.  p_hat = softmax(s'), O_hat = sum_t p_hat_t v'_t.  With Delta_t the
    perturbation of token t (0 where the key is exact):
      S = sum_t p_hat_t (e^Delta_t - 1),  A = sum_t p_hat_t e^-Delta_t,
      E_key = (S / A) * R        (TV(p, p_hat) <= S/A, times the value range)
      E_val = sum over blocks with INT4 values of mass_b * eta_b.
    """
    N, D = V.shape
    nb = s_hat.shape[0]
    T = nb * BLOCK
    int8_tok = ~np.repeat(kprom, BLOCK)
    s_prime = s_exact.astype(np.float64).copy()
    s_prime[:T][int8_tok] = s_hat.reshape(T)[int8_tok]
    delta_t = np.zeros(N)
    delta_t[:T][int8_tok] = np.repeat(delta, BLOCK)[int8_tok]
    p = softmax(s_prime)
    v_prime = V.astype(np.float64).copy()
    int4_tok = ~np.repeat(vprom, BLOCK)
    v_prime[:T][int4_tok] = v_hat.reshape(T, D)[int4_tok]
    out = p @ v_prime
    S = float(np.sum(p * np.expm1(delta_t)))
    A = float(np.sum(p * np.exp(-delta_t)))
    e_key = S / A * R
    pmass = p[:T].reshape(nb, BLOCK).sum(axis=1)
    tail_mass = float(p[T:].sum())
    e_val = float(np.sum(pmass[~vprom] * eta[~vprom].astype(np.float64)))
    return MixedResult(out, e_key, e_val, S, A, pmass, tail_mass)


def ranking_consistent(sel: list, lse8: np.ndarray, lse16: np.ndarray, positions: int = 1) -> bool:
    """Ranking-consistency check (Method §3).

    Reading A8: order the selected blocks S_h by INT8 block log-mass and by FP16 block
    log-mass (ties: lower block index first); consistent when the first `positions`
    entries of the two orders agree.
    """
    if len(sel) <= 1:
        return True
    by8 = sorted(sel, key=lambda b: (-lse8[b], b))[:positions]
    by16 = sorted(sel, key=lambda b: (-lse16[b], b))[:positions]
    return by8 == by16


def plan_ladder(res: MixedResult, kprom: np.ndarray, vprom: np.ndarray, delta: np.ndarray,
                eta: np.ndarray, R: float, eps: float, v_tol: float = math.inf):
    """Rungs 1 and 2 of the fallback ladder for one head (Method §3).

    Reading A8.  Certified at level 0 when E_key + E_val <= eps.  Otherwise:
      rung 1 (expand coverage) when E_key > eps/2: add INT8 blocks in descending
        contribution mass_b (e^Delta_b - 1) (ties: lower index; zero contributions
        never) until the projected (S - sum added)/A * R <= eps/2;
      rung 2 (value promotion) when projected E_key + E_val > eps, or E_val > v_tol:
        page in FP16 values of blocks in descending mass_b * eta_b (same tie rule) until
        the projected E_val <= min(v_tol, eps - projected E_key).
    Returns (level, blocks to add to the key set, blocks to add to the value set).
    """
    if res.e_key + res.e_val <= eps and res.e_val <= v_tol:
        return 0, [], []
    level = 0
    add_k: list = []
    S_proj = res.S
    if res.e_key > eps / 2:
        level = 1
        contrib = res.pmass * np.expm1(delta)
        cand = [b for b in range(len(contrib)) if not kprom[b] and contrib[b] > 0]
        cand.sort(key=lambda b: (-contrib[b], b))
        for b in cand:
            if S_proj / res.A * R <= eps / 2:
                break
            add_k.append(b)
            S_proj -= contrib[b]
    ekey_proj = S_proj / res.A * R
    add_v: list = []
    if ekey_proj + res.e_val > eps or res.e_val > v_tol:
        level = 2
        contrib_v = res.pmass * eta.astype(np.float64)
        cand = [b for b in range(len(contrib_v)) if not vprom[b] and contrib_v[b] > 0]
        cand.sort(key=lambda b: (-contrib_v[b], b))
        ev_proj = res.e_val
        for b in cand:
            if ekey_proj + ev_proj <= eps and ev_proj <= v_tol:
                break
            add_v.append(b)
            ev_proj -= contrib_v[b]
    return level, add_k, add_v


# --------------------------------------------------------------------------------------
# One decode step of one layer
# --------------------------------------------------------------------------------------

@dataclass
class DecodeResult:
    out: np.ndarray            # float16 [B, Hq, D]
    out64: np.ndarray          # float64 [B, Hq, D] before the final fp16 rounding
    e_key: np.ndarray          # [B, Hq]
    e_val: np.ndarray
    rank_ok: np.ndarray        # int [B, Hq]
    level: np.ndarray          # int [B, Hq]
    k_star: np.ndarray         # int [B, Hq]
    n_val_promoted: np.ndarray  # int [B, Hq]
    promoted_bytes: np.ndarray  # int64 [B, Hq]: tier-2 bytes paged in for the head's KV group
                                # (FP16 key blocks of the union U, plus rung-1 key blocks,
                                # rung-2 value blocks, and, when a head of the group goes
                                # dense, the values of every full block and the keys of
                                # the blocks not paged in before)
    ladder_level: np.ndarray   # int [B]
    # diagnostics for parity tests
    sel: list = field(default_factory=list)      # [B][Hq] selected blocks in order
    cum: list = field(default_factory=list)      # [B][Hq] covered mass after each pick
    mass: np.ndarray = None    # [B, Hq, nb] INT8-estimated mass
    lse8: np.ndarray = None    # [B, Hq, nb]
    lse16: np.ndarray = None   # [B, Hq, nb]
    delta: np.ndarray = None   # [B, Hq, nb]
    kprom0: np.ndarray = None  # bool [B, Hkv, nb] round-0 key set U
    kprom1: np.ndarray = None  # bool [B, Hkv, nb] round-1 key set (== kprom0 if none)
    vprom1: np.ndarray = None  # bool [B, Hkv, nb] round-1 value set
    round1: np.ndarray = None  # bool [B, Hq] head took a round-1 result
    planned: np.ndarray = None  # int [B, Hq] rung requested at round 0 (0, 1, 2; 3 = rank)
    e_key0: np.ndarray = None  # [B, Hq] round-0 bounds
    e_val0: np.ndarray = None


def decode_layer(q: np.ndarray, K: np.ndarray, V: np.ndarray, t1: Tier1,
                 tau_cov: float, eps: float, cfg: OracleConfig = OracleConfig()) -> DecodeResult:
    """Certified decode attention for one layer (Method §1-§3, deterministic recovery).

    q: float16 [B, Hq, D];  K, V: float16 [B, Hkv, N, D] (FP16 originals);  t1 from
    quantize_layer(K, V).  Returns outputs, per-head certificates and per-sequence
    ladder level.  Reading A8 for the ladder:
      * a head whose ranking check fails goes to rung 3 (dense for that head);
      * rungs 1/2 add key/value blocks to the KV group's promoted sets (union over the
        heads that ask), then the asking heads are recomputed ("round 1"); a head still
        above eps after that goes to rung 3; other heads keep their round-0 result;
      * rung 4: tau_cov >= 1, or at least l4_head_fraction of a sequence's heads at
        rung 3, sends every head of that sequence to dense attention;
      * rungs 3 and 4 return fp16(O_dense) with E_key = E_val = 0.
    """
    B, Hq, D = q.shape
    _, Hkv, N, _ = K.shape
    assert Hq == Hkv * cfg.n_rep
    nb = N // BLOCK
    T = nb * BLOCK
    blk_bytes = BLOCK * D * 2
    inv = 1.0 / math.sqrt(D)

    out64 = np.zeros((B, Hq, D))
    e_key = np.zeros((B, Hq)); e_val = np.zeros((B, Hq))
    e_key0 = np.zeros((B, Hq)); e_val0 = np.zeros((B, Hq))
    rank_ok = np.ones((B, Hq), np.int64)
    level = np.zeros((B, Hq), np.int64)
    planned = np.zeros((B, Hq), np.int64)
    k_star = np.zeros((B, Hq), np.int64)
    n_vprom = np.zeros((B, Hq), np.int64)
    round1 = np.zeros((B, Hq), bool)
    mass_all = np.zeros((B, Hq, nb)); lse8_all = np.zeros((B, Hq, nb))
    lse16_all = np.zeros((B, Hq, nb)); delta_all = np.zeros((B, Hq, nb))
    kprom0 = np.zeros((B, Hkv, nb), bool); kprom1 = np.zeros((B, Hkv, nb), bool)
    vprom1 = np.zeros((B, Hkv, nb), bool)
    group_bytes = np.zeros((B, Hkv), np.int64)
    sel_all = [[[] for _ in range(Hq)] for _ in range(B)]
    cum_all = [[[] for _ in range(Hq)] for _ in range(B)]

    if tau_cov >= 1.0:
        level[:] = 4
        k_star[:] = nb
    else:
        for b in range(B):
            for g in range(Hkv):
                heads = list(range(g * cfg.n_rep, (g + 1) * cfg.n_rep))
                Kg = K[b, g]; Vg = V[b, g]
                V64 = Vg.astype(np.float64)
                v_hat = dequantize_values(t1.vc[b, g], t1.vs[b, g], t1.vo[b, g])
                eta = t1.eta[b, g]
                R = float(np.max(t1.vmax[b, g].astype(np.float64) - t1.vmin[b, g].astype(np.float64)))
                per = {}
                for h in heads:
                    qh = q[b, h]
                    s_ex = Kg.astype(np.float64) @ qh.astype(np.float64) * inv
                    s_hat = int8_scores(qh, t1.kc[b, g], t1.ks[b, g])
                    lse8 = block_logsumexp(s_hat)
                    lse16 = block_logsumexp(s_ex[:T].reshape(nb, BLOCK))
                    tail_lse = logsumexp(s_ex[T:])
                    delta = score_perturbation(qh, t1.ks[b, g], cfg.kappa)
                    chosen, mass, _, cum = select_top_k_star(lse8, tail_lse, tau_cov)
                    per[h] = dict(s_ex=s_ex, s_hat=s_hat, lse8=lse8, lse16=lse16,
                                  delta=delta, chosen=chosen)
                    mass_all[b, h] = mass; lse8_all[b, h] = lse8
                    lse16_all[b, h] = lse16; delta_all[b, h] = delta
                    sel_all[b][h] = chosen; cum_all[b][h] = cum
                    k_star[b, h] = len(chosen)
                U = np.zeros(nb, bool)
                for h in heads:
                    U[per[h]["chosen"]] = True
                Vp = np.full(nb, cfg.value_fp16, bool)   # FP16 values resident in VRAM
                kprom0[b, g] = U
                group_bytes[b, g] += int(U.sum()) * blk_bytes
                adds_k, adds_v, asking = [], [], []
                for h in heads:
                    P = per[h]
                    r0 = mixed_attention(P["s_ex"], P["s_hat"], Vg, v_hat, P["delta"], eta, R, U, Vp)
                    P["r0"] = r0
                    out64[b, h] = r0.out
                    e_key[b, h] = e_key0[b, h] = r0.e_key
                    e_val[b, h] = e_val0[b, h] = r0.e_val
                    ok = ranking_consistent(P["chosen"], P["lse8"], P["lse16"], cfg.rank_positions)
                    rank_ok[b, h] = int(ok)
                    if not ok:
                        level[b, h] = planned[b, h] = 3
                        continue
                    lv, ak, av = plan_ladder(r0, U, Vp, P["delta"], eta, R, eps, cfg.v_tol)
                    level[b, h] = planned[b, h] = lv
                    if lv > 0:
                        asking.append(h); adds_k += ak; adds_v += av
                U1 = U.copy(); V1 = Vp.copy()
                if asking:
                    U1[adds_k] = True
                    V1[adds_v] = True
                    # each FP16 block is paged in once per call: rung 1 adds only the
                    # new key blocks, rung 2 the new value blocks
                    group_bytes[b, g] += (int(U1.sum()) - int(U.sum())
                                          + int(V1.sum()) - int(Vp.sum())) * blk_bytes
                    for h in asking:
                        P = per[h]
                        r1 = mixed_attention(P["s_ex"], P["s_hat"], Vg, v_hat, P["delta"], eta, R, U1, V1)
                        round1[b, h] = True
                        out64[b, h] = r1.out
                        e_key[b, h] = r1.e_key
                        e_val[b, h] = r1.e_val
                        n_vprom[b, h] = int(V1.sum()) - int(Vp.sum())   # paged in
                        if r1.e_key + r1.e_val > eps or r1.e_val > cfg.v_tol:
                            level[b, h] = 3
                kprom1[b, g] = U1; vprom1[b, g] = V1

        # rung 4: a sequence with enough heads at rung 3 goes dense as a whole
        for b in range(B):
            if np.sum(level[b] == 3) >= cfg.l4_head_fraction * Hq:
                level[b, :] = 4

    # rungs 3 and 4: exact dense recompute over the FP16 originals
    for b in range(B):
        for g in range(Hkv):
            heads = range(g * cfg.n_rep, (g + 1) * cfg.n_rep)
            if any(level[b, h] >= 3 for h in heads):
                # values of every full block from tier 2 (none with FP16 values resident),
                # keys of the blocks whose FP16 keys this call has not paged in already
                # (the FP16 scores of those are reused; all of them at tau_cov >= 1)
                k_new = nb - (int(kprom1[b, g].sum()) if tau_cov < 1.0 else 0)
                group_bytes[b, g] += (k_new + (0 if cfg.value_fp16 else nb)) * blk_bytes
            for h in heads:
                if level[b, h] >= 3:
                    out64[b, h] = dense_attention(q[b, h], K[b, g], V[b, g])
                    e_key[b, h] = 0.0
                    e_val[b, h] = 0.0

    promoted_bytes = np.zeros((B, Hq), np.int64)
    for h in range(Hq):
        promoted_bytes[:, h] = group_bytes[:, h // cfg.n_rep]
    return DecodeResult(
        out=out64.astype(np.float16), out64=out64, e_key=e_key, e_val=e_val,
        rank_ok=rank_ok, level=level, k_star=k_star, n_val_promoted=n_vprom,
        promoted_bytes=promoted_bytes, ladder_level=level.max(axis=1),
        sel=sel_all, cum=cum_all, mass=mass_all, lse8=lse8_all, lse16=lse16_all,
        delta=delta_all, kprom0=kprom0, kprom1=kprom1, vprom1=vprom1, round1=round1,
        planned=planned, e_key0=e_key0, e_val0=e_val0)


@dataclass
class UncertifiedResult:
    out: np.ndarray          # float16 [B, Hq, D]
    out64: np.ndarray        # float64 [B, Hq, D] before the final rounding
    e_key: np.ndarray        # [B, Hq] bound of the returned output (not enforced)
    e_val: np.ndarray


def uncertified_decode_layer(q: np.ndarray, K: np.ndarray, V: np.ndarray, t1: Tier1,
                             cfg: OracleConfig = OracleConfig()) -> UncertifiedResult:
    """The plain INT8/INT4 baseline the paper compares against (Experiments, retrieval):
    INT8 key scores and INT4 values on every full block, the FP16 originals on the
    partial block, nothing promoted and no ladder.  Its output is mixed_attention with
    empty promotion sets (every block value-promoted with FP16 values, cfg.value_fp16);
    the bounds are those of that output, reported only."""
    B, Hq, D = q.shape
    _, Hkv, N, _ = K.shape
    assert Hq % Hkv == 0
    n_rep = Hq // Hkv
    nb = N // BLOCK
    inv = 1.0 / math.sqrt(D)
    none = np.zeros(nb, bool)
    vprom = np.full(nb, cfg.value_fp16, bool)
    out64 = np.zeros((B, Hq, D))
    e_key = np.zeros((B, Hq)); e_val = np.zeros((B, Hq))
    for b in range(B):
        for g in range(Hkv):
            Kg, Vg = K[b, g], V[b, g]
            v_hat = dequantize_values(t1.vc[b, g], t1.vs[b, g], t1.vo[b, g])
            R = float(np.max(t1.vmax[b, g].astype(np.float64) - t1.vmin[b, g].astype(np.float64)))
            for h in range(g * n_rep, (g + 1) * n_rep):
                qh = q[b, h]
                s_ex = Kg.astype(np.float64) @ qh.astype(np.float64) * inv
                s_hat = int8_scores(qh, t1.kc[b, g], t1.ks[b, g])
                delta = score_perturbation(qh, t1.ks[b, g], cfg.kappa)
                r = mixed_attention(s_ex, s_hat, Vg, v_hat, delta, t1.eta[b, g], R, none, vprom)
                out64[b, h] = r.out
                e_key[b, h] = r.e_key
                e_val[b, h] = r.e_val
    return UncertifiedResult(out64.astype(np.float16), out64, e_key, e_val)

