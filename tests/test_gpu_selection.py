"""Top-K* block selection on the GPU at its tie path and with several histogram levels.

Every 64-token block of these caches is the same block, so each block's INT8 log-mass is
computed from identical codes and scales: on the GPU the heads' block masses tie exactly,
and in the oracle too.  The selection takes blocks by descending mass, ties to the lower
index (Runtime-Certified Bounded-Error Quantized Attention, Method §3: the fewest blocks
covering tau_cov of the estimated mass), so the selected set is the lowest indices, as
many as the oracle's cumulative count.  With more than 256 tied candidates the GPU no
longer ranks them one by one; it takes the tied key's blocks in index order.  One block
of each KV group made heavier widens the key range, so that histogram levels narrow it
down to the tied key before the tie rule applies.  A last case spreads the blocks' masses
a little, for the exact ranking of a bucket's candidates behind the heavier block.
"""

import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import workloads as W  # noqa: E402
from _parity import gpu_run, oracle_run  # noqa: E402

NB = 640          # blocks: more tied candidates than the selection ranks one by one (256)
OUTLIER = 100     # the heavier block of the second case


def _repeated_cache(seed, outlier_gain=0.0):
    """B = 1, 8 query / 2 KV heads, NB identical blocks (optionally one heavier block)."""
    q, K, V = W.tiny(seed=seed, ctx=64, Hq=8, Hkv=2, kscale=3.0)
    Kf = K.float().repeat(1, 1, NB, 1)
    Vf = V.float().repeat(1, 1, NB, 1)
    if outlier_gain:
        # add the group's summed queries to the block's keys: every head of the group
        # scores it higher (by about outlier_gain per token)
        qf = q.float().reshape(1, 2, 4, 128)
        for g in range(2):
            s = qf[0, g].sum(0)
            c = outlier_gain * math.sqrt(128.0) / float(qf[0, g].pow(2).sum(1).mean())
            Kf[0, g, 64 * OUTLIER:64 * (OUTLIER + 1)] += c * s
    return q, Kf.half(), Vf.half()


def _expected_sets(r, tau):
    """The oracle's selected blocks per head, and the margin of its boundary to tau."""
    sets, margin = {}, math.inf
    for h in range(r.level.shape[1]):
        sel = [int(i) for i in r.sel[0][h]]
        sets[h] = sel
        m = np.asarray(r.mass[0][h], dtype=np.float64)
        cum = float(np.sum(m[sel]))
        before = cum - float(m[sel[-1]])
        margin = min(margin, cum - tau, tau - before)
    return sets, margin


@pytest.mark.parametrize("tau", [0.9004, 0.5003])
def test_all_blocks_tied(tau):
    q, K, V = _repeated_cache(31)
    g = gpu_run(q, K, V, tau, 0.25)
    _, r = oracle_run(q, K, V, tau, 0.25)
    sets, margin = _expected_sets(r, tau)
    assert margin > 1e-5, f"tau {tau} too close to a block boundary ({margin:.2e})"
    sel = g["state"]["sel"].numpy().astype(bool)
    lse8 = g["state"]["lse8"].numpy()
    for h in range(8):
        assert np.all(lse8[0, h] == lse8[0, h, 0]), "block log-masses are not tied on the GPU"
        want = sets[h]
        assert want == list(range(len(want))), "oracle did not break the ties by index"
        got = np.nonzero(sel[0, h])[0].tolist()
        assert got == want, f"head {h}: selected {len(got)} blocks, first gap at " \
                            f"{next((i for i, x in enumerate(got) if i != x), None)}; want {len(want)}"
        assert int(g["cert"]["k_star"][0, h]) == len(want)


@pytest.mark.parametrize("tau", [0.9004, 0.7002])
def test_tied_blocks_behind_one_heavier_block(tau):
    q, K, V = _repeated_cache(32, outlier_gain=5.0)
    g = gpu_run(q, K, V, tau, 0.25)
    _, r = oracle_run(q, K, V, tau, 0.25)
    sets, margin = _expected_sets(r, tau)
    assert margin > 1e-5, f"tau {tau} too close to a block boundary ({margin:.2e})"
    sel = g["state"]["sel"].numpy().astype(bool)
    lse8 = g["state"]["lse8"].numpy()
    for h in range(8):
        others = np.delete(lse8[0, h], OUTLIER)
        assert np.all(others == others[0]) and lse8[0, h, OUTLIER] > others[0] + 2.0
        want = sets[h]
        assert want[0] == OUTLIER
        rest = sorted(want[1:])
        assert rest == [i for i in range(NB) if i != OUTLIER][:len(rest)], "oracle order"
        got = sorted(np.nonzero(sel[0, h])[0].tolist())
        assert got == sorted(want), f"head {h}: {len(got)} blocks selected, {len(want)} wanted"
        assert int(g["cert"]["k_star"][0, h]) == len(want)


def test_close_masses_behind_one_heavier_block():
    """Block i's keys scaled by 1 + 0.05 i / NB (rounded to fp16, so runs of a few
    consecutive blocks stay identical): the non-outlier masses span a few percent and
    fall into a handful of the outlier-stretched range's buckets, so the crossing bucket
    typically holds dozens of candidates, some tied, for the exact ranking.  The GPU's
    sets match the oracle's outside the selection band, and on the GPU's own log-masses
    every selected block ranks at or above every unselected one."""
    from _parity import ambiguous_blocks
    tau = 0.8
    q, K, V = _repeated_cache(33, outlier_gain=5.0)
    Kf = K.float()
    scale = 1.0 + 0.05 * torch.arange(NB, dtype=torch.float32) / NB
    Kf = Kf * scale.repeat_interleave(64).view(1, 1, -1, 1)
    K = Kf.half()
    g = gpu_run(q, K, V, tau, 0.25)
    _, r = oracle_run(q, K, V, tau, 0.25)
    sel = g["state"]["sel"].numpy().astype(bool)
    lse8 = g["state"]["lse8"].numpy().astype(np.float64)
    compared = 0
    for h in range(8):
        want = np.zeros(NB, bool)
        want[r.sel[0][h]] = True
        amb = ambiguous_blocks(r, 0, h, tau)
        bad = [int(i) for i in np.nonzero(sel[0, h] != want)[0] if int(i) not in amb]
        assert not bad, f"head {h}: selection differs from the oracle on blocks {bad[:10]}"
        compared += NB - len(amb)
        s, u = lse8[0, h][sel[0, h]], lse8[0, h][~sel[0, h]]
        assert sel[0, h, OUTLIER]
        assert u.size == 0 or u.max() <= s.min() + 1e-6, f"head {h}: an unselected block ranks higher"
        assert 256 < int(sel[0, h].sum()) < NB
    assert compared >= 8 * NB // 2, compared
