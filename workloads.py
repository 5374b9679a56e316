"""Seeded synthetic inputs for certified quantized-KV decode attention.

The shapes follow a Llama-3.1-8B attention layer (32 query heads, 8 KV heads,
head_dim 128), the model the paper evaluates on.  Trained weights and the paper's
datasets are not available, so random tensors with the structure described per
workload stand in for them.  This module draws q, K and V only: it holds none of the
method's arithmetic, and both the oracle and the CUDA path are fed from it.

Every generator takes a ``device``; tensors drawn on the CPU use a CPU
``torch.Generator`` and tensors drawn on a GPU a CUDA one, so the same seed gives
different (but equally distributed) values on the two devices.  A test draws once and
hands the same tensors to both sides.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

N_Q_HEADS = 32
N_KV_HEADS = 8
HEAD_DIM = 128
BLOCK = 64


@dataclass
class Workload:
    name: str
    batch: int
    ctx: int
    n_layers: int
    tau_cov: float
    eps: float
    seed: int
    n_q_heads: int = N_Q_HEADS
    n_kv_heads: int = N_KV_HEADS
    head_dim: int = HEAD_DIM


# Epsilon is not given by the paper; 0.25 (absolute, max-abs over the head's output)
# lets Gaussian values in 32-channel INT4 groups certify at rung 0 while value groups
# with an 8x range need rung 2.
DEFAULT_EPS = 0.25

WORKLOADS = {
    "c1_ctx4k": Workload("c1_ctx4k", 1, 4096, 1, 0.995, DEFAULT_EPS, 0),
    "c2_lowrank_ctx32k_b4": Workload("c2_lowrank_ctx32k_b4", 4, 32768, 1, 0.995, DEFAULT_EPS, 1),
    "c3_llama8b_ctx128k_32l": Workload("c3_llama8b_ctx128k_32l", 1, 131072, 32, 0.995, DEFAULT_EPS, 2),
    "c4_planted_ctx64k_b8": Workload("c4_planted_ctx64k_b8", 8, 65536, 1, 0.995, DEFAULT_EPS, 3),
}

C2_BETA = 10.0   # hot-block boost along the query direction (>= 99% of dense mass hot)
C2_RANK = 16
C2_HOT_FRACTION = 0.05


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(gen, shape, device, dtype=torch.float32):
    return torch.randn(*shape, generator=gen, device=device, dtype=dtype)


def outlier_keys(gen, B, Hkv, N, D, device, n_out=4, scale=20.0):
    """K ~ N(0,1) with `n_out` channels per KV head (drawn from gen) scaled by `scale`."""
    K = _randn(gen, (B, Hkv, N, D), device)
    for g in range(Hkv):
        ch = torch.randperm(D, generator=gen, device=device)[:n_out]
        K[:, g, :, ch] *= scale
    return K


def queries(gen, B, Hq, D, device):
    return _randn(gen, (B, Hq, D), device)


def c1(device="cpu", seed=0, batch=1, ctx=4096, Hq=N_Q_HEADS, Hkv=N_KV_HEADS, D=HEAD_DIM):
    """Gaussian q, K, V; four key channels per KV head scaled x20."""
    gen = _gen(device, seed)
    K = outlier_keys(gen, batch, Hkv, ctx, D, device)
    V = _randn(gen, (batch, Hkv, ctx, D), device)
    q = queries(gen, batch, Hq, D, device)
    return q.half(), K.half(), V.half()


def c2(device="cpu", seed=1, batch=4, ctx=32768, Hq=N_Q_HEADS, Hkv=N_KV_HEADS, D=HEAD_DIM,
       beta=C2_BETA):
    """Low-rank keys with the attention mass concentrated in ~5% of the blocks.

    Per KV head: K_t = U z_t + N(0, 0.1^2), U in R^{D x 16} with N(0, 1/16) entries,
    z_t ~ N(0, I_16).  The heads of the group query along U (w + 0.3 xi_h) with a shared
    w, scaled to norm sqrt(D).  On 5% of the blocks (drawn from the seed) every token
    gets z_t += beta * w / |w|.
    """
    gen = _gen(device, seed)
    n_rep = Hq // Hkv
    nb = ctx // BLOCK
    K = torch.empty(batch, Hkv, ctx, D, device=device)
    q = torch.empty(batch, Hq, D, device=device)
    for b in range(batch):
        for g in range(Hkv):
            U = _randn(gen, (D, C2_RANK), device) / math.sqrt(C2_RANK)
            w = _randn(gen, (C2_RANK,), device)
            z = _randn(gen, (ctx, C2_RANK), device)
            n_hot = max(1, int(round(C2_HOT_FRACTION * nb)))
            hot = torch.randperm(nb, generator=gen, device=device)[:n_hot]
            tok = (hot[:, None] * BLOCK + torch.arange(BLOCK, device=device)[None, :]).reshape(-1)
            z[tok] += beta * w / w.norm()
            K[b, g] = z @ U.T + 0.1 * _randn(gen, (ctx, D), device)
            for r in range(n_rep):
                wh = w + 0.3 * _randn(gen, (C2_RANK,), device)
                dirn = U @ wh
                q[b, g * n_rep + r] = math.sqrt(D) * dirn / dirn.norm()
    V = _randn(gen, (batch, Hkv, ctx, D), device)
    return q.half(), K.half(), V.half()


def c3_layer(layer: int, device="cpu", seed=2, batch=1, ctx=131072, Hq=N_Q_HEADS,
             Hkv=N_KV_HEADS, D=HEAD_DIM, group=32, frac=0.01, vscale=8.0):
    """One layer of the 128K workload: keys as c1; 1% of value groups with range x8."""
    gen = _gen(device, seed * 1000 + layer)
    K = outlier_keys(gen, batch, Hkv, ctx, D, device)
    V = _randn(gen, (batch, Hkv, ctx, D // group, group), device)
    big = torch.rand(batch, Hkv, ctx, D // group, generator=gen, device=device) < frac
    V = torch.where(big[..., None], V * vscale, V).reshape(batch, Hkv, ctx, D)
    q = queries(gen, batch, Hq, D, device)
    return q.half(), K.half(), V.half()


def c4(device="cpu", seed=3, batch=8, ctx=65536, Hq=N_Q_HEADS, Hkv=N_KV_HEADS, D=HEAD_DIM,
       margin=0.05):
    """Planted-needle retrieval where INT8 rounding flips the top block.

    Background keys as c1.  Per (sequence, KV head) the query heads share one query q,
    and two blocks are rewritten: a planted block in the first quarter of the context
    and a decoy block elsewhere.  Both contain an anchor token with every channel at
    -sign(q_c) * 127/32 (which pins every channel scale of the block to exactly 1/32),
    61..62 filler tokens N(0,1) clipped to +-3.9, and one needle token.  The planted
    needle has channel c at sign(q_c) (n + 7/16)/32, just below a half step, so INT8
    rounding lowers its score by (7/16)(1/32) sum|q_c| / sqrt(D); the decoy needle lies
    on the grid (exact in INT8) and scores `margin` (about) below the planted one in
    FP16.  INT8 then ranks the decoy first and FP16 the planted block.
    """
    gen = _gen(device, seed)
    n_rep = Hq // Hkv
    nb = ctx // BLOCK
    s0 = 1.0 / 32.0
    K = outlier_keys(gen, batch, Hkv, ctx, D, device)
    V = _randn(gen, (batch, Hkv, ctx, D), device)
    q = torch.empty(batch, Hq, D, device=device)
    info = []
    for b in range(batch):
        for g in range(Hkv):
            qg = _randn(gen, (D,), device).half().float()
            for r in range(n_rep):
                q[b, g * n_rep + r] = qg
            aq = qg.abs().double()
            sg = torch.sign(qg).double()
            sg[sg == 0] = 1.0
            pb = int(torch.randint(0, max(1, nb // 4), (1,), generator=gen, device=device))
            db = pb
            while db == pb:
                db = int(torch.randint(0, nb, (1,), generator=gen, device=device))
            # needle level: planted FP16 score near 25
            n = int(25.0 * math.sqrt(D) / (s0 * float(aq.sum()))) - 1
            n = max(1, min(n, 120))
            m = torch.full((D,), float(n), dtype=torch.float64, device=device)
            # raise decoy channels (largest |q| first) until its FP16 score is within margin
            gap = s0 * float(aq.sum()) * (7.0 / 16.0) / math.sqrt(D)
            need = (gap - margin) * math.sqrt(D) / s0
            for c in torch.argsort(aq, descending=True).tolist():
                if need <= 0:
                    break
                if float(aq[c]) <= need + 1e-12:
                    m[c] += 1.0
                    need -= float(aq[c])
            planted = sg * (n + 7.0 / 16.0) * s0
            decoy = sg * m * s0
            anchor = -sg * 127.0 * s0
            for blk, needle in ((pb, planted), (db, decoy)):
                rows = _randn(gen, (BLOCK, D), device).clamp(-3.9, 3.9).double()
                rows[0] = anchor
                rows[1 + int(torch.randint(0, BLOCK - 1, (1,), generator=gen, device=device))] = needle
                K[b, g, blk * BLOCK:(blk + 1) * BLOCK] = rows.float()
            info.append((b, g, pb, db))
    return q.half(), K.half(), V.half(), info


def c5_point(ctx: int, batch: int, device="cpu", seed=4, Hq=N_Q_HEADS, Hkv=N_KV_HEADS,
             D=HEAD_DIM, n_out=4, vscale=8.0):
    """Sweep point: keys as c1; values N(0,1) with four channels per KV head scaled x8."""
    gen = _gen(device, seed)
    K = outlier_keys(gen, batch, Hkv, ctx, D, device)
    V = outlier_keys(gen, batch, Hkv, ctx, D, device, n_out=n_out, scale=vscale)
    q = queries(gen, batch, Hq, D, device)
    return q.half(), K.half(), V.half()


def tiny(device="cpu", seed=0, batch=1, ctx=200, Hq=4, Hkv=1, D=HEAD_DIM, kscale=1.0):
    """Small Gaussian case for fast tests (several blocks plus a ragged partial block)."""
    gen = _gen(device, seed)
    K = _randn(gen, (batch, Hkv, ctx, D), device) * kscale
    V = _randn(gen, (batch, Hkv, ctx, D), device)
    q = queries(gen, batch, Hq, D, device)
    return q.half(), K.half(), V.half()
