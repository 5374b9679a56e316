"""Dense FP16 decode attention over K/V in device memory (kvq_dense_attention).

This is the dense baseline the certified path is measured against ("Runtime-Certified
Bounded-Error Quantized Attention", gist.science technical summary, Results: performance
overhead against dense FP16 attention; Method §1: dense FP16 attention is the ground
truth).  Its output is compared element by element with oracle.dense_attention (float64)
on ragged lengths (a partial last block, slices of a block with no valid token, a single
token), every GQA width 1-4, several sequences, lengths that split one group's blocks
over many CTAs and lengths where one CTA spans several groups, and at the full 128K
layer of the Llama-3.1-8B shape.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import certified_quantized_kv_gb300 as kvq  # noqa: E402
import oracle as O  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _inputs(B, Hq, Hkv, N, seed, key_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, 128, generator=g).half()
    K = (torch.randn(B, Hkv, N, 128, generator=g) * key_scale).half()
    V = torch.randn(B, Hkv, N, 128, generator=g).half()
    return q, K, V


def _run(q, K, V, workspace=None):
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    ws = kvq.dense_attention(q.cuda(), K.cuda().contiguous(), V.cuda().contiguous(), out, workspace)
    torch.cuda.synchronize()
    return out.cpu().float().numpy(), ws


def _check(out, q, K, V, heads=None):
    qn, Kn, Vn = q.numpy(), K.numpy(), V.numpy()
    B, Hq, _ = qn.shape
    n_rep = Hq // Kn.shape[1]
    worst = 0.0
    for b, h in heads or [(b, h) for b in range(B) for h in range(Hq)]:
        ref = O.dense_attention(qn[b, h], Kn[b, h // n_rep], Vn[b, h // n_rep])
        err = np.abs(out[b, h] - ref)
        assert np.all(np.isfinite(out[b, h])), (b, h)
        if np.max(np.abs(ref)) <= 2.0:
            assert err.max() <= ATOL, (b, h, err.max())
        assert np.all(err <= ATOL + RTOL * np.abs(ref)), (b, h, err.max())
        worst = max(worst, float(err.max()))
    return worst


@pytest.mark.parametrize("B,Hq,Hkv,N", [
    (1, 32, 8, 4096 + 37),     # Llama GQA shape, ragged last block
    (2, 8, 8, 1000),           # n_rep 1 (multi-head attention)
    (3, 6, 2, 64 * 5 + 1),     # n_rep 3, one token in the last block
    (1, 12, 4, 1),             # a single token
    (2, 4, 2, 9),              # n_rep 2, fewer tokens than one warp's slice
    (4, 32, 8, 64 * 40),       # exact blocks; one CTA range spans several groups
    (1, 4, 1, 64 * 1000 + 63), # one group split over every CTA
    (32, 16, 4, 130),          # 128 groups of three blocks: CTA ranges cross many groups
    (64, 8, 2, 100),           # fewer blocks than CTAs: one block per CTA
])
def test_dense_hbm_matches_oracle(B, Hq, Hkv, N):
    q, K, V = _inputs(B, Hq, Hkv, N, seed=B * 1000 + N)
    out, _ = _run(q, K, V)
    worst = _check(out, q, K, V)
    assert worst < ATOL


def test_dense_hbm_peaked_scores_and_reused_workspace():
    """Keys x8 make the softmax peaked (online-softmax rescaling fires inside blocks);
    a second call with the same workspace gives the same bits."""
    q, K, V = _inputs(2, 32, 8, 3000, seed=7, key_scale=8.0)
    out1, ws = _run(q, K, V)
    _check(out1, q, K, V)
    out2, _ = _run(q, K, V, workspace=ws)
    assert np.array_equal(out1, out2)


def test_dense_hbm_full_layer_128k():
    """One full 131072-token layer of the Llama-3.1-8B shape (32 q / 8 KV heads): every
    head against the oracle."""
    q, K, V = _inputs(1, 32, 8, 131072, seed=11)
    out, _ = _run(q, K, V)
    worst = _check(out, q, K, V)
    print(f"128K layer: max-abs error {worst:.2e}")


def test_dense_hbm_max_context():
    """The library's largest context, 2,097,152 tokens, one KV group of four query heads:
    every head against the oracle."""
    q, K, V = _inputs(1, 4, 1, 2097152, seed=13)
    out, _ = _run(q, K, V)
    _check(out, q, K, V)


def test_dense_hbm_argument_checks():
    q, K, V = _inputs(1, 8, 2, 100, seed=1)
    qd, Kd, Vd = q.cuda(), K.cuda(), V.cuda()
    out = torch.empty(1, 8, 128, dtype=torch.float16, device="cuda")
    lib = kvq.load_library()
    need = kvq.dense_attention_workspace(1, 8, 2, 100)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    # workspace too small
    st = lib.kvq_dense_attention(qd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), 1, 8, 2, 100, out.data_ptr(),
                                 ws.data_ptr(), need - 1, None)
    assert st == kvq.KVQ_ERR_INVALID and b"workspace" in lib.kvq_last_error()
    # host buffer
    st = lib.kvq_dense_attention(q.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), 1, 8, 2, 100, out.data_ptr(),
                                 ws.data_ptr(), need, None)
    assert st == kvq.KVQ_ERR_INVALID
    # unaligned key buffer
    st = lib.kvq_dense_attention(qd.data_ptr(), Kd.data_ptr() + 2, Vd.data_ptr(), 1, 8, 2, 99, out.data_ptr(),
                                 ws.data_ptr(), need, None)
    assert st == kvq.KVQ_ERR_INVALID
    # GQA width 5
    st = lib.kvq_dense_attention(qd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), 1, 10, 2, 100, out.data_ptr(),
                                 ws.data_ptr(), need, None)
    assert st == kvq.KVQ_ERR_INVALID
    torch.cuda.synchronize()
