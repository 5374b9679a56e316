"""Plain CPU oracle for runtime-certified, bounded-error quantized KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use
it.  It shares no code with the CUDA path.

The method follows "Runtime-Certified Bounded-Error Quantized Attention"
(gist.science technical summary, Japanese and French editions of arXiv 2605.20868):
  * Method §1  tiered storage with deterministic fallback
  * Method §2  two-term error decomposition (E_key, E_val) and the runtime monitor
  * Method §3  adaptive top-K* precision, ranking-consistency check, fallback ladder
  * Contributions, "deterministic recovery"  (return O_dense when the bound fails)

Arithmetic: the quantisation steps use the exact IEEE fp32 / fp16 operations written
out in ``kvq_oracle`` (they fix integer codes and fp16 scales, which the CUDA path
must reproduce bit for bit); everything else is float64.
"""

from .kvq_oracle import (  # noqa: F401
    KAPPA,
    OracleConfig,
    Tier1,
    f16_round_up,
    quantize_key_block,
    dequantize_keys,
    dequantize_values,
    softmax,
    logsumexp,
    MixedResult,
    DecodeResult,
    BLOCK,
    VALUE_GROUP,
    quantize_value_block,
    quantize_layer,
    dense_attention,
    int8_scores,
    block_logsumexp,
    score_perturbation,
    select_top_k_star,
    mixed_attention,
    ranking_consistent,
    plan_ladder,
    decode_layer,
    UncertifiedResult,
    uncertified_decode_layer,
)
