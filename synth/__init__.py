"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and the bench.

This package holds random draws, bf16 rounding of stored values and workload
shapes only. It contains none of the drafter's arithmetic: the oracle and the
CUDA library each compute everything else on their own.
"""
from .generators import (  # noqa: F401
    DrafterShape,
    TINY,
    QWEN3_8B,
    bf16_round,
    bf16_bits,
    bits_to_f32,
    make_weights_np,
    make_selector_weights_np,
    make_conv_weights_np,
    make_weights_torch,
    torch_weights_to_np,
    make_features_np,
    make_anchor_ids_np,
    make_serving_lengths,
    make_verify_case_np,
    make_target_logits_bf16_np,
)
