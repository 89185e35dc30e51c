"""Seeded synthetic workloads for the VBQ decode path.

This package draws the inputs only: per-group bit-widths, codes, fp16 scales and
bf16 activations. It does none of the method's arithmetic. The oracle, the tests
and the bench all take their inputs from here, so both sides of every parity
check consume the same arrays.
"""

from .workloads import (  # noqa: F401
    CONFIG0_PROBS,
    GROUP,
    HEAD,
    HEAD_PROBS,
    LAYER0_MLP_PROBS,
    PROJS,
    STRESS_CASES,
    ModelShape,
    VbqMatrixInputs,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    gen_matrix,
    gen_matrix_with_bits,
    gen_model_matrix,
    gen_stress,
    gen_x,
    model_1b,
    model_9b,
    model_matrix_list,
    model_matrix_probs,
    model_matrix_shape,
    model_tiny,
    stress_bits,
)
