"""CPU oracle for the quantised-base LoRA linear (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The library's compute path never imports it, and it shares no code,
tables or constants with the CUDA sources.
"""
from .qlora_oracle import (  # noqa: F401
    NF4_LEVELS,
    bf16_bits_to_f64,
    bf16_round_f32,
    dequant,
    dequant_bf16_bits,
    e2m1_value,
    e4m3_value,
    q4_k_scale_min,
    linear_fwd,
    linear_bwd,
    linear_fwd_rows,
    linear_bwd_rows,
    linear_bwd_adapter_grads,
    grouped_fwd,
    grouped_bwd,
    multi_linear_fwd,
    multi_linear_bwd,
    stacked_linear_fwd,
    stacked_linear_bwd,
    swiglu_fwd,
    swiglu_bwd,
    swiglu_grad_gate_up,
)
