"""CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library does not.
"""
from .moe_lora_oracle import (  # noqa: F401
    bf16_bits_to_f64, f64_to_bf16_bits, route_topk, permute, silu, expert_slot,
    LoraFactors, moe_lora_forward, factors_from_inputs, forward_inputs,
    expert_slot_general, decode_adapter, moe_lora_forward_general,
    e4m3_to_f64, dequant_fp8_blocks, f64_weights_to_bf16_bits_exact, moe_lora_forward_fp8,
    forward_inputs_fp8,
)
