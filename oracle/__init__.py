"""fp64 CPU oracle of the fused MoE-LoRA expert layer.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this package. The CUDA library never calls it, shares
no code with it, and must fail loudly rather than fall back to it.
"""
from .moe_lora import (  # noqa: F401
    ERR_ADAPTER_RANGE,
    ERR_EXPERT_RANGE,
    align,
    as_f64,
    combine,
    gather_rows,
    grouped_gemm,
    lora_delta_rows,
    lora_expand_add,
    lora_shrink,
    moe_lora_layer,
    moe_lora_layer_scalar,
    route_topk_softmax,
    silu,
    swiglu,
)
