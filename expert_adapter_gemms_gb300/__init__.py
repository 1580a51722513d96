"""Fused MoE-LoRA expert layer for NVIDIA GB300 (sm_103a).

A C-ABI library (include/moe_lora.h, built from csrc/ into libmoe_lora.so) with a
thin Python binding of the same names. Nothing here computes on the CPU: when
the library is missing, calls raise MoeLoraUnavailable.
"""
from ._lib import (  # noqa: F401
    LAYER_NUM_STAGES,
    LAYER_STAGE_NAMES,
    LIB_PATH,
    MoeLoraError,
    MoeLoraUnavailable,
    lib,
    status_string,
)
from .api import (  # noqa: F401
    Align,
    HostIO,
    align_layout,
    clear_error,
    get_error,
    lora_expand_add,
    lora_shrink,
    moe_gather_rows,
    moe_grouped_gemm,
    moe_lora_align,
    moe_lora_host_io_layout,
    moe_lora_layer,
    moe_lora_layer_host,
    moe_lora_layer_plan,
    moe_lora_layer_tiles,
    moe_lora_workspace_size,
    moe_topk_softmax,
    new_align,
    new_host_io,
    new_workspace,
)
