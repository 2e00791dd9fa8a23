"""GB300-native (sm_103a) segmented gather LoRA apply: SGMV shrink, expand and the fused
shrink->expand, as a C-ABI CUDA library (libsgmv_gb300.so) with a thin Python binding.

    from segmented_gather_gemm_sgmv_gb300 import lora_apply, sgmv_shrink, sgmv_expand
"""
from .binding import (AdapterPool, Plan, SgmvError, lora_apply, lora_apply_multi, lora_apply_planned,
                      lora_apply_base, lora_apply_ranked, lora_apply_static_plan,
                      sgmv_expand, sgmv_expand_planned, sgmv_get_error, sgmv_plan,
                      sgmv_plan_size, sgmv_set_wait_limit, sgmv_shrink, sgmv_shrink_planned,
                      sgmv_validate, sgmv_validate_pointers, sgmv_version, status_string)

__all__ = ["lora_apply", "sgmv_shrink", "sgmv_expand", "sgmv_plan", "sgmv_plan_size",
           "lora_apply_planned", "sgmv_shrink_planned", "sgmv_expand_planned",
           "lora_apply_multi", "lora_apply_ranked", "lora_apply_base", "lora_apply_static_plan", "AdapterPool", "Plan", "sgmv_validate", "sgmv_validate_pointers",
           "sgmv_get_error", "sgmv_set_wait_limit", "sgmv_version", "status_string", "SgmvError"]
