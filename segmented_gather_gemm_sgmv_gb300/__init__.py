"""GB300-native (sm_103a) segmented gather LoRA apply: SGMV shrink, expand and the fused
shrink->expand, as a C-ABI CUDA library (libsgmv_gb300.so) with a thin Python binding.

    from segmented_gather_gemm_sgmv_gb300 import lora_apply, sgmv_shrink, sgmv_expand
"""
from .binding import (SgmvError, lora_apply, sgmv_expand, sgmv_get_error, sgmv_set_wait_limit,
                      sgmv_shrink, sgmv_validate, sgmv_validate_pointers, sgmv_version,
                      status_string)

__all__ = ["lora_apply", "sgmv_shrink", "sgmv_expand", "sgmv_validate", "sgmv_validate_pointers", "sgmv_get_error",
           "sgmv_set_wait_limit", "sgmv_version", "status_string", "SgmvError"]
