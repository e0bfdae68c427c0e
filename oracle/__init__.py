"""CPU oracle for the fused MoE-LoRA expert layer (test infrastructure only:
imported by tests, the smoke check and the benchmark's CPU baseline, never by
the library)."""
from .moe_lora_ref import (as_f64, align_ref, moe_lora_forward_ref,  # noqa: F401
                           moe_lora_linear_ref, router_topk_ref, silu)
