"""GB300 (sm_103a) routed mixture-of-experts expert computation.

The compute path lives in ``libmoe_gb300.so`` (hand-written CUDA, C ABI in
``include/moe_gb300.h``); ``moe`` is its Python binding (argument marshalling only).
"""
from .moe import (  # noqa: F401
    MoEError, MoELayer, moe_plan_weights, moe_prepared_bytes, moe_prepare_weights, moe_unprepare_weights, moe_plan,
    moe_plan_set_swiglu_alpha_beta, moe_plan_set_backend, moe_plan_set_fc1_kernel, moe_plan_set_expert_offset, moe_plan_set_router_weight_on_input, moe_plan_set_debug_copies, moe_plan_set_wait_probe, moe_plan_set_kept_a8,
    moe_scratch_bytes, moe_run, moe_run_chunked, moe_run_static_scratch, moe_io_bytes, moe_run_host,
    moe_get_device_error, moe_get_device_error_static, moe_debug_routing, moe_debug_actq, moe_debug_h, moe_destroy_weight_plan,
    moe_destroy_prepared, moe_destroy_plan, moe_plan_set_profile_events, moe_profile_stage_names, moe_call_launches, moe_status_str,
    moe_version,
    MOE_W4A8_MXFP4, MOE_W4A16_NVFP4, MOE_W4A16_HYBRID, MOE_W4A16_HYBRID_MX, MOE_W4A8_NVFP4, MOE_W4A4_NVFP4, MOE_W13_UP_GATE, MOE_W13_GATE_UP,
    MOE_TIER_NVFP4, MOE_TIER_NF3,
)
