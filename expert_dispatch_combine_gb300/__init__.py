"""GB300 (sm_103a) decode-time MoE layer: gate top-k routing, INT8 FusedDispatch
into static per-rank buffers, grouped W8A8 SwiGLU experts, EPLB replica map,
FusedCombine -- a C-ABI CUDA library (include/moe.h) with a thin ctypes binding.

    from expert_dispatch_combine_gb300 import binding, layer, synth
"""
from .binding import (MOE_MSG_BF16, MOE_MSG_INT8, MoeError, Shape, load, moe_combine,  # noqa: F401
                      moe_dispatch, moe_eplb_plan, moe_expert_ffn, moe_gemm_workspace_bytes,
                      moe_grouped_gemm_s8, moe_layer, moe_query_layout, moe_route,
                      moe_static_buffer_bytes, moe_status_string)

__all__ = ["Shape", "MoeError", "load", "moe_route", "moe_dispatch", "moe_expert_ffn",
           "moe_combine", "moe_layer", "moe_query_layout", "moe_static_buffer_bytes",
           "moe_eplb_plan", "moe_grouped_gemm_s8", "moe_gemm_workspace_bytes",
           "moe_status_string", "MOE_MSG_BF16", "MOE_MSG_INT8"]
