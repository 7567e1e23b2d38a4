"""B300 (sm_103a) sparse Mixture-of-Experts FFN forward: a C-ABI CUDA library
(libmoe_b300.so, include/moe.h) with a thin Python binding.

    from sparse_mixture_experts_scan_b300 import MoELayer, config, make_inputs
    cfg = config("switch")
    layer = MoELayer(cfg, make_inputs(cfg, device="cuda"))
    out = layer.run()   # y, expert_idx, gates, counts, dropped, aux, perm_row
"""
from ._lib import (moe_combine, moe_dispatch, moe_forward, moe_grouped_gemm, moe_last_device_status,
                   moe_router, moe_status_string, moe_workspace_size)
from .inputs import CONFIGS, LayerConfig, config, make_inputs
from .layer import MoEError, MoELayer, check, forward, make_params

__all__ = [
    "moe_forward", "moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine",
    "moe_workspace_size", "moe_last_device_status", "moe_status_string",
    "CONFIGS", "LayerConfig", "config", "make_inputs", "MoEError", "MoELayer", "check",
    "forward", "make_params",
]
