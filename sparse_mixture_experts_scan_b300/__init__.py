"""B300 (sm_103a) sparse Mixture-of-Experts FFN layer (forward, backward, noisy
gating, 8- and 4-bit expert weights, expert parallelism over emulated ranks): a C-ABI
CUDA library
(libmoe_b300.so, include/moe.h) with a thin Python binding.

    from sparse_mixture_experts_scan_b300 import MoELayer, config, make_inputs
    cfg = config("switch")
    layer = MoELayer(cfg, make_inputs(cfg, device="cuda"))
    out = layer.run()   # y, expert_idx, gates, counts, dropped, aux, perm_row
"""
from ._lib import (moe_backward, moe_combine, moe_dispatch, moe_ep_workspace_size, moe_forward, moe_forward_ep,
                   moe_grouped_gemm, moe_kernel_launches, moe_last_device_status, moe_quantize_int4,
                   moe_quantize_int8, moe_prepare_router_weights, moe_router, moe_router_weights_size,
                   moe_status_string, moe_workspace_size)
from .inputs import CONFIGS, LayerConfig, config, make_inputs
from .layer import (MoEError, MoELayer, check, forward, make_params, quantize_expert_weights, quantize_int4,
                    quantize_int8)

__all__ = [
    "moe_forward", "moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine",
    "moe_workspace_size", "moe_last_device_status", "moe_status_string", "moe_backward",
    "moe_quantize_int8", "moe_quantize_int4", "moe_kernel_launches", "moe_forward_ep", "moe_ep_workspace_size",
    "moe_router_weights_size", "moe_prepare_router_weights",
    "quantize_int8", "quantize_int4", "quantize_expert_weights",
    "CONFIGS", "LayerConfig", "config", "make_inputs", "MoEError", "MoELayer", "check",
    "forward", "make_params",
]
