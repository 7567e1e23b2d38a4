"""The allocation-free dispatch entry point (moe_dispatch_positions_noalloc).

It serves callers that cannot allocate device memory while routing (an engine
that owns all device memory, a path that cannot pay cudaMalloc's implicit
synchronisation).  Its output must equal what the workspace-based entry points
(moe_router + moe_dispatch) produce for the same router selection, and the
fp64 oracle's counts, capacity drops and permutation rows for the same expert
indices, on two calls in a row (the second call reuses the static scratch the
first one left behind).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs, make_params

pytestmark = pytest.mark.gpu


def _reference(cfg):
    inp = make_inputs(cfg, 0, device="cuda")
    layer = MoELayer(cfg, inp, want_perm=True)
    layer.run("moe_router")
    layer.run("moe_dispatch")
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    return layer.out


@pytest.mark.parametrize("cfg", [
    config("switch", T=4096, d=128, E=64, F=128),          # capacity 1.25, drops
    config("deepseek", T=3000, d=128, E=64, k=6, F=128),    # many chunks, no capacity
    config("skewed", T=2048, d=128, E=256, k=8, F=128),     # Zipf-skewed, heavy drops
], ids=["switch_like", "deepseek_like", "skewed_like"])
def test_noalloc_dispatch_matches_workspace_path_twice(cfg):
    ref = _reference(cfg)
    # the oracle's token-order capacity on the same selection (bit-exact bar)
    idx_cpu = ref["expert_idx"].cpu().numpy()
    want = orc.dispatch(idx_cpu, cfg.E, orc.capacity(cfg.T, cfg.E, cfg.cf))
    params = make_params(cfg)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        counts = torch.full((cfg.E,), -7, dtype=torch.int32, device="cuda")
        dropped = torch.full((cfg.T, cfg.k), 9, dtype=torch.uint8, device="cuda")
        perm = torch.full((cfg.T, cfg.k), -7, dtype=torch.int32, device="cuda")
        st = _lib.moe_dispatch_positions_noalloc(params, ref["expert_idx"].data_ptr(),
                                                 counts.data_ptr(), dropped.data_ptr(),
                                                 perm.data_ptr(), stream)
        assert st == _lib.MOE_OK, _lib.moe_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(counts, ref["counts"])
        assert torch.equal(dropped, ref["dropped"])
        assert torch.equal(perm, ref["perm_row"])
        np.testing.assert_array_equal(counts.cpu().numpy(), want.counts)
        np.testing.assert_array_equal(dropped.cpu().numpy(), want.dropped)
        np.testing.assert_array_equal(perm.cpu().numpy(), want.perm_row)


def test_noalloc_dispatch_rejects_oversized_problems():
    cfg = config("deepseek", T=_lib.MOE_NOALLOC_MAX_SLOTS // 6 + 1, d=128, E=64, k=6, F=128)
    params = make_params(cfg)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    st = _lib.moe_dispatch_positions_noalloc(params, p, p, p, p,
                                             torch.cuda.current_stream().cuda_stream)
    assert st == _lib.MOE_ERR_INVALID_ARG
