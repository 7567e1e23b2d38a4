"""GPU parity of 4-bit expert weights (MOE_WEIGHTS_INT4) and of the tensor-memory
quantised-weight kernel that serves them.

moe_quantize_int4 is compared bit for bit (packed values and group scales) with the
oracle's quantisation, which takes the rounding decision in the same IEEE fp32
arithmetic.  The 4-bit layer is compared with the fp64 oracle run on the exactly
dequantised weights q * scale: routing bit-exact (the router is untouched), the
output within the bf16 bar (relative Frobenius <= 2e-2; the kernel rounds each
dequantised weight once to bf16), dropped tokens equal to x."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from parity_utils import (check_dropped_tokens_pass_x, check_router_vs_fp64, check_routing_bitexact,
                          quantized_oracle_rows, rel_frobenius, sample_tokens, to_cpu)
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs, quantize_expert_weights, quantize_int4

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_int4_matches_oracle_bitwise(dtype):
    g = torch.Generator(device="cuda").manual_seed(4)
    w = torch.randn(300, 512, generator=g, device="cuda") * torch.rand(300, 1, generator=g, device="cuda") * 3
    w[7] = 0.0                                 # all-zero row
    w[9, 128:256] = 0.0                        # one all-zero group
    w[11, 5] = 1e4                             # one large element dominates a group
    w[13, :128] = torch.linspace(-3.5, 3.5, 128, device="cuda")  # amax 3.5: scale 0.5, ties at quarter steps
    w = w.to(dtype)
    q, s = quantize_int4(w)
    torch.cuda.synchronize()
    q_ref, s_ref = orc.quantize_int4(w.cpu())
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


SMALL = {
    "relu_capacity": config("switch", T=1000, d=256, E=16, k=1, F=384, cf=1.0, weights="int4"),
    "switch_like": config("switch", T=2048, d=256, E=32, k=1, F=512, cf=1.25, weights="int4"),
    "swiglu_many_tokens": config("mixtral", T=700, d=256, E=8, k=2, F=512, weights="int4"),   # several token tiles
    "gelu_tanh_bias": config("tiny", T=257, d=128, E=4, k=2, F=256, dtype="bf16", weights="int4"),
    "ragged_tiles": config("mixtral", T=77, d=384, E=5, k=2, F=640, weights="int4"),         # partial 128-row tiles
    "many_experts_drops": config("skewed", T=512, d=128, E=256, k=8, F=128, weights="int4"),
    "one_token": config("mixtral", T=1, d=128, E=8, k=2, F=128, weights="int4"),
}


def _run(cfg, seed=0):
    inp = make_inputs(cfg, seed, device="cuda")
    if inp["b1"] is not None:
        g = torch.Generator(device="cuda").manual_seed(seed + 7)
        inp["b1"] = (torch.randn(inp["b1"].shape, generator=g, device="cuda") * 0.5).to(inp["b1"].dtype)
        inp["b2"] = (torch.randn(inp["b2"].shape, generator=g, device="cuda") * 0.5).to(inp["b2"].dtype)
    qinp = quantize_expert_weights(inp, bits=4)
    layer = MoELayer(cfg, qinp, want_logits=True, want_probs=True)
    layer.run()
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    return to_cpu(inp), to_cpu(qinp), to_cpu(layer.out)


def _dequantize(q, scale):
    return orc.dequantize_int4(q, scale)


def _check(cfg, inp, qinp, out, tokens=None):
    r = check_routing_bitexact(cfg, out)
    check_router_vs_fp64(cfg, inp, out)
    tok = np.arange(cfg.T) if tokens is None else tokens
    y_ref = quantized_oracle_rows(cfg, inp, qinp, r, tok, _dequantize)
    err = rel_frobenius(out["y"][torch.as_tensor(tok)].double().numpy(), y_ref)
    assert err <= 2e-2, err
    check_dropped_tokens_pass_x(cfg, inp, out)
    return err


@pytest.mark.parametrize("name", sorted(SMALL))
def test_int4_layer_matches_oracle(name):
    cfg = SMALL[name]
    _check(cfg, *_run(cfg))


@pytest.mark.parametrize("name", ["switch", "skewed", "decode_nocap"])
def test_int4_full_size(name):
    cfg = config(name, weights="int4")
    inp, qinp, out = _run(cfg)
    _check(cfg, inp, qinp, out, sample_tokens(cfg, out, 128))


def test_int4_rejects_unsupported_shapes():
    cfg = config("mixtral", T=64, d=192, E=8, k=2, F=256, weights="int4")  # d not a multiple of 128
    from sparse_mixture_experts_scan_b300 import make_params
    assert _lib.moe_workspace_size(make_params(cfg))[0] == _lib.MOE_ERR_UNSUPPORTED
