"""GPU parity of the backward pass (moe_backward) against the fp64 oracle.

The oracle's gradients are taken with the device forward's discrete decisions
(expert_idx, dropped), so the comparison isolates the arithmetic.  Bars:
relative Frobenius error per gradient <= 1e-4 for fp32 layers, <= 2e-2 for bf16
layers (inputs, hidden activations and gradients pass through bf16 several
times); gradients of experts that received no token are exactly zero."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs
from parity_utils import oracle_noise, rel_frobenius, to_cpu

pytestmark = pytest.mark.gpu

TRAIN = _lib.MOE_FLAG_TRAINING
G_TOL = {"bf16": 2e-2, "f32": 1e-4}

CASES = {
    "tiny_fp32_gelu_tanh_bias": config("tiny"),
    "gelu_tanh_bias_ragged": config("tiny", T=257, d=128, E=4, k=2, F=256, dtype="bf16"),
    "gelu_erf_k_eq_E": config("tiny", T=130, d=64, E=3, k=3, F=64, act="gelu_erf", dtype="bf16"),
    "relu_capacity_k1": config("switch", T=1000, d=192, E=16, k=1, F=384, cf=1.0),
    "swiglu_renorm": config("mixtral", T=300, d=256, E=8, k=2, F=512),
    "swiglu_shared": config("deepseek", T=200, d=128, E=16, k=4, F=200),
    "swiglu_shared_fused": config("deepseek", T=260, d=128, E=16, k=3, F=192),  # shared experts in the fused kernel
    "fp32_swiglu_shared": config("deepseek", T=100, d=64, E=8, k=2, F=48, dtype="f32"),
    "ragged_dims": config("mixtral", T=77, d=200, E=5, k=2, F=328),
    "noisy_switch_capacity": config("switch", T=1000, d=256, E=32, k=1, F=384, cf=1.25, noisy=True,
                                    noise_min_std=0.01),
    "noisy_router_split_k": config("skewed", T=64, d=2048, E=64, k=4, F=128, cf=None, noisy=True),
    "many_experts_drops": config("skewed", T=512, d=128, E=256, k=8, F=128),
    "residual_all_tokens": config("switch", T=500, d=128, E=8, k=2, F=256, cf=0.5, residual_mode=1),
}


def _inputs(cfg, seed=0):
    inp = make_inputs(cfg, seed, device="cuda")
    if inp["b1"] is not None:  # non-zero biases so that their gradients are exercised
        g = torch.Generator(device="cuda").manual_seed(seed + 7)
        inp["b1"] = (torch.randn(inp["b1"].shape, generator=g, device="cuda") * 0.5).to(inp["b1"].dtype)
        inp["b2"] = (torch.randn(inp["b2"].shape, generator=g, device="cuda") * 0.5).to(inp["b2"].dtype)
        inp["b_gate"] = torch.randn(cfg.E, generator=g, device="cuda") * 0.1
    return inp


def _dy(cfg, seed=11):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(cfg.T, cfg.d, generator=g, device="cuda").to(cfg.torch_dtype)


def run_backward(cfg, inp, dy, d_aux, flags=0):
    layer = MoELayer(cfg, inp, flags=TRAIN | flags, want_logits=False, want_probs=False)
    layer.run()
    grads = layer.backward(dy, d_aux)
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    return to_cpu(layer.out), to_cpu(grads), layer


def oracle_grads(cfg, inp, out, dy, d_aux):
    cpu = to_cpu(inp)
    return orc.backward(cpu["x"], cpu["W_gate"], cpu["b_gate"], cpu["W1"], cpu["W3"], cpu["W2"], cpu["b1"],
                        cpu["b2"], idx=out["expert_idx"].numpy(), dropped=out["dropped"].numpy(),
                        dy=dy.cpu(), d_aux=d_aux, E=cfg.E, S=cfg.S, act_name=cfg.act,
                        renormalize=cfg.renormalize, residual_mode=cfg.residual_mode,
                        noise=oracle_noise(cfg, cpu))


def compare(cfg, dev, ref, out):
    errs = {}
    for name, r in ref.items():
        if r is None:
            assert dev[name] is None, name
            continue
        d = dev[name].double().numpy()
        errs[name] = rel_frobenius(d, r)
        assert errs[name] <= G_TOL[cfg.dtype], (name, errs[name])
    # experts that received no kept token get exactly zero weight gradients
    kept = np.zeros(cfg.E, dtype=bool)
    idx, drop = out["expert_idx"].numpy(), out["dropped"].numpy().astype(bool)
    kept[np.unique(idx[~drop])] = True
    for name in ("dW1", "dW2", "dW3", "db1", "db2"):
        if dev[name] is not None and (~kept).any():
            assert torch.count_nonzero(dev[name][: cfg.E][torch.from_numpy(~kept)]) == 0, name
    return errs


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name):
    cfg = CASES[name]
    inp = _inputs(cfg)
    dy = _dy(cfg)
    out, grads, _ = run_backward(cfg, inp, dy, 0.37)
    compare(cfg, grads, oracle_grads(cfg, inp, out, dy, 0.37), out)


def test_backward_with_capacity_zero_passes_dy_through():
    # C = 0: every slot dropped, y = x, so dx = dy + the router's share and the experts get nothing
    cfg = config("switch", T=100, d=64, E=128, k=1, F=64, cf=1.0)
    inp = _inputs(cfg)
    dy = _dy(cfg)
    out, grads, _ = run_backward(cfg, inp, dy, 0.5)
    assert out["dropped"].all()
    for name in ("dW1", "dW2"):
        assert torch.count_nonzero(grads[name]) == 0
    compare(cfg, grads, oracle_grads(cfg, inp, out, dy, 0.5), out)


def test_backward_is_deterministic():
    cfg = CASES["swiglu_shared"]
    inp = _inputs(cfg)
    dy = _dy(cfg)
    layer = MoELayer(cfg, inp, flags=TRAIN)
    layer.run()
    g1 = {k: (None if v is None else v.clone()) for k, v in layer.backward(dy, 0.2).items()}
    layer.run()
    g2 = layer.backward(dy, 0.2)
    torch.cuda.synchronize()
    for k, v in g1.items():
        if v is not None:
            assert torch.equal(v, g2[k]), k


def test_backward_needs_the_training_flag():
    cfg = CASES["swiglu_renorm"]
    layer = MoELayer(cfg, _inputs(cfg))
    layer.run()
    with pytest.raises(ValueError):
        layer.backward(_dy(cfg))


def test_aux_gradient_alone_reaches_only_the_router():
    # dy = 0: only d_aux drives the gradients; the experts and the residual get none
    cfg = CASES["swiglu_renorm"]
    inp = _inputs(cfg)
    dy = torch.zeros(cfg.T, cfg.d, dtype=cfg.torch_dtype, device="cuda")
    out, grads, _ = run_backward(cfg, inp, dy, 1.0)
    for name in ("dW1", "dW2", "dW3"):
        assert torch.count_nonzero(grads[name]) == 0
    ref = oracle_grads(cfg, inp, out, dy, 1.0)
    assert rel_frobenius(grads["dW_gate"].double().numpy(), ref["dW_gate"]) <= 1e-3
    assert rel_frobenius(grads["dx"].double().numpy(), ref["dx"]) <= 2e-2


@pytest.mark.parametrize("name", ["relu_capacity_k1", "swiglu_shared", "gelu_tanh_bias_ragged",
                                  "many_experts_drops", "noisy_switch_capacity"])
def test_backward_ffma_experts_match_oracle(name):
    # the CUDA-core cross-check path of the expert backward (bf16 layers)
    cfg = CASES[name]
    inp = _inputs(cfg)
    dy = _dy(cfg)
    layer = MoELayer(cfg, inp, flags=TRAIN | _lib.MOE_FLAG_FFMA_EXPERTS)
    layer.run()
    grads = to_cpu(layer.backward(dy, 0.37))
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    out = to_cpu(layer.out)
    compare(cfg, grads, oracle_grads(cfg, inp, out, dy, 0.37), out)


@pytest.mark.parametrize("name", ["relu_capacity_k1", "swiglu_shared", "gelu_tanh_bias_ragged"])
def test_tensor_core_and_ffma_backward_agree(name):
    cfg = CASES[name]
    inp = _inputs(cfg)
    dy = _dy(cfg)
    _, g_tc, _ = run_backward(cfg, inp, dy, 0.37)
    _, g_ff, _ = run_backward(cfg, inp, dy, 0.37, flags=_lib.MOE_FLAG_FFMA_EXPERTS)
    for k, v in g_tc.items():
        if v is not None:
            assert rel_frobenius(v.double().numpy(), g_ff[k].double().numpy()) <= 1e-2, k


@pytest.mark.parametrize("name", ["noisy_switch_capacity", "swiglu_renorm", "noisy_router_split_k"])
def test_backward_ffma_router_matches_oracle(name):
    # the CUDA-core router gradients (the tensor-core split-term path is the default)
    cfg = CASES[name]
    inp = _inputs(cfg)
    dy = _dy(cfg)
    out, grads, _ = run_backward(cfg, inp, dy, 0.37, flags=_lib.MOE_FLAG_FFMA_ROUTER)
    compare(cfg, grads, oracle_grads(cfg, inp, out, dy, 0.37), out)
