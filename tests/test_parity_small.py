"""GPU parity on small layers the oracle computes in full: every token, every
output element, for each kernel path (tcgen05 and FFMA experts), plus the edge
cases of the method (ragged sizes, k = E, one expert, capacity 0, exact ties,
all tokens on one expert, shared experts, biases, residual modes)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs
from parity_utils import (check_dropped_tokens_pass_x, check_output, check_router_vs_fp64,
                          check_routing_bitexact, run_device, to_cpu)

pytestmark = pytest.mark.gpu

FFMA = _lib.MOE_FLAG_FFMA_EXPERTS


def _case(base, **kw):
    return config(base, **kw)


SMALL = {
    # name: config
    "swiglu_renorm": _case("mixtral", T=300, d=256, E=8, k=2, F=512),
    "relu_capacity": _case("switch", T=1000, d=192, E=16, k=1, F=384, cf=1.0),
    "switch_like_k1": _case("switch", T=2048, d=256, E=32, k=1, F=512, cf=1.25),
    "gelu_tanh_bias": _case("tiny", T=257, d=128, E=4, k=2, F=256, dtype="bf16"),
    "gelu_erf_k_eq_E": _case("tiny", T=130, d=64, E=3, k=3, F=64, act="gelu_erf", dtype="bf16"),
    "shared_experts": _case("deepseek", T=200, d=128, E=16, k=4, F=200),
    # d_ff a multiple of 64: the shared experts run inside the fused expert kernel
    "shared_experts_fused": _case("deepseek", T=333, d=256, E=16, k=3, F=192, S=3),
    "shared_experts_capacity": _case("deepseek", T=400, d=128, E=16, k=2, F=128, cf=0.5),
    "single_expert": _case("mixtral", T=1000, d=128, E=1, k=1, F=256),
    "ragged_dims": _case("mixtral", T=77, d=200, E=5, k=2, F=328),
    "many_experts_drops": _case("skewed", T=512, d=128, E=256, k=8, F=128),
    "max_experts": _case("mixtral", T=256, d=64, E=512, k=4, F=64),
    "one_token": _case("mixtral", T=1, d=64, E=8, k=2, F=64),
    "router_split_k": _case("skewed", T=64, d=2048, E=64, k=4, F=128, cf=None),  # few tokens, long K
    "tiny_fp32": config("tiny"),
    "fp32_swiglu_shared": _case("deepseek", T=100, d=64, E=8, k=2, F=48, dtype="f32"),
}


def _inputs(cfg, seed=0, random_bias=False):
    inp = make_inputs(cfg, seed, device="cuda")
    if random_bias and inp["b1"] is not None:
        g = torch.Generator(device="cuda").manual_seed(seed + 7)
        inp["b1"] = (torch.randn(inp["b1"].shape, generator=g, device="cuda") * 0.5).to(inp["b1"].dtype)
        inp["b2"] = (torch.randn(inp["b2"].shape, generator=g, device="cuda") * 0.5).to(inp["b2"].dtype)
        inp["b_gate"] = torch.randn(cfg.E, generator=g, device="cuda") * 0.1
    return inp


def _full_check(cfg, inp, flags=0, residual_mode=None):
    out = run_device(cfg, inp, flags=flags, residual_mode=residual_mode)
    cpu = to_cpu(inp)
    r = check_routing_bitexact(cfg, out)
    check_router_vs_fp64(cfg, cpu, out)
    err = check_output(cfg, cpu, out, r, residual_mode=residual_mode)
    check_dropped_tokens_pass_x(cfg, cpu, out, residual_mode)
    return out, err


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_layer_matches_oracle(name):
    cfg = SMALL[name]
    _full_check(cfg, _inputs(cfg, random_bias=True))


@pytest.mark.parametrize("name", ["swiglu_renorm", "relu_capacity", "gelu_tanh_bias", "shared_experts",
                                  "ragged_dims"])
def test_small_layer_ffma_experts_match_oracle(name):
    cfg = SMALL[name]
    _full_check(cfg, _inputs(cfg, random_bias=True), flags=FFMA)


def test_worked_example_on_gpu():
    # the 3-expert example embedded in d = F = 8 (extra rows/columns zero): logits
    # [1,2,3], expert outputs 10/20/30 on component 0; y_0 = 25.752..., page 25.8
    cfg = config("tiny", T=1, d=8, E=3, k=3, F=8, act="relu", bias=False)
    x = torch.zeros(1, 8)
    x[0, 0] = 1.0
    Wg = torch.zeros(3, 8)
    Wg[:, 0] = torch.tensor([1.0, 2.0, 3.0])
    W1 = torch.zeros(3, 8, 8)
    W1[:, 0, 0] = 1.0
    W2 = torch.zeros(3, 8, 8)
    W2[:, 0, 0] = torch.tensor([10.0, 20.0, 30.0])
    inp = {"x": x.cuda(), "W_gate": Wg.cuda(), "b_gate": None, "W1": W1.cuda(), "W3": None,
           "W2": W2.cuda(), "b1": None, "b2": None}
    out = run_device(cfg, inp)
    np.testing.assert_allclose(out["logits"][0].numpy(), [1.0, 2.0, 3.0])
    np.testing.assert_array_equal(out["expert_idx"][0].numpy(), [2, 1, 0])
    np.testing.assert_allclose(out["gates"][0].numpy(), [0.66524096, 0.24472847, 0.09003057],
                               atol=1e-6)
    assert round(float(out["y"][0, 0]), 1) == 25.8
    assert abs(float(out["y"][0, 0]) - 25.7521038) < 1e-4
    assert torch.count_nonzero(out["y"][0, 1:]) == 0


def test_capacity_zero_returns_x_exactly():
    cfg = _case("switch", T=64, d=128, E=256, k=2, F=128, cf=1.0)  # C = floor(64/256) = 0
    inp = _inputs(cfg)
    out = run_device(cfg, inp)
    assert out["dropped"].bool().all()
    assert torch.equal(out["y"], inp["x"].cpu())
    check_routing_bitexact(cfg, out)


def test_residual_mode_one_adds_x_everywhere():
    cfg = SMALL["swiglu_renorm"]
    inp = _inputs(cfg)
    _full_check(cfg, inp, residual_mode=1)


def test_exact_logit_ties_pick_lower_expert():
    cfg = _case("mixtral", T=256, d=64, E=8, k=2, F=64)
    inp = _inputs(cfg)
    Wg = inp["W_gate"].clone()
    Wg[5] = Wg[2]  # experts 2 and 5 score identically for every token
    Wg[7] = Wg[0]
    inp["W_gate"] = Wg
    out, _ = _full_check(cfg, inp)
    idx = out["expert_idx"].numpy()
    # equal logits: whenever expert 5 (7) is selected, expert 2 (0) is selected too
    for t in range(cfg.T):
        row = set(idx[t].tolist())
        assert not ({5} <= row and 2 not in row), idx[t]
        assert not ({7} <= row and 0 not in row), idx[t]


def test_all_tokens_on_one_expert():
    cfg = _case("mixtral", T=700, d=128, E=8, k=1, F=256, renormalize=False)
    inp = _inputs(cfg)
    bg = torch.zeros(cfg.E, device="cuda")
    bg[3] = 60.0
    inp["b_gate"] = bg
    out, _ = _full_check(cfg, inp)
    assert (out["expert_idx"] == 3).all()
    assert out["counts"][3] == cfg.T


def test_stage_entry_points_equal_forward():
    cfg = SMALL["shared_experts"]
    inp = _inputs(cfg)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp, stages=["moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine"])
    for k in ("y", "expert_idx", "gates", "counts", "dropped", "aux", "perm_row", "logits"):
        assert torch.equal(a[k], b[k]), k


def test_repeated_calls_are_deterministic():
    cfg = SMALL["relu_capacity"]
    inp = _inputs(cfg)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp)
    for k in ("y", "gates", "aux", "probs", "perm_row"):
        assert torch.equal(a[k], b[k]), k


def test_tcgen05_and_ffma_experts_agree():
    cfg = _case("mixtral", T=2048, d=512, E=8, k=2, F=1024)
    inp = _inputs(cfg)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp, flags=FFMA)
    ya, yb = a["y"].double(), b["y"].double()
    assert float((ya - yb).norm() / yb.norm()) < 1e-2


@pytest.mark.parametrize("name", ["switch_like_k1", "max_experts", "ragged_dims", "many_experts_drops",
                                  "gelu_erf_k_eq_E", "router_split_k"])
def test_ffma_router_matches_oracle_and_tensor_core_router(name):
    # bf16 layers compute router logits on the tensor core (three-term bf16 split of
    # W_gate); the CUDA-core FFMA router is the cross-check.  Both must route
    # bit-exactly on their own logits and agree with the fp64 oracle.
    cfg = SMALL[name]
    inp = _inputs(cfg, random_bias=True)
    cpu = to_cpu(inp)
    tc = run_device(cfg, inp)
    ff = run_device(cfg, inp, flags=_lib.MOE_FLAG_FFMA_ROUTER)
    for out in (tc, ff):
        check_routing_bitexact(cfg, out)
        check_router_vs_fp64(cfg, cpu, out)
    scale = max(1.0, float(ff["logits"].abs().max()))
    assert float((tc["logits"] - ff["logits"]).abs().max()) <= 2e-5 * scale


@pytest.mark.parametrize("name", ["swiglu_renorm", "relu_capacity", "switch_like_k1", "gelu_tanh_bias",
                                  "shared_experts", "shared_experts_fused", "shared_experts_capacity",
                                  "ragged_dims", "many_experts_drops", "max_experts", "single_expert"])
def test_fused_and_two_launch_experts_agree_bitwise(name):
    # The fused persistent kernel (dynamic tiles, GEMM2 tiles waiting on GEMM1 tiles)
    # and the two grouped-GEMM launches accumulate every output element in the same
    # order, so their outputs must be identical bit for bit.
    cfg = SMALL[name]
    inp = _inputs(cfg, random_bias=True)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp, flags=_lib.MOE_FLAG_UNFUSED_EXPERTS)
    assert torch.equal(a["y"], b["y"])
    for _ in range(3):  # the scheduler counters re-arm themselves between launches
        c = run_device(cfg, inp)
        assert torch.equal(a["y"], c["y"])


def test_nan_tokens_route_to_valid_experts():
    # Non-finite inputs must never produce an expert index outside [0, E): NaN logits
    # compete as -inf in the selection (so an all-NaN row takes experts 0, 1, ...,
    # as the oracle's selection on the same logits does), and the finite tokens are
    # unaffected.
    cfg = _case("mixtral", T=300, d=128, E=8, k=2, F=128, cf=1.0)
    inp = _inputs(cfg)
    x = inp["x"].clone()
    bad = torch.tensor([0, 7, 150, 299], device="cuda")
    x[bad] = float("nan")
    inp["x"] = x
    out = run_device(cfg, inp)
    idx = out["expert_idx"]
    assert int(idx.min()) >= 0 and int(idx.max()) < cfg.E
    check_routing_bitexact(cfg, out)
    good = np.setdiff1d(np.arange(cfg.T), bad.cpu().numpy())
    r = orc.route_from_logits(out["logits"].numpy(), k=cfg.k, renormalize=cfg.renormalize, cf=cfg.cf)
    from parity_utils import check_output
    check_output(cfg, to_cpu(inp), out, r, tokens=good)


# ---------------------------------------------------------------- noisy top-k gating

NOISY = {
    "noisy_switch_k1": _case("switch", T=1000, d=256, E=32, k=1, F=384, cf=1.25, noisy=True,
                             noise_min_std=0.01),
    "noisy_top2_renorm": _case("mixtral", T=300, d=256, E=8, k=2, F=512, noisy=True),
    "noisy_router_split_k": _case("skewed", T=64, d=2048, E=64, k=4, F=128, cf=None, noisy=True),
    "noisy_many_experts_drops": _case("skewed", T=512, d=128, E=256, k=8, F=128, noisy=True),
    "noisy_max_experts": _case("mixtral", T=256, d=64, E=512, k=4, F=64, noisy=True),
    "noisy_fp32": config("tiny", noisy=True, noise_min_std=0.01),
}
_NOISE_KEYS = ("W_noise", "b_noise", "noise_eps")


@pytest.mark.parametrize("name", sorted(NOISY))
def test_noisy_gating_matches_oracle(name):
    cfg = NOISY[name]
    _full_check(cfg, _inputs(cfg, random_bias=True))


@pytest.mark.parametrize("name", ["noisy_switch_k1", "noisy_router_split_k", "noisy_max_experts"])
def test_noisy_gating_ffma_router_matches_oracle(name):
    cfg = NOISY[name]
    _full_check(cfg, _inputs(cfg), flags=_lib.MOE_FLAG_FFMA_ROUTER)


@pytest.mark.parametrize("name", ["noisy_switch_k1", "noisy_router_split_k", "noisy_fp32"])
def test_noisy_gating_with_zero_draws_equals_clean_bitwise(name):
    # eps = 0: the noisy logits are the clean ones exactly (x + 0 * s = x), so every
    # output equals the run without noisy gating bit for bit
    cfg = NOISY[name]
    inp = _inputs(cfg)
    inp["noise_eps"] = torch.zeros_like(inp["noise_eps"])
    noisy = run_device(cfg, inp)
    clean_cfg = replace(cfg, noisy=False)
    clean = run_device(clean_cfg, {k: v for k, v in inp.items() if k not in _NOISE_KEYS})
    for key in ("logits", "probs", "expert_idx", "gates", "counts", "dropped", "aux", "perm_row", "y"):
        assert torch.equal(noisy[key], clean[key]), key


def test_noisy_gating_moves_the_selection():
    # with unit normal draws a sizeable share of top-1 choices moves, and only where the
    # oracle's noisy logits say so (checked in full by the parity test above)
    cfg = NOISY["noisy_switch_k1"]
    inp = _inputs(cfg)
    noisy = run_device(cfg, inp)
    clean_cfg = replace(cfg, noisy=False)
    clean = run_device(clean_cfg, {k: v for k, v in inp.items() if k not in _NOISE_KEYS})
    moved = (noisy["expert_idx"] != clean["expert_idx"]).any(dim=1).float().mean().item()
    assert 0.05 < moved < 1.0, moved


@pytest.mark.parametrize("name", ["swiglu_renorm", "gelu_tanh_bias", "shared_experts", "relu_capacity"])
def test_training_flag_leaves_forward_outputs_unchanged(name):
    # MOE_FLAG_TRAINING only adds stores (logits, pre-activations): every output is bit-identical
    cfg = SMALL[name]
    inp = _inputs(cfg, random_bias=True)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp, flags=_lib.MOE_FLAG_TRAINING)
    for key, v in a.items():
        if v is not None:
            assert torch.equal(v, b[key]), key


def test_stage_entry_points_equal_forward_with_noise_and_int8():
    from sparse_mixture_experts_scan_b300 import quantize_expert_weights
    for cfg, quant in ((NOISY["noisy_top2_renorm"], False),
                       (config("mixtral", T=300, d=256, E=8, k=2, F=512, weights="int8"), True)):
        inp = _inputs(cfg)
        if quant:
            inp = quantize_expert_weights(inp)
        a = run_device(cfg, inp)
        b = run_device(cfg, inp, stages=["moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine"])
        for key, v in a.items():
            if v is not None:
                assert torch.equal(v, b[key]), key


def test_empty_batch_forward_and_backward():
    # T = 0: no kernel; counts and aux are zero, gradients are zero
    cfg = config("mixtral", T=0, d=64, E=8, k=2, F=64)
    inp = make_inputs(config("mixtral", T=1, d=64, E=8, k=2, F=64), 0, device="cuda")
    inp["x"] = inp["x"][:0]
    layer = MoELayer(cfg, inp, flags=_lib.MOE_FLAG_TRAINING)
    layer.out["counts"].fill_(7)
    layer.out["aux"].fill_(7.0)
    n0 = _lib.moe_kernel_launches()
    layer.run()
    grads = layer.backward(torch.zeros(0, cfg.d, dtype=cfg.torch_dtype, device="cuda"), 0.5)
    torch.cuda.synchronize()
    assert _lib.moe_kernel_launches() == n0
    assert layer.device_status() == _lib.MOE_OK
    assert int(layer.out["counts"].abs().sum()) == 0 and float(layer.out["aux"][0]) == 0.0
    for k, v in grads.items():
        if v is not None:
            assert int(torch.count_nonzero(v)) == 0, k


def test_maximum_top_k():
    # k = MOE_MAX_TOPK = 32 of E = 64 (and of E = 512) experts
    for cfg in (config("mixtral", T=200, d=64, E=64, k=32, F=64),
                config("mixtral", T=100, d=64, E=512, k=32, F=64, cf=1.0)):
        _full_check(cfg, _inputs(cfg))


def test_layers_of_growing_size_in_one_process():
    # kernels whose dynamic shared memory depends on the layer (router for few experts,
    # dispatch scan) raise their limit when a later layer needs more
    for cfg in (config("mixtral", T=64, d=64, E=8, k=2, F=64), config("mixtral", T=64, d=4096, E=8, k=2, F=64),
                config("skewed", T=64, d=64, E=64, k=4, F=64), config("skewed", T=64, d=64, E=512, k=4, F=64)):
        _full_check(cfg, _inputs(cfg))


def _random_config(seed):
    rng = np.random.default_rng(1000 + seed)
    act = ["relu", "gelu_tanh", "swiglu", "gelu_erf", "swiglu", "swiglu"][seed % 6]
    E = [1, 3, 8, 16, 31, 64, 100, 300, 24, 130, 7, 48][seed % 12]
    k = int(rng.integers(1, min(E, 8) + 1))
    S = int(rng.integers(1, 3)) if act == "swiglu" and seed % 2 == 0 else 0
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    cf = None if rng.random() < 0.4 else float(rng.choice([0.5, 1.0, 1.25, 2.0]))
    return config("mixtral", T=int(rng.integers(1, 700)), d=8 * int(rng.integers(1, 48)),
                  F=8 * int(rng.integers(1, 64)), E=E, k=k, S=S, act=act, dtype=dtype, cf=cf,
                  renormalize=bool(rng.integers(2)), bias=act != "swiglu" and bool(rng.integers(2)),
                  residual_mode=int(rng.integers(2)), noisy=bool(rng.random() < 0.25),
                  noise_min_std=0.01)


@pytest.mark.parametrize("seed", range(12))
def test_random_layers_match_oracle(seed):
    # seeded random shapes and options: every combination of router tile width, K split,
    # fused top-k, combine segmentation and expert path that the heuristics can pick
    cfg = _random_config(seed)
    out, _ = _full_check(cfg, _inputs(cfg, seed=seed, random_bias=True), residual_mode=cfg.residual_mode)
    assert out["expert_idx"].shape == (cfg.T, cfg.k)


def test_expired_device_wait_is_reported_and_the_context_stays_usable():
    # a bounded wait that runs out (a barrier nothing arrives at, 20 ms) sets the
    # workspace's error word; moe_last_device_status reports it once, then the layer runs
    cfg = SMALL["swiglu_renorm"]
    inp = _inputs(cfg)
    layer = MoELayer(cfg, inp, want_logits=True, want_probs=True)
    st = torch.cuda.current_stream().cuda_stream
    assert _lib.moe_check_bounded_wait(layer.workspace.data_ptr(), layer.workspace_bytes, 20000, st) == _lib.MOE_OK
    assert layer.device_status() == _lib.MOE_ERR_DEVICE_TIMEOUT
    assert layer.device_status() == _lib.MOE_OK  # read and cleared
    layer.run()
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    out = to_cpu(layer.out)
    r = check_routing_bitexact(cfg, out)
    check_output(cfg, to_cpu(inp), out, r)


@pytest.mark.parametrize("name", ["switch_like_k1", "swiglu_renorm", "max_experts", "router_split_k",
                                  "many_experts_drops"])
def test_prepared_router_weights_give_identical_outputs(name):
    # The router weights split once (moe_prepare_router_weights) are the same bits the
    # per-call split writes into the workspace, so every output is identical.
    cfg = SMALL[name]
    inp = _inputs(cfg, random_bias=True)
    a = MoELayer(cfg, inp, want_logits=True, want_probs=True)
    b = MoELayer(cfg, inp, want_logits=True, want_probs=True, prepared_router=True)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert b.device_status() == _lib.MOE_OK
    for k in ("y", "logits", "probs", "expert_idx", "gates", "counts", "dropped", "aux", "perm_row"):
        assert torch.equal(a.out[k], b.out[k]), k
    # the prepared buffer does not depend on the batch size: reuse it for a smaller, ragged batch
    t2 = min(77, cfg.T - 5)
    small = replace(cfg, T=t2)
    sinp = dict(inp)
    sinp["x"] = inp["x"][:t2].contiguous()
    c = MoELayer(small, sinp, want_logits=True)
    d = MoELayer(small, sinp, want_logits=True)
    d.inputs.router_weights = b.router_weights.data_ptr()
    c.run()
    d.run()
    torch.cuda.synchronize()
    for k in ("y", "logits", "expert_idx", "gates", "aux"):
        assert torch.equal(c.out[k], d.out[k]), k


def test_prepared_router_weights_with_noisy_gating():
    cfg = _case("mixtral", T=300, d=128, E=24, k=3, F=128, noisy=True, noise_min_std=0.01)
    inp = _inputs(cfg)
    a = MoELayer(cfg, inp, want_logits=True)
    b = MoELayer(cfg, inp, want_logits=True, prepared_router=True)
    a.run()
    b.run()
    torch.cuda.synchronize()
    for k in ("y", "logits", "expert_idx", "gates", "aux"):
        assert torch.equal(a.out[k], b.out[k]), k


def test_top1_stage_entry_points_equal_forward():
    # top-1 layers finish the combine inside the expert stage (its GEMM2 epilogue writes y,
    # the dispatch copies dropped tokens): the stage calls still compose to the forward
    cfg = SMALL["switch_like_k1"]
    inp = _inputs(cfg)
    a = run_device(cfg, inp)
    b = run_device(cfg, inp, stages=["moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine"])
    for k in ("y", "expert_idx", "gates", "counts", "dropped", "aux", "perm_row", "logits"):
        assert torch.equal(a[k], b[k]), k
    assert int(a["dropped"].sum()) > 0  # the case has dropped tokens (y = x for them)
