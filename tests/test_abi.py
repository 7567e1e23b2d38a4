"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import pytest

from sparse_mixture_experts_scan_b300 import _lib, config, make_params


def test_library_exports_every_header_function():
    names = _lib.header_functions()
    assert set(names) == {"moe_workspace_size", "moe_forward", "moe_router", "moe_dispatch",
                          "moe_grouped_gemm", "moe_combine", "moe_last_device_status",
                          "moe_status_string", "moe_dispatch_positions_noalloc",
                          "moe_kernel_launches", "moe_backward", "moe_quantize_int8",
                          "moe_check_bounded_wait", "moe_ep_workspace_size", "moe_forward_ep",
                          "moe_quantize_int4", "moe_router_weights_size", "moe_prepare_router_weights"}
    L = _lib.load()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (2, "MOE_ERR_UNSUPPORTED"),
                       (3, "MOE_ERR_WORKSPACE"), (4, "MOE_ERR_CUDA"), (5, "MOE_ERR_DEVICE_TIMEOUT")]:
        assert _lib.moe_status_string(code) == name


def test_struct_layouts_match_header():
    # moe_params_t: 11 int32/float fields, uint32 flags, noisy_gating, noise_min_std, weight_format
    assert ctypes.sizeof(_lib.moe_params_t) == 15 * 4
    assert ctypes.sizeof(_lib.moe_inputs_t) == 15 * 8
    assert ctypes.sizeof(_lib.moe_outputs_t) == 9 * 8


@pytest.mark.parametrize("name", ["tiny", "switch", "mixtral", "deepseek", "skewed", "decode"])
def test_workspace_size_of_configs(name):
    cfg = config(name)
    st, n = _lib.moe_workspace_size(make_params(cfg))
    assert st == _lib.MOE_OK and n > 0
    # the permuted activations alone need at least the kept rows of x (bf16 / fp32)
    esz = 2 if cfg.dtype == "bf16" else 4
    assert n >= min(cfg.T * cfg.k, cfg.T * cfg.k) * cfg.d * esz or cfg.cf is not None


def test_workspace_grows_with_tokens():
    cfg = config("switch")
    sizes = [_lib.moe_workspace_size(make_params(cfg, T=t))[1] for t in (128, 1024, 8192, 65536)]
    assert sizes == sorted(sizes) and len(set(sizes)) == 4


@pytest.mark.parametrize("field,value", [
    ("k", 0), ("k", 9), ("E", 0), ("E", 513), ("d_model", 12), ("d_ff", 20), ("T", -1),
    ("renormalize", 2), ("residual_mode", 5), ("act", 7), ("dtype", 3), ("flags", 16),
    ("n_shared", -1)])
def test_invalid_params_rejected(field, value):
    p = make_params(config("mixtral"))
    setattr(p, field, value)
    st, _ = _lib.moe_workspace_size(p)
    assert st == _lib.MOE_ERR_INVALID_ARG


def test_k_above_topk_limit_rejected():
    p = make_params(config("skewed"))
    p.k = 33
    assert _lib.moe_workspace_size(p)[0] == _lib.MOE_ERR_INVALID_ARG


def test_shared_experts_need_swiglu():
    p = make_params(config("switch"))
    p.n_shared = 1
    assert _lib.moe_workspace_size(p)[0] == _lib.MOE_ERR_UNSUPPORTED


def test_nan_capacity_rejected():
    p = make_params(config("switch"))
    p.capacity_factor = float("nan")
    assert _lib.moe_workspace_size(p)[0] == _lib.MOE_ERR_INVALID_ARG


def _fake_io(cfg, aligned=True):
    """Structs filled with fake (never dereferenced) 256-byte aligned addresses."""
    base = 1 << 40
    a = lambda i: base + i * (1 << 30) + (0 if aligned else 4)  # noqa: E731
    ins = _lib.moe_inputs_t(x=a(0), W_gate=a(1), b_gate=None, W1=a(2),
                            W3=a(3) if cfg.act == "swiglu" else None, W2=a(4))
    outs = _lib.moe_outputs_t(y=a(5), expert_idx=a(6), gates=a(7), counts=a(8), dropped=a(9),
                              aux=a(10))
    return ins, outs


@pytest.mark.parametrize("stage", _lib.STAGES)
def test_host_validation_happens_before_any_launch(stage):
    cfg = config("mixtral")
    p = make_params(cfg)
    ins, outs = _fake_io(cfg)
    _, need = _lib.moe_workspace_size(p)
    ws = 1 << 44
    fn = getattr(_lib, stage)
    bad = make_params(cfg)
    bad.k = 0
    assert fn(bad, ins, outs, ws, need, None) == _lib.MOE_ERR_INVALID_ARG
    # workspace missing, too small, unaligned
    assert fn(p, ins, outs, None, need, None) == _lib.MOE_ERR_WORKSPACE
    assert fn(p, ins, outs, ws, need - 1, None) == _lib.MOE_ERR_WORKSPACE
    assert fn(p, ins, outs, ws + 16, need, None) == _lib.MOE_ERR_WORKSPACE
    # required pointers
    ins2, outs2 = _fake_io(cfg)
    ins2.W3 = None  # SwiGLU needs W3
    assert fn(p, ins2, outs2, ws, need, None) == _lib.MOE_ERR_INVALID_ARG
    ins3, outs3 = _fake_io(cfg)
    outs3.aux = None
    assert fn(p, ins3, outs3, ws, need, None) == _lib.MOE_ERR_INVALID_ARG
    ins4, outs4 = _fake_io(cfg, aligned=False)
    assert fn(p, ins4, outs4, ws, need, None) == _lib.MOE_ERR_INVALID_ARG


def test_relu_layer_rejects_w3_and_swiglu_rejects_biases():
    cfg = config("switch")
    p = make_params(cfg)
    ins, outs = _fake_io(cfg)
    ins.W3 = ins.W1
    _, need = _lib.moe_workspace_size(p)
    assert _lib.moe_forward(p, ins, outs, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG
    cfg2 = config("mixtral")
    p2 = make_params(cfg2)
    ins2, outs2 = _fake_io(cfg2)
    ins2.b1 = ins2.W1
    _, need2 = _lib.moe_workspace_size(p2)
    assert _lib.moe_forward(p2, ins2, outs2, 1 << 44, need2, None) == _lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("noisy_gating", 2), ("noisy_gating", -1),
                                         ("noise_min_std", -0.5), ("noise_min_std", float("nan")),
                                         ("noise_min_std", float("inf"))])
def test_invalid_noise_params_rejected(field, value):
    p = make_params(config("switch", noisy=True))
    setattr(p, field, value)
    assert _lib.moe_workspace_size(p)[0] == _lib.MOE_ERR_INVALID_ARG


def test_noisy_gating_needs_more_workspace():
    for name in ("switch", "tiny", "router_split"):
        cfg = config("skewed", T=64, d=2048, E=64, k=4, cf=None) if name == "router_split" else config(name)
        st0, n0 = _lib.moe_workspace_size(make_params(cfg))
        st1, n1 = _lib.moe_workspace_size(make_params(cfg.__class__(**{**cfg.__dict__, "noisy": True})))
        assert st0 == st1 == _lib.MOE_OK
        assert n1 >= n0 + 4 * cfg.T * cfg.E  # at least the [T, E] noise logits


def test_noise_pointers_must_match_the_mode():
    base = 1 << 40
    for noisy in (False, True):
        cfg = config("switch", noisy=noisy)
        p = make_params(cfg)
        _, need = _lib.moe_workspace_size(p)
        cases = []
        if noisy:
            for missing in ("W_noise", "noise_eps"):
                ins, outs = _fake_io(cfg)
                ins.W_noise, ins.noise_eps = base + 20 * (1 << 30), base + 21 * (1 << 30)
                setattr(ins, missing, None)
                cases.append((ins, outs))
            ins, outs = _fake_io(cfg)
            ins.W_noise, ins.noise_eps = base + 20 * (1 << 30) + 4, base + 21 * (1 << 30)  # unaligned
            cases.append((ins, outs))
        else:
            for extra in ("W_noise", "b_noise", "noise_eps"):
                ins, outs = _fake_io(cfg)
                setattr(ins, extra, base + 22 * (1 << 30))
                cases.append((ins, outs))
        for ins, outs in cases:
            for stage in ("moe_forward", "moe_router"):
                assert getattr(_lib, stage)(p, ins, outs, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG


def test_launch_counter_does_not_move_on_rejected_calls():
    n0 = _lib.moe_kernel_launches()
    cfg = config("mixtral")
    p = make_params(cfg)
    p.k = 0
    ins, outs = _fake_io(cfg)
    assert _lib.moe_forward(p, ins, outs, 1 << 44, 1 << 30, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_kernel_launches() == n0


def test_training_flag_reserves_backward_buffers():
    for name in ("switch", "mixtral", "deepseek", "tiny"):
        cfg = config(name)
        n0 = _lib.moe_workspace_size(make_params(cfg))[1]
        n1 = _lib.moe_workspace_size(make_params(cfg, flags=_lib.MOE_FLAG_TRAINING))[1]
        assert n1 > n0 + 4 * cfg.T * cfg.d  # at least the router's share of dx


def _fake_grads(cfg, ins, base=1 << 41):
    a = lambda i: base + i * (1 << 30)  # noqa: E731
    return _lib.moe_grads_t(dx=a(0), dW_gate=a(1), db_gate=a(2) if ins.b_gate else None, dW1=a(3),
                            dW3=a(4) if cfg.act == "swiglu" else None, dW2=a(5),
                            db1=a(6) if ins.b1 else None, db2=a(7) if ins.b2 else None)


def test_backward_validation_happens_before_any_launch():
    cfg = config("mixtral")
    p = make_params(cfg, flags=_lib.MOE_FLAG_TRAINING)
    _, need = _lib.moe_workspace_size(p)
    ins, outs = _fake_io(cfg)
    dy = 1 << 42
    n0 = _lib.moe_kernel_launches()
    # no training flag
    p0 = make_params(cfg)
    assert _lib.moe_backward(p0, ins, outs, dy, 0.0, _fake_grads(cfg, ins), 1 << 44, need,
                             None) == _lib.MOE_ERR_INVALID_ARG
    # missing dy, non-finite d_aux, missing or extra gradient arrays, unaligned pointers
    g = _fake_grads(cfg, ins)
    assert _lib.moe_backward(p, ins, outs, None, 0.0, g, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_backward(p, ins, outs, dy, float("nan"), g, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG
    for field, value in (("dW3", None), ("dx", None), ("db1", 1 << 43), ("dW_noise", 1 << 43),
                         ("dW2", (1 << 43) + 4)):
        g = _fake_grads(cfg, ins)
        setattr(g, field, value)
        assert _lib.moe_backward(p, ins, outs, dy, 0.0, g, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG
    # workspace too small
    assert _lib.moe_backward(p, ins, outs, dy, 0.0, _fake_grads(cfg, ins), 1 << 44, need - 1,
                             None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_kernel_launches() == n0


@pytest.mark.parametrize("base,over,expect", [
    ("switch", {}, _lib.MOE_OK),
    ("mixtral", {}, _lib.MOE_OK),
    ("tiny", {}, _lib.MOE_ERR_UNSUPPORTED),                     # fp32 layer
    ("deepseek", {}, _lib.MOE_ERR_UNSUPPORTED),                 # shared experts
    ("switch", {"flags": 1}, _lib.MOE_ERR_UNSUPPORTED),          # FFMA experts
    ("switch", {"flags": 8}, _lib.MOE_ERR_UNSUPPORTED),          # training
    ("switch", {"d_model": 776}, _lib.MOE_ERR_UNSUPPORTED),      # d not a multiple of 16
    ("switch", {"weight_format": 2}, _lib.MOE_OK),               # the 4-bit format (d, F multiples of 128)
    ("switch", {"weight_format": 3}, _lib.MOE_ERR_INVALID_ARG),
])
def test_int8_weight_combinations(base, over, expect):
    p = make_params(config(base, weights="int8"))
    for k, v in over.items():
        setattr(p, k, v)
    assert _lib.moe_workspace_size(p)[0] == expect


def test_int8_scales_must_match_the_format():
    base = 1 << 40
    for fmt in ("int8", "dtype"):
        cfg = config("mixtral", weights=fmt)
        p = make_params(cfg)
        _, need = _lib.moe_workspace_size(p)
        ins, outs = _fake_io(cfg)
        if fmt == "int8":
            ins.W1_scale, ins.W2_scale = base + 30 * (1 << 30), base + 31 * (1 << 30)  # W3_scale missing
        else:
            ins.W2_scale = base + 31 * (1 << 30)  # a scale with bf16 weights
        assert _lib.moe_forward(p, ins, outs, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG


def test_quantize_rejects_bad_arguments():
    assert _lib.moe_quantize_int8(None, _lib.MOE_BF16, 4, 8, 1 << 40, 1 << 41, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_quantize_int8(1 << 40, 7, 4, 8, 1 << 40, 1 << 41, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_quantize_int8(1 << 40, _lib.MOE_BF16, 4, 0, 1 << 40, 1 << 41, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_quantize_int8(1 << 40, _lib.MOE_BF16, 0, 8, 1 << 40, 1 << 41, None) == _lib.MOE_OK  # nothing to do


def test_empty_batch_is_valid():
    for name in ("switch", "mixtral", "tiny"):
        p = make_params(config(name), T=0)
        st, n = _lib.moe_workspace_size(p)
        assert st == _lib.MOE_OK and n > 0


def test_bounded_wait_check_validates_before_launch():
    n0 = _lib.moe_kernel_launches()
    assert _lib.moe_check_bounded_wait(None, 1024, 1000, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_check_bounded_wait(1 << 40, 2, 1000, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_check_bounded_wait((1 << 40) + 16, 1024, 1000, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_check_bounded_wait(1 << 40, 1024, 0, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_check_bounded_wait(1 << 40, 1024, 2000000, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_kernel_launches() == n0


# ---- expert parallelism over G emulated ranks ---------------------------------

@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseek", "skewed"])
def test_ep_workspace_size(name):
    cfg = config(name)
    p = make_params(cfg)
    one = _lib.moe_workspace_size(p)[1]
    for G in (1, 2, 4, 8):
        if cfg.E % G:
            continue
        st, n = _lib.moe_ep_workspace_size(p, G)
        assert st == _lib.MOE_OK
        assert n > one  # every rank's private region plus the owners' receive buffers


@pytest.mark.parametrize("G,expect", [(0, _lib.MOE_ERR_INVALID_ARG), (-1, _lib.MOE_ERR_INVALID_ARG),
                                      (17, _lib.MOE_ERR_INVALID_ARG), (3, _lib.MOE_ERR_INVALID_ARG),
                                      (16, _lib.MOE_ERR_INVALID_ARG), (8, _lib.MOE_OK)])
def test_ep_rank_count_validated(G, expect):
    # mixtral: E = 8, so G must divide 8 (16 > E fails the divisibility)
    st, _ = _lib.moe_ep_workspace_size(make_params(config("mixtral")), G)
    assert st == expect


@pytest.mark.parametrize("over,flags", [({"weights": "int8"}, 0), ({}, _lib.MOE_FLAG_TRAINING),
                                        ({}, _lib.MOE_FLAG_UNFUSED_EXPERTS)])
def test_ep_unsupported_combinations(over, flags):
    p = make_params(config("switch", **over), flags=flags)
    assert _lib.moe_ep_workspace_size(p, 2)[0] == _lib.MOE_ERR_UNSUPPORTED


def test_ep_forward_validates_before_any_launch():
    cfg = config("tiny")
    p = make_params(cfg)
    n0 = _lib.moe_kernel_launches()
    inputs, outputs = _lib.moe_inputs_t(), _lib.moe_outputs_t()
    # null pointers everywhere: rejected on the host, nothing launched
    assert _lib.moe_forward_ep(p, 2, inputs, outputs, None, 0, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_forward_ep(p, 3, inputs, outputs, None, 0, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_kernel_launches() == n0


# ---- 4-bit expert weights -------------------------------------------------------

@pytest.mark.parametrize("over,expect", [
    ({}, _lib.MOE_OK),
    ({"d": 192}, _lib.MOE_ERR_UNSUPPORTED),                  # d_model not a multiple of the group
    ({"F": 320}, _lib.MOE_ERR_UNSUPPORTED),                  # d_ff not a multiple of the group
    ({"dtype": "f32"}, _lib.MOE_ERR_UNSUPPORTED),
    ({"S": 2}, _lib.MOE_ERR_UNSUPPORTED),                    # shared experts
])
def test_int4_weight_combinations(over, expect):
    kw = dict(T=64, d=256, E=8, k=2, F=512, weights="int4")
    kw.update(over)
    cfg = config("mixtral", **kw)
    assert _lib.moe_workspace_size(make_params(cfg))[0] == expect


def test_int4_training_unsupported():
    cfg = config("mixtral", T=64, d=256, E=8, k=2, F=512, weights="int4")
    assert _lib.moe_workspace_size(make_params(cfg, flags=_lib.MOE_FLAG_TRAINING))[0] == _lib.MOE_ERR_UNSUPPORTED


def test_quantize_int4_rejects_bad_arguments():
    n0 = _lib.moe_kernel_launches()
    assert _lib.moe_quantize_int4(16, _lib.MOE_BF16, 4, 100, 16, 16, None) == _lib.MOE_ERR_INVALID_ARG  # cols % 128
    assert _lib.moe_quantize_int4(None, _lib.MOE_BF16, 4, 128, 16, 16, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_quantize_int4(16, 7, 4, 128, 16, 16, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_quantize_int4(16, _lib.MOE_BF16, 0, 128, 16, 16, None) == _lib.MOE_OK  # nothing to do
    assert _lib.moe_kernel_launches() == n0


# ---- router weights prepared once per weight update ------------------------------

@pytest.mark.parametrize("name,noisy", [("switch", False), ("deepseek", False), ("skewed", True), ("mixtral", True)])
def test_router_weights_size(name, noisy):
    cfg = config(name, noisy=noisy)
    st, n = _lib.moe_router_weights_size(make_params(cfg))
    e_pad = (cfg.E + 63) // 64 * 64
    assert st == _lib.MOE_OK and n == 3 * 2 * e_pad * cfg.d * (2 if noisy else 1)
    # independent of the batch size
    assert _lib.moe_router_weights_size(make_params(cfg, T=7))[1] == n


def test_router_weights_need_the_tensor_core_router():
    assert _lib.moe_router_weights_size(make_params(config("tiny")))[0] == _lib.MOE_ERR_UNSUPPORTED
    p = make_params(config("switch"), flags=_lib.MOE_FLAG_FFMA_ROUTER)
    assert _lib.moe_router_weights_size(p)[0] == _lib.MOE_ERR_UNSUPPORTED
    n0 = _lib.moe_kernel_launches()
    p = make_params(config("switch"))
    _, n = _lib.moe_router_weights_size(p)
    assert _lib.moe_prepare_router_weights(p, None, None, 1 << 40, n, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_prepare_router_weights(p, 1 << 40, None, 1 << 41, n - 1, None) == _lib.MOE_ERR_WORKSPACE
    assert _lib.moe_prepare_router_weights(p, 1 << 40, 1 << 42, 1 << 41, n, None) == _lib.MOE_ERR_INVALID_ARG  # no noise
    assert _lib.moe_prepare_router_weights(p, (1 << 40) + 4, None, 1 << 41, n, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_kernel_launches() == n0


def test_prepared_router_weights_rejected_for_cuda_core_routers():
    cfg = config("tiny")
    p = make_params(cfg)
    _, need = _lib.moe_workspace_size(p)
    ins, outs = _fake_io(cfg)
    ins.router_weights = 1 << 41
    n0 = _lib.moe_kernel_launches()
    assert _lib.moe_forward(p, ins, outs, 1 << 44, need, None) == _lib.MOE_ERR_INVALID_ARG
    assert _lib.moe_kernel_launches() == n0
