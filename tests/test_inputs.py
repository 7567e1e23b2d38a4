"""The seeded input recipe (CPU): determinism, shapes, distributions."""
import math

import torch

from sparse_mixture_experts_scan_b300 import config, make_inputs


def test_same_seed_same_bits_and_different_seed_differs():
    cfg = config("tiny")
    a, b, c = make_inputs(cfg, 0), make_inputs(cfg, 0), make_inputs(cfg, 1)
    for k in ("x", "W_gate", "W1", "W2"):
        assert torch.equal(a[k], b[k])
        assert not torch.equal(a[k], c[k])


def test_shapes_and_dtypes_small_switch_like():
    cfg = config("switch", T=256, d=64, E=8, F=128)
    t = make_inputs(cfg)
    assert t["x"].shape == (256, 64) and t["x"].dtype == torch.bfloat16
    assert t["W_gate"].dtype == torch.float32 and t["W_gate"].shape == (8, 64)
    assert t["W1"].shape == (8, 128, 64) and t["W2"].shape == (8, 64, 128)
    assert t["W3"] is None and t["b1"] is None
    # truncated normal, var 0.1/fan_in, cut at 2 sigma
    s = math.sqrt(0.1 / 64)
    assert t["W1"].float().abs().max() <= 2 * s * 1.01
    assert abs(t["W1"].float().std().item() - s * 0.88) < 0.1 * s  # std of N cut at 2 sigma


def test_shared_expert_weights_are_appended():
    cfg = config("deepseek", T=64, d=64, F=32)
    t = make_inputs(cfg)
    assert t["W1"].shape == (66, 32, 64) and t["W3"].shape == (66, 32, 64)
    assert t["W2"].shape == (66, 64, 32)


def test_zipf_router_bias():
    cfg = config("skewed", T=16, d=64, F=64)
    t = make_inputs(cfg)
    bg = t["b_gate"].double()
    p = torch.softmax(bg, 0)
    ranked = torch.sort(p, descending=True).values
    r = torch.arange(1, 257, dtype=torch.float64)
    zipf = r ** -1.2 / (r ** -1.2).sum()
    torch.testing.assert_close(ranked, zipf, rtol=1e-6, atol=1e-9)


def test_decode_is_prefix_of_skewed():
    sk = make_inputs(config("skewed", d=64, F=64))
    de = make_inputs(config("decode", d=64, F=64))
    assert torch.equal(de["x"], sk["x"][:64])
    assert torch.equal(de["W1"], sk["W1"])
