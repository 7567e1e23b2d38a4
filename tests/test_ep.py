"""Expert parallelism over G ranks emulated on one GPU (moe_forward_ep) against the
oracle's rank-by-rank layer (orc.ep_forward).

Expert parallelism places the experts on different devices while the tokens are
sharded over the workers, and tokens travel between them by an AllToAll
("MoE架构解析" §3.2 分布式训练优化, §5 问题3; "MoE混合专家模型原理与实战" §4.2
专家分片).  Bars (the layer's specification):
  - expert indices, per-shard capacity drops, counts and the receive-order rows
    (perm_row): bit-exact against the oracle's exchange re-run on the device's
    fp32 logits;
  - gates <= 1e-5 absolute, balance statistic <= 1e-5 relative;
  - layer output: relative Frobenius error <= 2e-2 (bf16) or 1e-4 (fp32);
  - without a capacity limit, the G-rank output equals the single-rank
    moe_forward output bit for bit wherever the two routers produced the same
    logits (every expert row is computed by the same kernels in the same order).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from parity_utils import PROB_TOL, Y_TOL, oracle_noise, rel_frobenius, sample_tokens, to_cpu
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs

pytestmark = pytest.mark.gpu


def run_ep(cfg, inp, G, **kw):
    layer = MoELayer(cfg, inp, want_logits=True, want_probs=True, ep_ranks=G, **kw)
    layer.run()
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    return to_cpu(layer.out)


def check_ep(cfg, inp_cpu, out, G, tokens=None):
    """Bit-exact exchange on the device logits, then gates, aux and y against fp64."""
    ref = orc.ep_forward(inp_cpu["x"], inp_cpu["W_gate"], inp_cpu["b_gate"], inp_cpu["W1"], inp_cpu["W3"],
                         inp_cpu["W2"], inp_cpu["b1"], inp_cpu["b2"], E=cfg.E, S=cfg.S, k=cfg.k, G=G,
                         act_name=cfg.act, renormalize=cfg.renormalize, cf=cfg.cf,
                         residual_mode=cfg.residual_mode, tokens=tokens,
                         logits=out["logits"].numpy())
    np.testing.assert_array_equal(out["expert_idx"].numpy(), ref.idx)
    np.testing.assert_array_equal(out["dropped"].numpy(), ref.ex.dropped)
    np.testing.assert_array_equal(out["counts"].numpy(), ref.counts)
    np.testing.assert_array_equal(out["perm_row"].numpy(), ref.ex.recv_row)
    np.testing.assert_allclose(out["gates"].numpy(), ref.gates, rtol=0, atol=PROB_TOL)
    np.testing.assert_allclose(out["probs"].numpy(), ref.probs, rtol=0, atol=PROB_TOL)
    aux = float(out["aux"][0])
    assert abs(aux - ref.aux) <= 1e-5 * max(1.0, abs(ref.aux)), (aux, ref.aux)
    tok = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    err = rel_frobenius(out["y"][torch.as_tensor(tok, dtype=torch.long)].double().numpy(), ref.y)
    assert err <= Y_TOL[cfg.dtype], err
    # tokens whose routed slots were all dropped return x exactly (mode 0, no shared experts)
    if cfg.residual_mode == 0 and cfg.S == 0:
        gone = out["dropped"].bool().all(dim=1)
        if int(gone.sum()):
            assert torch.equal(out["y"][gone], inp_cpu["x"][gone])
    return ref, err


SMALL = {
    "tiny_f32": config("tiny", T=203),                                           # FFMA experts, biases, GELU
    "tiny_f32_cap": config("tiny", T=203, cf=1.0),
    "bf16_swiglu": config("mixtral", T=500, d=256, E=8, k=2, F=384),
    "bf16_swiglu_cap": config("mixtral", T=500, d=256, E=8, k=2, F=384, cf=1.0),
    "bf16_relu_k1_cap": config("switch", T=777, d=128, E=16, F=256),              # Switch-like, drops
    "bf16_shared": config("deepseek", T=333, d=256, E=16, k=3, F=200, S=2),       # shared experts, ragged F
    "bf16_residual1": config("mixtral", T=300, d=128, E=8, k=2, F=256, residual_mode=1, cf=1.25),
    "bf16_noisy": config("mixtral", T=256, d=128, E=8, k=2, F=256, noisy=True, noise_min_std=0.01),
}


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("name", list(SMALL))
def test_ep_small_layers(name, G):
    cfg = SMALL[name]
    if cfg.E % G:
        pytest.skip("E not a multiple of G")
    inp = make_inputs(cfg, 0, device="cuda")
    out = run_ep(cfg, inp, G)
    cpu = to_cpu(inp)
    if cfg.noisy:  # the oracle's noisy logits are the device logits' reference
        r64 = orc.route(cpu["x"], cpu["W_gate"], cpu["b_gate"], k=cfg.k, renormalize=cfg.renormalize,
                        cf=cfg.cf, noise=oracle_noise(cfg, cpu))
        tol = 1e-5 * max(1.0, float(np.abs(cpu["noise_eps"].double().numpy()).max()))
        assert np.abs(out["logits"].double().numpy() - r64.logits).max() <= tol
    check_ep(cfg, cpu, out, G)


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("name", ["tiny_f32", "bf16_swiglu", "bf16_shared"])
def test_ep_without_capacity_equals_single_rank_bitwise(name, G):
    cfg = SMALL[name]
    if cfg.E % G:
        pytest.skip("E not a multiple of G")
    inp = make_inputs(cfg, 0, device="cuda")
    ep = run_ep(cfg, inp, G)
    one = MoELayer(cfg, inp, want_logits=True)
    one.run()
    torch.cuda.synchronize()
    single = to_cpu(one.out)
    same = (ep["logits"] == single["logits"]).all(dim=1)  # tokens whose router logits agree bitwise
    assert int(same.sum()) > 0
    assert torch.equal(ep["expert_idx"][same], single["expert_idx"][same])
    assert torch.equal(ep["gates"][same], single["gates"][same])
    assert torch.equal(ep["y"][same], single["y"][same])  # a token's output depends on its own routing only
    if bool(same.all()):
        assert torch.equal(ep["perm_row"], single["perm_row"])
        assert torch.equal(ep["counts"], single["counts"])
        assert torch.equal(ep["y"], single["y"])


def test_ep_rank_with_no_tokens():
    # T < G: rank 3 (of 4) holds no token; its experts still receive rows from the others
    cfg = config("mixtral", T=3, d=128, E=8, k=2, F=256)
    inp = make_inputs(cfg, 0, device="cuda")
    out = run_ep(cfg, inp, 4)
    check_ep(cfg, to_cpu(inp), out, 4)


def test_ep_repeated_calls_reuse_the_workspace():
    cfg = SMALL["bf16_swiglu_cap"]
    inp = make_inputs(cfg, 0, device="cuda")
    layer = MoELayer(cfg, inp, want_logits=True, want_probs=True, ep_ranks=4)
    layer.run()
    torch.cuda.synchronize()
    first = to_cpu(layer.out)
    inp2 = make_inputs(cfg, 1, device="cuda")
    layer.set_x(inp2["x"])
    layer.run()
    layer.set_x(inp["x"])
    layer.run()
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    again = to_cpu(layer.out)
    for key in ("y", "expert_idx", "dropped", "perm_row", "counts", "aux"):
        assert torch.equal(first[key], again[key]), key


# full-size layers (the shapes the expert-parallel question is asked about)
FULL_SAMPLE = 192


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("name", ["deepseek", "skewed"])
def test_ep_full_size(name, G):
    cfg = config(name)
    inp = make_inputs(cfg, 0, device="cuda")
    out = run_ep(cfg, inp, G)
    cpu = to_cpu(inp)
    del inp
    torch.cuda.empty_cache()
    tokens = sample_tokens(cfg, out, FULL_SAMPLE)
    ref, err = check_ep(cfg, cpu, out, G, tokens=tokens)
    print(f"{name} G={G}: per-shard capacity {ref.C_rank[0]}, kept slots {int((ref.ex.dropped == 0).sum())}, "
          f"rel-Frobenius {err:.3e} on {len(tokens)} tokens, aux {float(out['aux'][0]):.6f}")
