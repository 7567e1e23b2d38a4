"""GPU parity of the backward pass at the full sizes of the layer configurations.

The oracle cannot run the whole backward at these sizes, so it checks what it
can compute from a few tokens, with the device's routing decisions:
  - dx of a seeded token sample (with d_aux = 0 the input gradient of a token
    depends on that token alone), against the oracle run on the sample;
  - the weight gradients of the least-loaded touched expert (they depend only on
    the tokens routed to it), against the oracle run on those tokens;
and compares every gradient with the CUDA-core cross-check path.  Bars as in
the small-size tests: relative Frobenius error <= 2e-2 against the oracle, and
<= 1e-2 between the tensor-core and CUDA-core paths.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import MoELayer, _lib, config, make_inputs
from parity_utils import oracle_noise, rel_frobenius, to_cpu

pytestmark = pytest.mark.gpu

TRAIN = _lib.MOE_FLAG_TRAINING
N_TOKENS = {"switch": 64, "deepseek": 16, "skewed": 8, "mixtral": 4}


def _sub_oracle(cfg, cpu, out, dy, tokens):
    """Oracle gradients for the sub-batch `tokens` (d_aux = 0)."""
    t = torch.as_tensor(tokens, dtype=torch.long)
    sub = {k: v for k, v in cpu.items()}
    sub["x"] = cpu["x"][t]
    if cfg.noisy:
        sub["noise_eps"] = cpu["noise_eps"][t]
    return orc.backward(sub["x"], sub["W_gate"], sub["b_gate"], sub["W1"], sub["W3"], sub["W2"], sub["b1"],
                        sub["b2"], idx=out["expert_idx"][t].numpy(), dropped=out["dropped"][t].numpy(),
                        dy=dy[t], d_aux=0.0, E=cfg.E, S=cfg.S, act_name=cfg.act,
                        renormalize=cfg.renormalize, residual_mode=cfg.residual_mode,
                        noise=oracle_noise(cfg, sub))


@pytest.mark.parametrize("name", ["switch", "deepseek", "skewed", "mixtral"])
def test_full_size_backward(name):
    cfg = config(name)
    inp = make_inputs(cfg, 0, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(cfg.T, cfg.d, generator=g, device="cuda").to(cfg.torch_dtype)
    layer = MoELayer(cfg, inp, flags=TRAIN)
    layer.run()
    grads = {k: (None if v is None else v.clone()) for k, v in layer.backward(dy, 0.0).items()}
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    out = to_cpu(layer.out)
    cpu = to_cpu(inp)
    dy_cpu = dy.cpu()

    # the CUDA-core cross-check path on the same forward
    ff = MoELayer(cfg, inp, flags=TRAIN | _lib.MOE_FLAG_FFMA_EXPERTS)
    ff.run()
    g_ff = ff.backward(dy, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(ff.out["expert_idx"], layer.out["expert_idx"])
    for k, v in grads.items():
        if v is not None:
            assert rel_frobenius(v.double().cpu().numpy(), g_ff[k].double().cpu().numpy()) <= 1e-2, k
    del ff, g_ff

    # dx of a token sample against the oracle
    rng = np.random.default_rng(9)
    tokens = np.sort(rng.choice(cfg.T, size=N_TOKENS[name], replace=False))
    ref = _sub_oracle(cfg, cpu, out, dy_cpu, tokens)
    dx = grads["dx"][torch.as_tensor(tokens, device="cuda")].double().cpu().numpy()
    assert rel_frobenius(dx, ref["dx"]) <= 2e-2

    # weight gradients of the least-loaded touched expert (routed experts only)
    idx, drop = out["expert_idx"].numpy(), out["dropped"].numpy().astype(bool)
    counts = np.bincount(idx[~drop], minlength=cfg.E)
    e = int(np.argmin(np.where(counts > 0, counts, np.iinfo(np.int64).max)))
    if counts[e] <= 64 and cfg.S == 0:
        tok_e = np.nonzero(((idx == e) & ~drop).any(axis=1))[0]
        ref = _sub_oracle(cfg, cpu, out, dy_cpu, tok_e)
        for k in ("dW1", "dW2", "dW3"):
            if ref[k] is not None:
                assert rel_frobenius(grads[k][e].double().cpu().numpy(), ref[k][e]) <= 2e-2, k


# Weight gradients at the full layer widths against the oracle.  The device backward
# runs on a token subset of the full-size inputs (the full weights), so that every
# expert holds few enough tokens for the oracle to compute its whole gradient in fp64.
# An expert's weight gradients depend only on the tokens routed to it: they equal
# those of a one-expert layer whose only expert is e, fed those tokens with
# dL/d(expert output) = gate * dy (a layer whose router gives gate 1).
SUB_T = {"mixtral": 128, "deepseek": 256}


def _expert_grads_oracle(cfg, cpu, e, tokens, gates, dy):
    t = torch.as_tensor(tokens, dtype=torch.long)
    n = len(tokens)
    one = lambda k: None if cpu.get(k) is None else cpu[k][e:e + 1]  # noqa: E731
    dyg = (torch.as_tensor(gates, dtype=torch.float64)[:, None] * dy[t].double()).numpy()
    ref = orc.backward(cpu["x"][t], torch.zeros(1, cfg.d), None, one("W1"), one("W3"), one("W2"), None, None,
                       idx=np.zeros((n, 1), np.int32), dropped=np.zeros((n, 1), np.uint8), dy=dyg, d_aux=0.0,
                       E=1, S=0, act_name=cfg.act, renormalize=False, residual_mode=0)
    return {k: (None if ref[k] is None else ref[k][0]) for k in ("dW1", "dW3", "dW2")}


@pytest.mark.parametrize("name", ["mixtral", "deepseek"])
def test_full_width_expert_gradients_on_a_token_subset(name):
    full = config(name)
    cfg = config(name, T=SUB_T[name])
    inp = make_inputs(full, 0, device="cuda")
    rng = np.random.default_rng(13)
    tokens = np.sort(rng.choice(full.T, size=cfg.T, replace=False))
    sub = dict(inp)
    sub["x"] = inp["x"][torch.as_tensor(tokens, device="cuda")].contiguous()
    g = torch.Generator(device="cuda").manual_seed(6)
    dy = torch.randn(cfg.T, cfg.d, generator=g, device="cuda").to(cfg.torch_dtype)
    layer = MoELayer(cfg, sub, flags=TRAIN)
    layer.run()
    grads = {k: (None if v is None else v.cpu()) for k, v in layer.backward(dy, 0.37).items()}
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    out = to_cpu(layer.out)
    cpu = to_cpu(sub)
    del inp, sub
    dy_cpu = dy.cpu()
    idx, drop = out["expert_idx"].numpy(), out["dropped"].numpy().astype(bool)
    gates = out["gates"].numpy()
    counts = np.bincount(idx[~drop], minlength=cfg.E)
    touched = np.nonzero(counts)[0]
    # routed experts: the least and the most loaded (all of them for the fine-grained layer)
    check = touched if cfg.E > 8 else [touched[np.argmin(counts[touched])], touched[np.argmax(counts[touched])]]
    for e in check:
        hit = (idx == e) & ~drop
        tok_e = np.nonzero(hit.any(axis=1))[0]
        ref = _expert_grads_oracle(cfg, cpu, int(e), tok_e, gates[hit], dy_cpu)
        for k in ("dW1", "dW3", "dW2"):
            if ref[k] is not None:
                err = rel_frobenius(grads[k][e].double().numpy(), ref[k])
                assert err <= 2e-2, (int(e), k, err)
    # untouched experts get exactly zero
    for e in np.nonzero(counts == 0)[0]:
        assert not grads["dW2"][e].any() and not grads["dW1"][e].any()
    # shared experts: every token, gate 1
    for s in range(cfg.S):
        ref = _expert_grads_oracle(cfg, cpu, cfg.E + s, np.arange(cfg.T), np.ones(cfg.T), dy_cpu)
        for k in ("dW1", "dW3", "dW2"):
            err = rel_frobenius(grads[k][cfg.E + s].double().numpy(), ref[k])
            assert err <= 2e-2, ("shared", s, k, err)
