"""Helpers for the GPU parity tests: run the CUDA layer through the C ABI and
compare it with the fp64 CPU oracle on the same seeded inputs.

Bars (per the layer's specification):
  - expert indices, counts, capacity drops and permutation rows: bit-exact
    against the oracle's selection re-run on the device's fp32 logits;
  - noisy top-k gating: the noisy logits within 1e-5 * max(1, max |eps|) absolute
    of the fp64 oracle's (fp32 accumulation of two d-long projections);
  - router probabilities and gates: <= 1e-5 absolute against the fp64 oracle
    (tokens whose k-th and (k+1)-th fp64 probabilities are within 1e-6 are
    excluded from the index comparison against the oracle's own selection, and
    counted);
  - layer output: relative Frobenius error <= 2e-2 (bf16) or 1e-4 (fp32);
  - tokens whose routed slots were all dropped: y == x bit-exactly.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import MoELayer, _lib

PROB_TOL = 1e-5
LOGIT_TOL = 1e-5
NEAR_TIE = 1e-6
Y_TOL = {"bf16": 2e-2, "f32": 1e-4}


def to_cpu(d: dict) -> dict:
    return {k: (None if v is None else v.detach().cpu()) for k, v in d.items()}


def run_device(cfg, inputs: dict, *, flags: int = 0, residual_mode=None, stages=None) -> dict:
    layer = MoELayer(cfg, inputs, flags=flags, residual_mode=residual_mode, want_logits=True,
                     want_probs=True)
    if stages is None:
        layer.run()
    else:
        for s in stages:
            layer.run(s)
    torch.cuda.synchronize()
    assert layer.device_status() == _lib.MOE_OK
    return to_cpu(layer.out)


def check_routing_bitexact(cfg, out: dict):
    """Selection, counts, drops and permutation order vs the oracle re-run on the device logits."""
    r = orc.route_from_logits(out["logits"].numpy(), k=cfg.k, renormalize=cfg.renormalize, cf=cfg.cf)
    np.testing.assert_array_equal(out["expert_idx"].numpy(), r.idx)
    np.testing.assert_array_equal(out["counts"].numpy(), r.counts)
    np.testing.assert_array_equal(out["dropped"].numpy(), r.dropped)
    np.testing.assert_array_equal(out["perm_row"].numpy(), r.perm_row)
    # gates of the re-run use fp64 softmax of the same logits
    np.testing.assert_allclose(out["gates"].numpy(), r.gates, rtol=0, atol=PROB_TOL)
    return r


def check_router_vs_fp64(cfg, inp: dict, out: dict) -> int:
    """Probabilities, gates, selection and aux against the fp64 oracle; returns near-tie count."""
    r64 = orc.route(inp["x"], inp["W_gate"], inp["b_gate"], k=cfg.k, renormalize=cfg.renormalize,
                    cf=cfg.cf, noise=oracle_noise(cfg, inp))
    if cfg.noisy:
        # noisy logits: fp32 accumulation of the two projections; the noise term scales the
        # projection error by |eps| (a few units for normal draws)
        tol = LOGIT_TOL * max(1.0, float(np.abs(inp["noise_eps"].double().numpy()).max()))
        assert np.abs(out["logits"].double().numpy() - r64.logits).max() <= tol
    p_dev = out["probs"].double().numpy()
    assert np.abs(p_dev - r64.probs).max() <= PROB_TOL
    E = cfg.E
    ps = -np.sort(-r64.probs, axis=1)
    kk = min(cfg.k + 1, E)
    gaps = ps[:, : kk - 1] - ps[:, 1:kk] if kk > 1 else np.ones((cfg.T, 1))
    near = (gaps <= NEAR_TIE).any(axis=1)
    ok = ~near
    np.testing.assert_array_equal(out["expert_idx"].numpy()[ok], r64.idx[ok])
    assert np.abs(out["gates"].double().numpy()[ok] - r64.gates[ok]).max(initial=0.0) <= PROB_TOL
    aux_dev = float(out["aux"][0])
    assert abs(aux_dev - r64.aux) <= 1e-5 * max(1.0, abs(r64.aux)), (aux_dev, r64.aux)
    return int(near.sum())


def oracle_noise(cfg, inp: dict):
    """The oracle's noise argument for noisy top-k gating, or None."""
    if not cfg.noisy:
        return None
    return (inp["W_noise"], inp["b_noise"], inp["noise_eps"], cfg.noise_min_std)


def oracle_rows(cfg, inp: dict, r, tokens, residual_mode=None):
    mode = cfg.residual_mode if residual_mode is None else residual_mode
    return orc.output_rows(inp["x"], inp["W1"], inp["W3"], inp["W2"], inp["b1"], inp["b2"], r.idx,
                           r.gates, r.dropped, E=cfg.E, S=cfg.S, act_name=cfg.act,
                           residual_mode=mode, tokens=tokens)


def rel_frobenius(a: np.ndarray, b: np.ndarray) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def check_output(cfg, inp: dict, out: dict, r, tokens=None, residual_mode=None) -> float:
    T = cfg.T
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    y_ref = oracle_rows(cfg, inp, r, tok, residual_mode)
    y_dev = out["y"][torch.as_tensor(tok, dtype=torch.long)].double().numpy()
    err = rel_frobenius(y_dev, y_ref)
    assert err <= Y_TOL[cfg.dtype], err
    return err


def check_dropped_tokens_pass_x(cfg, inp: dict, out: dict, residual_mode=None):
    """Tokens whose routed slots were all dropped return x exactly (no shared experts)."""
    mode = cfg.residual_mode if residual_mode is None else residual_mode
    if mode != 0 or cfg.S != 0:
        return 0
    all_dropped = out["dropped"].bool().all(dim=1)
    n = int(all_dropped.sum())
    if n:
        assert torch.equal(out["y"][all_dropped], inp["x"][all_dropped])
    return n


def sample_tokens(cfg, out: dict, n: int, seed: int = 1234) -> np.ndarray:
    """Seeded subsample plus the first/last tokens and those of the least-loaded expert."""
    rng = np.random.default_rng(seed)
    T = cfg.T
    picks = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    counts = out["counts"].numpy()
    nz = np.nonzero(counts)[0]
    if len(nz):
        e = nz[np.argmin(counts[nz])]
        hit = np.nonzero((out["expert_idx"].numpy() == e).any(axis=1))[0][:64]
        picks |= set(hit.tolist())
    return np.array(sorted(picks))


def quantized_oracle_rows(cfg, inp: dict, qinp: dict, r, tokens, dequantize):
    """Oracle rows of the listed tokens for a layer with quantised expert weights, on the
    exactly dequantised weights, one expert at a time (a full-size layer's dequantised
    weights would not fit the host's memory in fp64): the experts' outputs for the
    tokens' kept slots (orc.expert_apply), then the oracle's combine."""
    tok = np.asarray(tokens, dtype=np.int64)
    slots = [(int(t), j) for t in tok for j in range(cfg.k) if not r.dropped[t, j]]
    row_of = np.full((cfg.T, cfg.k), -1, dtype=np.int32)
    for n, (t, j) in enumerate(slots):
        row_of[t, j] = n
    o = np.zeros((max(len(slots), 1), cfg.d))
    for e in sorted({int(r.idx[t, j]) for t, j in slots}):
        sel = [n for n, (t, j) in enumerate(slots) if r.idx[t, j] == e]
        one = {}
        for name in ("W1", "W3", "W2"):
            q = qinp.get(name)
            one[name] = None if q is None else dequantize(q[e:e + 1].numpy(), qinp[name + "_scale"][e:e + 1].numpy())
        b1 = None if inp.get("b1") is None else inp["b1"][e:e + 1]
        b2 = None if inp.get("b2") is None else inp["b2"][e:e + 1]
        o[sel] = orc.expert_apply(inp["x"], one["W1"], one["W3"], one["W2"], b1, b2,
                                  [slots[n][0] for n in sel], np.zeros(len(sel), dtype=np.int32), act_name=cfg.act)
    return orc.combine_rows(inp["x"], r.gates, r.dropped, row_of, o, residual_mode=cfg.residual_mode, tokens=tok)
