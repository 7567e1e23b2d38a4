"""Seeded synthetic inputs for the layer configurations (no layer arithmetic).

Shared by the tests and the benchmark: the CUDA library and the CPU oracle are
fed the same bits.  Every tensor is drawn from a seeded torch.Generator in the
fixed order x, W_gate, b_gate, W1, W3, W2, b1, b2, generated in fp32 and
rounded once (round-to-nearest-even) to the layer dtype; the router weights
stay fp32.

Configurations (shapes and distributions of the workloads the pages discuss):
  tiny      T=256  d=64   E=8   k=2 F=128   GELU(tanh)+biases, no capacity, fp32;
            x~N(0,1), W_gate/W1/W2~N(0,0.02^2), biases 0
  switch    T=8192 d=768  E=128 k=1 F=3072  ReLU, capacity factor 1.25, bf16 (raw p gate);
            x~N(0,1), all weights truncated normal, var 0.1/fan_in, cut at +-2 sigma
  mixtral   T=16384 d=4096 E=8  k=2 F=14336 SwiGLU, renormalised gates, bf16;
            x~N(0,1), W1/W3/W2~N(0,1/fan_in), W_gate~N(0,0.02^2)
  deepseek  T=16384 d=2048 E=64 (+2 shared) k=6 F=1408 SwiGLU, raw p gates, bf16; as mixtral
  skewed    T=4096 d=7168 E=256 k=8 F=2048 SwiGLU, capacity factor 1.0, renormalised, bf16;
            as mixtral plus a router bias b[pi(r)] = -1.2 ln r (r = 1..E, pi a seeded
            permutation), so the bias alone gives Zipf(1.2) expert popularity
  decode    the first 64 tokens of skewed with the same weights (capacity 1.0 -> C = 0)
  decode_nocap  the same without a capacity limit

Int8 / int4 expert weights (weights="int8" / "int4"): the tensors above are drawn
as usual; the library quantises W1, W3, W2 itself (moe_quantize_int8 /
moe_quantize_int4), so the inputs carry no quantisation arithmetic.

Noisy top-k gating (any config with noisy=True): after the tensors above, W_noise
and b_noise ~ U(-1/sqrt(d), 1/sqrt(d)) (nn.Linear's default initialisation of the
noise projection; noise scales softplus(x W_noise + b) around 0.4-1.1) and
noise_eps ~ N(0,1) of shape [T, E] (the standard normal draws the gate scales); for
a config with a parent, the first T rows of the parent's draws.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    S: int = 0
    act: str = "swiglu"          # relu | gelu_tanh | gelu_erf | swiglu
    cf: float | None = None      # capacity factor, None = no limit
    dtype: str = "bf16"          # bf16 | f32
    renormalize: bool = True
    residual_mode: int = 0
    bias: bool = False           # expert biases present (zero-initialised)
    init: str = "fan_in"         # small | trunc | fan_in
    zipf: float | None = None    # router-bias Zipf exponent
    parent: str | None = None    # take the first T tokens of this config's inputs
    noisy: bool = False          # noisy top-k gating (training mode)
    noise_min_std: float = 0.0   # floor added to the softplus noise scale
    weights: str = "dtype"       # dtype | int8 (per output row) | int4 (per group of 128 inputs)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def expert_flops(self, kept_slots: int) -> float:
        """Multiply-add flops of the expert GEMMs for `kept_slots` routed rows."""
        per_row = 2 * self.d * self.F * (3 if self.act == "swiglu" else 2)
        return float(per_row) * (kept_slots + self.S * self.T)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, d=64, E=8, k=2, F=128, act="gelu_tanh", cf=None,
                        dtype="f32", renormalize=True, bias=True, init="small"),
    "switch": LayerConfig("switch", T=8192, d=768, E=128, k=1, F=3072, act="relu", cf=1.25,
                          dtype="bf16", renormalize=False, init="trunc"),
    "mixtral": LayerConfig("mixtral", T=16384, d=4096, E=8, k=2, F=14336, act="swiglu",
                           dtype="bf16", renormalize=True),
    "deepseek": LayerConfig("deepseek", T=16384, d=2048, E=64, k=6, F=1408, S=2, act="swiglu",
                            dtype="bf16", renormalize=False),
    "skewed": LayerConfig("skewed", T=4096, d=7168, E=256, k=8, F=2048, act="swiglu", cf=1.0,
                          dtype="bf16", renormalize=True, zipf=1.2),
    "decode": LayerConfig("decode", T=64, d=7168, E=256, k=8, F=2048, act="swiglu", cf=1.0,
                          dtype="bf16", renormalize=True, zipf=1.2, parent="skewed"),
    "decode_nocap": LayerConfig("decode_nocap", T=64, d=7168, E=256, k=8, F=2048, act="swiglu",
                                cf=None, dtype="bf16", renormalize=True, zipf=1.2, parent="skewed"),
}


def config(name: str, **overrides) -> LayerConfig:
    return replace(CONFIGS[name], **overrides)


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _trunc(shape, std, g, device):
    t = torch.empty(shape, device=device, dtype=torch.float32)
    torch.nn.init.trunc_normal_(t, mean=0.0, std=std, a=-2 * std, b=2 * std, generator=g)
    return t


def make_inputs(cfg: LayerConfig, seed: int = 0, device="cpu") -> dict:
    """Seeded tensors for `cfg` on `device` (weights of all E + S experts)."""
    if cfg.parent is not None:
        base = make_inputs(replace(CONFIGS[cfg.parent], d=cfg.d, E=cfg.E, k=cfg.k, F=cfg.F,
                                   noisy=cfg.noisy), seed, device)
        base["x"] = base["x"][: cfg.T].contiguous()
        if cfg.noisy:
            base["noise_eps"] = base["noise_eps"][: cfg.T].contiguous()
        return base
    g = torch.Generator(device=device).manual_seed(seed)
    T, d, E, F, S = cfg.T, cfg.d, cfg.E, cfg.F, cfg.S
    ES = E + S
    dt = cfg.torch_dtype
    if cfg.init == "small":
        w = lambda shape, fan_in: _normal(shape, 0.02, g, device)  # noqa: E731
        wg_std = 0.02
    elif cfg.init == "trunc":
        w = lambda shape, fan_in: _trunc(shape, math.sqrt(0.1 / fan_in), g, device)  # noqa: E731
        wg_std = None
    else:
        w = lambda shape, fan_in: _normal(shape, 1.0 / math.sqrt(fan_in), g, device)  # noqa: E731
        wg_std = 0.02
    out = {}
    out["x"] = _normal((T, d), 1.0, g, device).to(dt)
    out["W_gate"] = (_trunc((E, d), math.sqrt(0.1 / d), g, device) if wg_std is None
                     else _normal((E, d), wg_std, g, device))
    if cfg.zipf is not None:
        perm = torch.randperm(E, generator=g, device=device)
        ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
        bg = torch.empty(E, device=device, dtype=torch.float64)
        bg[perm] = -cfg.zipf * torch.log(ranks)
        out["b_gate"] = bg.float()
    elif cfg.bias:
        out["b_gate"] = torch.zeros(E, device=device, dtype=torch.float32)
    else:
        out["b_gate"] = None
    out["W1"] = w((ES, F, d), d).to(dt)
    out["W3"] = w((ES, F, d), d).to(dt) if cfg.act == "swiglu" else None
    out["W2"] = w((ES, d, F), F).to(dt)
    out["b1"] = torch.zeros(ES, F, device=device, dtype=dt) if cfg.bias else None
    out["b2"] = torch.zeros(ES, d, device=device, dtype=dt) if cfg.bias else None
    if cfg.noisy:
        # the noise projection as nn.Linear initialises it (U(-1/sqrt(d), 1/sqrt(d)) for the
        # weight and the bias), as in the NoisyTop1Gate listing
        bound = 1.0 / math.sqrt(d)
        out["W_noise"] = (torch.rand((E, d), generator=g, device=device) * 2.0 - 1.0) * bound
        out["b_noise"] = (torch.rand((E,), generator=g, device=device) * 2.0 - 1.0) * bound
        out["noise_eps"] = _normal((T, E), 1.0, g, device)
    else:
        out["W_noise"] = out["b_noise"] = out["noise_eps"] = None
    return out
