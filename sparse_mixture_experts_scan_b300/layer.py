"""Torch-facing convenience over the C ABI: allocation and pointer marshalling.

PyTorch provides device memory and streams only; every step of the layer runs
in libmoe_b300.so through the C entry points of `_lib`.
"""
from __future__ import annotations

import torch

from . import _lib
from .inputs import LayerConfig

ACT_CODES = {"relu": _lib.MOE_ACT_RELU, "gelu_tanh": _lib.MOE_ACT_GELU_TANH,
             "gelu_erf": _lib.MOE_ACT_GELU_ERF, "swiglu": _lib.MOE_ACT_SWIGLU}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_lib.moe_status_string(status)} ({status})")
        self.status = status


def check(status: int, where: str = "moe") -> None:
    if status != _lib.MOE_OK:
        raise MoEError(status, where)


def make_params(cfg: LayerConfig, *, flags: int = 0, residual_mode: int | None = None,
                T: int | None = None) -> _lib.moe_params_t:
    return _lib.moe_params_t(
        T=cfg.T if T is None else T, d_model=cfg.d, d_ff=cfg.F, E=cfg.E, k=cfg.k, n_shared=cfg.S,
        capacity_factor=0.0 if cfg.cf is None else float(cfg.cf),
        renormalize=int(cfg.renormalize),
        residual_mode=cfg.residual_mode if residual_mode is None else residual_mode,
        act=ACT_CODES[cfg.act], dtype=_lib.MOE_BF16 if cfg.dtype == "bf16" else _lib.MOE_F32,
        flags=flags, noisy_gating=int(cfg.noisy), noise_min_std=float(cfg.noise_min_std),
        weight_format={"int8": _lib.MOE_WEIGHTS_INT8, "int4": _lib.MOE_WEIGHTS_INT4}.get(cfg.weights,
                                                                                         _lib.MOE_WEIGHTS_DTYPE))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class MoELayer:
    """Outputs and workspace for one layer configuration, preallocated on `device`.

    `run()` is one C call (moe_forward by default) on the current torch stream.
    """

    def __init__(self, cfg: LayerConfig, weights: dict, device="cuda", *, flags: int = 0,
                 residual_mode: int | None = None, want_logits: bool = False,
                 want_probs: bool = False, want_perm: bool = True, ep_ranks: int | None = None,
                 prepared_router: bool = False):
        self.cfg = cfg
        self.device = torch.device(device)
        self.params = make_params(cfg, flags=flags, residual_mode=residual_mode)
        # ep_ranks = G: the layer runs expert-parallel over G ranks emulated on this GPU
        # (moe_forward_ep); only the whole forward is available then
        self.ep_ranks = ep_ranks
        if ep_ranks is None:
            st, nbytes = _lib.moe_workspace_size(self.params)
            check(st, "moe_workspace_size")
        else:
            st, nbytes = _lib.moe_ep_workspace_size(self.params, ep_ranks)
            check(st, "moe_ep_workspace_size")
        self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        self.workspace_bytes = nbytes
        self.weights = {k: (None if v is None else v.contiguous()) for k, v in weights.items()}
        T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
        dev = self.device
        self.out = {
            "y": torch.empty(T, d, dtype=cfg.torch_dtype, device=dev),
            "expert_idx": torch.empty(T, k, dtype=torch.int32, device=dev),
            "gates": torch.empty(T, k, dtype=torch.float32, device=dev),
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "dropped": torch.empty(T, k, dtype=torch.uint8, device=dev),
            "aux": torch.empty(1, dtype=torch.float32, device=dev),
            "logits": torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None,
            "probs": torch.empty(T, E, dtype=torch.float32, device=dev) if want_probs else None,
            "perm_row": torch.empty(T, k, dtype=torch.int32, device=dev) if want_perm else None,
        }
        w = self.weights
        self.inputs = _lib.moe_inputs_t(
            x=_ptr(w["x"]), W_gate=_ptr(w["W_gate"]), b_gate=_ptr(w.get("b_gate")), W1=_ptr(w["W1"]),
            W3=_ptr(w.get("W3")), W2=_ptr(w["W2"]), b1=_ptr(w.get("b1")), b2=_ptr(w.get("b2")),
            W_noise=_ptr(w.get("W_noise")), b_noise=_ptr(w.get("b_noise")),
            noise_eps=_ptr(w.get("noise_eps")), W1_scale=_ptr(w.get("W1_scale")),
            W3_scale=_ptr(w.get("W3_scale")), W2_scale=_ptr(w.get("W2_scale")))
        # prepared_router: split the router weights once (moe_prepare_router_weights) instead
        # of on every call; the buffer stays valid until the router weights change
        self.router_weights = None
        if prepared_router:
            self.prepare_router()
        o = self.out
        self.outputs = _lib.moe_outputs_t(
            y=_ptr(o["y"]), expert_idx=_ptr(o["expert_idx"]), gates=_ptr(o["gates"]),
            counts=_ptr(o["counts"]), dropped=_ptr(o["dropped"]), aux=_ptr(o["aux"]),
            logits=_ptr(o["logits"]), probs=_ptr(o["probs"]), perm_row=_ptr(o["perm_row"]))

    def prepare_router(self, stream=None) -> None:
        """(Re)make the split router weights from the current W_gate (and W_noise)."""
        st, nbytes = _lib.moe_router_weights_size(self.params)
        check(st, "moe_router_weights_size")
        if self.router_weights is None or self.router_weights.numel() < nbytes:
            self.router_weights = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.device)
        w = self.weights
        check(_lib.moe_prepare_router_weights(self.params, w["W_gate"].data_ptr(), _ptr(w.get("W_noise")),
                                              self.router_weights.data_ptr(), nbytes, _stream_handle(stream)),
              "moe_prepare_router_weights")
        self.inputs.router_weights = self.router_weights.data_ptr()

    def set_x(self, x: torch.Tensor) -> None:
        """Point the layer at a new [T, d] input (kept alive by the layer)."""
        x = x.contiguous()
        self.weights["x"] = x
        self.inputs.x = x.data_ptr()

    def run(self, stage: str = "moe_forward", stream=None) -> dict:
        if self.ep_ranks is not None:
            if stage != "moe_forward":
                raise ValueError("an expert-parallel layer runs the whole forward only")
            check(_lib.moe_forward_ep(self.params, self.ep_ranks, self.inputs, self.outputs,
                                      self.workspace.data_ptr(), self.workspace_bytes,
                                      _stream_handle(stream)), "moe_forward_ep")
            return self.out
        fn = getattr(_lib, stage)
        check(fn(self.params, self.inputs, self.outputs, self.workspace.data_ptr(),
                 self.workspace_bytes, _stream_handle(stream)), stage)
        return self.out

    def backward(self, dy: torch.Tensor, d_aux: float = 0.0, stream=None) -> dict:
        """moe_backward for the last run() of this layer (needs MOE_FLAG_TRAINING).

        Allocates the gradient arrays on first use; returns them by input name."""
        if not (self.params.flags & _lib.MOE_FLAG_TRAINING):
            raise ValueError("the layer was built without MOE_FLAG_TRAINING")
        cfg, dev, w = self.cfg, self.device, self.weights
        if not hasattr(self, "grads"):
            ES = cfg.E + cfg.S
            dt = cfg.torch_dtype
            f32 = torch.float32
            like = lambda key, shape, dtype: (torch.empty(shape, dtype=dtype, device=dev)  # noqa: E731
                                              if w.get(key) is not None else None)
            self.grads = {
                "dx": torch.empty(cfg.T, cfg.d, dtype=dt, device=dev),
                "dW_gate": torch.empty(cfg.E, cfg.d, dtype=f32, device=dev),
                "db_gate": like("b_gate", (cfg.E,), f32),
                "dW1": torch.empty(ES, cfg.F, cfg.d, dtype=dt, device=dev),
                "dW3": like("W3", (ES, cfg.F, cfg.d), dt),
                "dW2": torch.empty(ES, cfg.d, cfg.F, dtype=dt, device=dev),
                "db1": like("b1", (ES, cfg.F), dt),
                "db2": like("b2", (ES, cfg.d), dt),
                "dW_noise": like("W_noise", (cfg.E, cfg.d), f32),
                "db_noise": like("b_noise", (cfg.E,), f32),
            }
            g = self.grads
            self._grads_c = _lib.moe_grads_t(**{k: _ptr(v) for k, v in g.items()})
        dy = dy.contiguous()
        self._dy = dy  # alive until the next call
        check(_lib.moe_backward(self.params, self.inputs, self.outputs, dy.data_ptr(), float(d_aux),
                                self._grads_c, self.workspace.data_ptr(), self.workspace_bytes,
                                _stream_handle(stream)), "moe_backward")
        return self.grads

    def device_status(self, stream=None) -> int:
        return _lib.moe_last_device_status(self.workspace.data_ptr(), self.workspace_bytes,
                                           _stream_handle(stream))


def quantize_int8(w: torch.Tensor, stream=None):
    """Per-row int8 quantisation of a [..., cols] device tensor (moe_quantize_int8):
    returns (q int8 of the same shape, scale fp32 of shape [...])."""
    w = w.contiguous()
    cols = w.shape[-1]
    rows = w.numel() // cols
    q = torch.empty(w.shape, dtype=torch.int8, device=w.device)
    scale = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    dt = _lib.MOE_BF16 if w.dtype == torch.bfloat16 else _lib.MOE_F32
    check(_lib.moe_quantize_int8(w.data_ptr(), dt, rows, cols, q.data_ptr(), scale.data_ptr(),
                                 _stream_handle(stream)), "moe_quantize_int8")
    return q, scale


def quantize_int4(w: torch.Tensor, stream=None):
    """Group-wise 4-bit quantisation of a [..., cols] device tensor (moe_quantize_int4):
    returns (q uint8 [..., cols / 2], two values per byte; scale fp32 [..., cols / 128])."""
    w = w.contiguous()
    cols = w.shape[-1]
    rows = w.numel() // cols
    q = torch.empty((*w.shape[:-1], cols // 2), dtype=torch.uint8, device=w.device)
    scale = torch.empty((*w.shape[:-1], cols // _lib.MOE_INT4_GROUP), dtype=torch.float32, device=w.device)
    dt = _lib.MOE_BF16 if w.dtype == torch.bfloat16 else _lib.MOE_F32
    check(_lib.moe_quantize_int4(w.data_ptr(), dt, rows, cols, q.data_ptr(), scale.data_ptr(),
                                 _stream_handle(stream)), "moe_quantize_int4")
    return q, scale


def quantize_expert_weights(weights: dict, stream=None, bits: int = 8) -> dict:
    """The layer's inputs with W1, W3, W2 replaced by int8 + per-row scales (bits = 8)
    or packed 4-bit values + group scales (bits = 4)."""
    quant = {8: quantize_int8, 4: quantize_int4}[bits]
    out = dict(weights)
    for k in ("W1", "W3", "W2"):
        if weights.get(k) is not None:
            out[k], out[k + "_scale"] = quant(weights[k], stream)
    return out


def forward(cfg: LayerConfig, weights: dict, **kw) -> dict:
    """One-shot layer forward: allocate, run moe_forward, return the outputs."""
    layer = MoELayer(cfg, weights, device=weights["x"].device, **kw)
    return layer.run()
