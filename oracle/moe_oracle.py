"""fp64 CPU oracle for the sparse MoE FFN forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA library:
the arithmetic lives in ``moe_oracle.c`` (plain double-precision loops over
tokens and experts, written from the pages' definitions); this wrapper only
marshals arrays and chains the steps in the pages' order:

1. router logits, 2. softmax, 3. top-k, 4. gates, 5. counts, 6. capacity in
token order, 7-9. expert FFNs, shared experts and the gate-weighted combine,
plus the Switch load-balancing statistic N * sum_i f_i P_i.

Sources are cited by page title and section in ``moe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "libmoe_oracle.so")

F64, F32, BF16 = 0, 1, 2
ACTS = {"relu": 0, "gelu_tanh": 1, "gelu_erf": 2, "swiglu": 3}

_lib_handle = None


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so next to it (gcc, OpenMP)."""
    stamp = _SO + ".srchash"
    fresh = (os.path.exists(_SO) and os.path.exists(stamp)
             and open(stamp).read().strip() == _src_hash())
    if force or not fresh:
        cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
               "-o", _SO, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        with open(stamp, "w") as f:
            f.write(_src_hash())
    return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        L = ctypes.CDLL(_SO)
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_capacity.restype = ctypes.c_longlong
        L.orc_capacity.argtypes = [ctypes.c_longlong, ctypes.c_longlong, dbl]
        L.orc_router_logits.restype = None
        L.orc_router_logits.argtypes = [i32, i32, i32, vp, i32, vp, i32, vp, i32, vp]
        L.orc_softplus.restype = dbl
        L.orc_softplus.argtypes = [dbl]
        L.orc_noisy_logits.restype = None
        L.orc_noisy_logits.argtypes = [i32, i32, vp, vp, vp, i32, dbl, vp]
        L.orc_softmax.restype = None
        L.orc_softmax.argtypes = [i32, i32, vp, vp]
        L.orc_topk.restype = None
        L.orc_topk.argtypes = [i32, i32, i32, vp, vp]
        L.orc_gates.restype = None
        L.orc_gates.argtypes = [i32, i32, i32, vp, vp, i32, vp]
        L.orc_dispatch.restype = None
        L.orc_dispatch.argtypes = [i32, i32, i32, vp, ctypes.c_longlong, vp, vp, vp, vp]
        L.orc_aux.restype = dbl
        L.orc_aux.argtypes = [i32, i32, i32, vp, vp]
        L.orc_act.restype = dbl
        L.orc_act.argtypes = [i32, dbl]
        L.orc_output_rows.restype = None
        L.orc_output_rows.argtypes = [i32] * 8 + [vp, i32, vp, vp, vp, i32, vp, vp, i32,
                                                  vp, vp, vp, i32, vp, vp]
        L.orc_act_grad.restype = dbl
        L.orc_act_grad.argtypes = [i32, dbl]
        L.orc_backward.restype = None
        L.orc_backward.argtypes = ([i32] * 9 + [vp, i32, vp, i32, vp, i32, vp, vp, vp, i32, vp, vp, i32,
                                                vp, vp, vp, i32, dbl, vp, vp, vp, dbl] + [vp] * 10)
        L.orc_quantize_int8.restype = None
        L.orc_quantize_int8.argtypes = [i32, i32, vp, i32, vp, vp]
        L.orc_num_threads.restype = i32
        L.orc_num_threads.argtypes = []
        L.orc_quantize_int4.restype = None
        L.orc_quantize_int4.argtypes = [i32, i32, i32, vp, i32, vp, vp]
        L.orc_ep_exchange.restype = None
        L.orc_ep_exchange.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.orc_expert_apply.restype = None
        L.orc_expert_apply.argtypes = [i32, i32, i32, vp, i32, vp, vp, vp, i32, vp, vp, i32, i32, vp, vp, vp]
        L.orc_ep_combine.restype = None
        L.orc_ep_combine.argtypes = [i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp]
        L.orc_ep_aux.restype = dbl
        L.orc_ep_aux.argtypes = [i32, i32, i32, i32, vp, vp]
        _lib_handle = L
    return _lib_handle


# --------------------------------------------------------------------------
# array marshalling (no arithmetic)

def _as_array(a):
    """Return (contiguous numpy array kept alive, storage code).

    Accepts numpy arrays (float64/float32) and CPU torch tensors
    (float64/float32/bfloat16).  bf16 tensors are passed as their raw 16-bit
    patterns; the C side widens them exactly.
    """
    if a is None:
        return None, F64
    if isinstance(a, np.ndarray):
        if a.dtype == np.float64:
            return np.ascontiguousarray(a), F64
        if a.dtype == np.float32:
            return np.ascontiguousarray(a), F32
        raise TypeError(f"unsupported numpy dtype {a.dtype}")
    import torch  # only for tensors handed in by the caller
    if not isinstance(a, torch.Tensor):
        return _as_array(np.asarray(a, dtype=np.float64))
    t = a.detach().to("cpu").contiguous()
    if t.dtype == torch.float64:
        return t.numpy(), F64
    if t.dtype == torch.float32:
        return t.numpy(), F32
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy(), BF16
    raise TypeError(f"unsupported tensor dtype {t.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# --------------------------------------------------------------------------
# single steps

def capacity(T: int, E: int, cf) -> int:
    """floor(T*cf/E); -1 when cf is None or <= 0 (no limit)."""
    return int(_lib().orc_capacity(T, E, -1.0 if cf is None else float(cf)))


def router_logits(x, Wg, bg=None) -> np.ndarray:
    xa, xc = _as_array(x)
    wa, wc = _as_array(Wg)
    ba, bc = _as_array(bg)
    T, d = xa.shape
    E = wa.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _lib().orc_router_logits(T, d, E, _ptr(xa), xc, _ptr(wa), wc, _ptr(ba), bc, _ptr(out))
    return out


def softplus(z: float) -> float:
    return float(_lib().orc_softplus(float(z)))


def noisy_logits(clean, noise_logits, eps, min_std: float = 0.0) -> np.ndarray:
    """clean + eps * (softplus(noise_logits) + min_std), elementwise, in fp64."""
    ca = np.ascontiguousarray(np.asarray(clean, dtype=np.float64))
    na = np.ascontiguousarray(np.asarray(noise_logits, dtype=np.float64))
    ea, ec = _as_array(eps)
    if ca.shape != na.shape or ea.shape != ca.shape:
        raise ValueError("clean, noise_logits and eps must have the same [T,E] shape")
    T, E = ca.shape
    out = np.empty_like(ca)
    _lib().orc_noisy_logits(T, E, _ptr(ca), _ptr(na), _ptr(ea), ec, float(min_std), _ptr(out))
    return out


def softmax(logits) -> np.ndarray:
    la = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T, E = la.shape
    out = np.empty_like(la)
    _lib().orc_softmax(T, E, _ptr(la), _ptr(out))
    return out


def topk(scores, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, descending; ties -> lower index.

    ``scores`` may be fp32 (e.g. device logits): the comparison is exact after
    widening to double, so the selection is the one fp32 comparisons make.
    """
    sa = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    T, E = sa.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((T, k), dtype=np.int32)
    _lib().orc_topk(T, E, k, _ptr(sa), _ptr(idx))
    return idx


def gates(probs, idx, renormalize: bool) -> np.ndarray:
    pa = np.ascontiguousarray(np.asarray(probs, dtype=np.float64))
    ia = _i32(idx)
    T, E = pa.shape
    k = ia.shape[1]
    out = np.empty((T, k), dtype=np.float64)
    _lib().orc_gates(T, E, k, _ptr(pa), _ptr(ia), int(bool(renormalize)), _ptr(out))
    return out


@dataclass
class Dispatch:
    counts: np.ndarray    # [E] int32, router selection before drops
    pos: np.ndarray       # [T,k] int32, token-order position inside the expert
    dropped: np.ndarray   # [T,k] uint8
    perm_row: np.ndarray  # [T,k] int32, unpadded expert-contiguous row or -1


def dispatch(idx, E: int, C: int) -> Dispatch:
    ia = _i32(idx)
    T, k = ia.shape
    counts = np.empty(E, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    dropped = np.empty((T, k), dtype=np.uint8)
    perm_row = np.empty((T, k), dtype=np.int32)
    _lib().orc_dispatch(T, E, k, _ptr(ia), int(C), _ptr(counts), _ptr(pos), _ptr(dropped),
                        _ptr(perm_row))
    return Dispatch(counts, pos, dropped, perm_row)


def aux(counts, probs, k: int) -> float:
    ca = _i32(counts)
    pa = np.ascontiguousarray(np.asarray(probs, dtype=np.float64))
    T, E = pa.shape
    return float(_lib().orc_aux(T, E, k, _ptr(ca), _ptr(pa)))


def act(name: str, z: float) -> float:
    return float(_lib().orc_act(ACTS[name], float(z)))


def output_rows(x, W1, W3, W2, b1, b2, idx, gate_vals, dropped, *, E: int, S: int,
                act_name: str, residual_mode: int, tokens=None) -> np.ndarray:
    """Layer output (fp64) for the listed tokens (all tokens if None)."""
    xa, xc = _as_array(x)
    w1, wc = _as_array(W1)
    w3, wc3 = _as_array(W3)
    w2, wc2 = _as_array(W2)
    if W3 is not None and wc3 != wc or wc2 != wc:
        raise TypeError("W1, W3 and W2 must share a storage type")
    ba1, bc = _as_array(b1)
    ba2, bc2 = _as_array(b2)
    if b1 is not None and b2 is not None and bc != bc2:
        raise TypeError("b1 and b2 must share a storage type")
    if b1 is None:
        bc = bc2
    T, d = xa.shape
    F = w1.shape[1]
    ia = _i32(idx)
    k = ia.shape[1]
    ga = np.ascontiguousarray(np.asarray(gate_vals, dtype=np.float64))
    da = np.ascontiguousarray(np.asarray(dropped, dtype=np.uint8))
    tok = _i32(np.arange(T) if tokens is None else tokens)
    y = np.empty((tok.shape[0], d), dtype=np.float64)
    _lib().orc_output_rows(T, d, F, E, S, k, ACTS[act_name], int(residual_mode),
                           _ptr(xa), xc, _ptr(w1), _ptr(w3), _ptr(w2), wc,
                           _ptr(ba1), _ptr(ba2), bc,
                           _ptr(ia), _ptr(ga), _ptr(da), tok.shape[0], _ptr(tok), _ptr(y))
    return y


def act_grad(name: str, z: float) -> float:
    return float(_lib().orc_act_grad(ACTS[name], float(z)))


def backward(x, Wg, bg, W1, W3, W2, b1, b2, *, idx, dropped, dy, d_aux: float, E: int, S: int,
             act_name: str, renormalize: bool, residual_mode: int, noise=None) -> dict:
    """Gradients (fp64) of L with dL/dy = dy and dL/daux = d_aux, the forward's
    top-k choice ``idx`` and capacity drops ``dropped`` held fixed.

    Returns dx, dW_gate, db_gate, dW1, dW3, dW2, db1, db2, dW_noise, db_noise
    (None for inputs the layer does not have)."""
    xa, xc = _as_array(x)
    ga, gc = _as_array(Wg)
    gba, gbc = _as_array(bg)
    w1, wc = _as_array(W1)
    w3, _ = _as_array(W3)
    w2, _ = _as_array(W2)
    ba1, bc = _as_array(b1)
    ba2, bc2 = _as_array(b2)
    if b1 is None:
        bc = bc2
    if noise is not None:
        Wn, bn, eps, min_std = noise
        na, nc = _as_array(Wn)
        nba, nbc = _as_array(bn)
        ea, ec = _as_array(eps)
        if (bn is not None and nbc != nc) or ec != nc:
            raise TypeError("W_noise, b_noise and eps must share a storage type")
    else:
        na = nba = ea = None
        nc, min_std = 0, 0.0
    T, d = xa.shape
    F = w1.shape[1]
    ia = _i32(idx)
    k = ia.shape[1]
    da = np.ascontiguousarray(np.asarray(dropped, dtype=np.uint8))
    if not isinstance(dy, np.ndarray):
        import torch  # a tensor handed in by the caller
        dy = dy.detach().to("cpu", torch.float64).numpy()
    dya = np.ascontiguousarray(dy, dtype=np.float64)
    ES = E + S
    out = {"dx": np.empty((T, d)), "dW_gate": np.empty((E, d)),
           "db_gate": np.empty(E) if bg is not None else None,
           "dW1": np.empty((ES, F, d)), "dW3": np.empty((ES, F, d)) if W3 is not None else None,
           "dW2": np.empty((ES, d, F)), "db1": np.empty((ES, F)) if b1 is not None else None,
           "db2": np.empty((ES, d)) if b2 is not None else None,
           "dW_noise": np.empty((E, d)) if noise is not None else None,
           "db_noise": np.empty(E) if noise is not None and noise[1] is not None else None}
    o = out
    _lib().orc_backward(T, d, F, E, S, k, ACTS[act_name], int(bool(renormalize)), int(residual_mode),
                        _ptr(xa), xc, _ptr(ga), gc, _ptr(gba), gbc, _ptr(w1), _ptr(w3), _ptr(w2), wc,
                        _ptr(ba1), _ptr(ba2), bc, _ptr(na), _ptr(nba), _ptr(ea), nc, float(min_std),
                        _ptr(ia), _ptr(da), _ptr(dya), float(d_aux),
                        _ptr(o["dx"]), _ptr(o["dW_gate"]), _ptr(o["db_gate"]), _ptr(o["dW1"]),
                        _ptr(o["dW3"]), _ptr(o["dW2"]), _ptr(o["db1"]), _ptr(o["db2"]),
                        _ptr(o["dW_noise"]), _ptr(o["db_noise"]))
    return out


def quantize_int8(w):
    """Per-row symmetric int8 quantisation of a 2-D array: (q int8, scale fp32)."""
    wa, wc = _as_array(w)
    rows, cols = wa.shape
    q = np.empty((rows, cols), dtype=np.int8)
    sc = np.empty(rows, dtype=np.float32)
    _lib().orc_quantize_int8(rows, cols, _ptr(wa), wc, _ptr(q), _ptr(sc))
    return q, sc


def dequantize_int8(q, scale):
    """q * scale per row, exactly, in fp64."""
    return np.asarray(q, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


INT4_GROUP = 128  # columns per scale group of the 4-bit weights


def quantize_int4(w, group: int = INT4_GROUP):
    """Group-wise symmetric 4-bit quantisation of a 2-D array: (packed uint8 [rows, cols/2],
    scale fp32 [rows, cols/group]); column 2i in the low nibble, 2i+1 in the high one."""
    wa, wc = _as_array(w)
    rows, cols = wa.shape
    if cols % group or group % 2:
        raise ValueError("cols must be a multiple of an even group size")
    packed = np.zeros((rows, cols // 2), dtype=np.uint8)
    sc = np.empty((rows, cols // group), dtype=np.float32)
    _lib().orc_quantize_int4(rows, cols, group, _ptr(wa), wc, _ptr(packed), _ptr(sc))
    return packed, sc


def unpack_int4(packed) -> np.ndarray:
    """The signed 4-bit values of a packed array (marshalling: two nibbles per byte)."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int8)
    hi = (p >> 4).astype(np.int8)
    q = np.stack([lo, hi], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    return np.where(q > 7, q - 16, q).astype(np.int8)


def dequantize_int4(packed, scale, group: int = INT4_GROUP):
    """q * scale of every element, exactly, in fp64."""
    q = unpack_int4(packed).astype(np.float64)
    s = np.repeat(np.asarray(scale, dtype=np.float64), group, axis=-1)
    return q * s


def num_threads() -> int:
    return int(_lib().orc_num_threads())


# --------------------------------------------------------------------------
# chained steps

@dataclass
class Routing:
    logits: np.ndarray
    probs: np.ndarray
    idx: np.ndarray
    gates: np.ndarray
    counts: np.ndarray
    pos: np.ndarray
    dropped: np.ndarray
    perm_row: np.ndarray
    aux: float
    C: int


def route_from_logits(logits, *, k: int, renormalize: bool, cf) -> Routing:
    """Steps 2-6 and the aux statistic on a given [T,E] logits array.

    Fed with the device's fp32 logits this is the bit-exact re-run of the
    selection, counts, capacity drops and permutation order.
    """
    la = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    T, E = la.shape
    probs = softmax(la)
    idx = topk(la, k)
    g = gates(probs, idx, renormalize)
    C = capacity(T, E, cf)
    dsp = dispatch(idx, E, C)
    a = aux(dsp.counts, probs, k)
    return Routing(la, probs, idx, g, dsp.counts, dsp.pos, dsp.dropped, dsp.perm_row, a, C)


def route(x, Wg, bg=None, *, k: int, renormalize: bool, cf, noise=None) -> Routing:
    """Steps 1-6 and the aux statistic in fp64.

    ``noise`` = (W_noise, b_noise or None, eps, min_std) selects noisy top-k
    gating: every later step sees the noisy logits.
    """
    logits = router_logits(x, Wg, bg)
    if noise is not None:
        Wn, bn, eps, min_std = noise
        logits = noisy_logits(logits, router_logits(x, Wn, bn), eps, min_std)
    return route_from_logits(logits, k=k, renormalize=renormalize, cf=cf)


def forward(x, Wg, bg, W1, W3, W2, b1, b2, *, E: int, S: int, k: int, act_name: str,
            renormalize: bool, cf, residual_mode: int = 0, tokens=None, noise=None):
    """Whole layer in fp64: returns (y rows for ``tokens``, Routing)."""
    r = route(x, Wg, bg, k=k, renormalize=renormalize, cf=cf, noise=noise)
    y = output_rows(x, W1, W3, W2, b1, b2, r.idx, r.gates, r.dropped, E=E, S=S,
                    act_name=act_name, residual_mode=residual_mode, tokens=tokens)
    return y, r


# --------------------------------------------------------------------------
# expert parallelism over G ranks (host-side emulation of the exchange)

def shard_bounds(T: int, G: int) -> list:
    """Token shard of each rank: rank r holds [b[r], b[r+1]), b[r] = floor(r T / G)."""
    return [r * T // G for r in range(G + 1)]


@dataclass
class EPExchange:
    counts_rank: np.ndarray  # [G, E] int32, each rank's slots per expert before drops
    dropped: np.ndarray      # [T, k] uint8, per-shard capacity drops
    recv_row: np.ndarray     # [T, k] int32, row in the concatenated receive buffers or -1
    recv_rows: np.ndarray    # [G] int32, rows each rank receives
    recv_slot: np.ndarray    # [sum recv_rows] int32, slot t*k+j held by each received row


def ep_exchange(idx, E: int, G: int, C_rank) -> EPExchange:
    ia = _i32(idx)
    T, k = ia.shape
    if G < 1 or E % G != 0:
        raise ValueError("need E to be a multiple of G")
    cr = np.ascontiguousarray(np.asarray(C_rank, dtype=np.int64))
    if cr.shape != (G,):
        raise ValueError("one capacity per rank")
    counts_rank = np.empty((G, E), dtype=np.int32)
    dropped = np.empty((T, k), dtype=np.uint8)
    recv_row = np.empty((T, k), dtype=np.int32)
    recv_rows = np.empty(G, dtype=np.int32)
    recv_slot = np.full(max(T * k, 1), -1, dtype=np.int32)
    _lib().orc_ep_exchange(T, E, k, G, _ptr(ia), _ptr(cr), _ptr(counts_rank), _ptr(dropped),
                           _ptr(recv_row), _ptr(recv_rows), _ptr(recv_slot))
    return EPExchange(counts_rank, dropped, recv_row, recv_rows, recv_slot[: int(recv_rows.sum())])


def expert_apply(x, W1, W3, W2, b1, b2, tokens, experts, *, act_name: str) -> np.ndarray:
    """out[r] = FFN_{experts[r]}(x[tokens[r]]) in fp64."""
    xa, xc = _as_array(x)
    w1, wc = _as_array(W1)
    w3, _ = _as_array(W3)
    w2, _ = _as_array(W2)
    ba1, bc = _as_array(b1)
    ba2, bc2 = _as_array(b2)
    if b1 is None:
        bc = bc2
    d = xa.shape[1]
    F = w1.shape[1]
    tok = _i32(tokens)
    exp = _i32(experts)
    out = np.empty((tok.shape[0], d), dtype=np.float64)
    if tok.shape[0]:
        _lib().orc_expert_apply(d, F, ACTS[act_name], _ptr(xa), xc, _ptr(w1), _ptr(w3), _ptr(w2), wc,
                                _ptr(ba1), _ptr(ba2), bc, tok.shape[0], _ptr(tok), _ptr(exp), _ptr(out))
    return out


def combine_rows(x, gates, dropped, row_of, o, *, S: int = 0, ys=None, residual_mode: int = 0,
                 tokens=None) -> np.ndarray:
    """The combine for the listed tokens: sum over kept slots (slot order) of
    gates[t,j] * o[row_of[t,j]] + the shared outputs ys [S, T, d] + pass(t) x[t]."""
    xa, xc = _as_array(x)
    T, d = xa.shape
    ga = np.ascontiguousarray(np.asarray(gates, dtype=np.float64))
    k = ga.shape[1]
    da = np.ascontiguousarray(np.asarray(dropped, dtype=np.uint8))
    ra = _i32(row_of)
    oa = np.ascontiguousarray(np.asarray(o, dtype=np.float64))
    tok = np.arange(T, dtype=np.int32) if tokens is None else _i32(tokens)
    ysa = None if ys is None else np.ascontiguousarray(np.asarray(ys, dtype=np.float64))
    y = np.empty((tok.shape[0], d), dtype=np.float64)
    _lib().orc_ep_combine(T, d, k, S, int(residual_mode), _ptr(xa), xc, _ptr(ga), _ptr(da), _ptr(ra), _ptr(oa),
                          _ptr(ysa) if ysa is not None else None, tok.shape[0], _ptr(tok), _ptr(y))
    return y


def ep_aux(counts_rank, probs, k: int) -> float:
    ca = _i32(counts_rank)
    pa = np.ascontiguousarray(np.asarray(probs, dtype=np.float64))
    T, E = pa.shape
    return float(_lib().orc_ep_aux(T, E, k, ca.shape[0], _ptr(ca), _ptr(pa)))


@dataclass
class EPResult:
    logits: np.ndarray
    probs: np.ndarray
    idx: np.ndarray
    gates: np.ndarray
    counts: np.ndarray       # [E] all ranks' slots per expert before drops
    ex: EPExchange
    C_rank: list
    aux: float
    y: np.ndarray | None     # rows of the listed tokens


def ep_forward(x, Wg, bg, W1, W3, W2, b1, b2, *, E: int, S: int, k: int, G: int, act_name: str,
               renormalize: bool, cf, residual_mode: int = 0, tokens=None, noise=None,
               logits=None) -> EPResult:
    """The layer computed rank by rank over G ranks, in fp64.

    Each rank routes its token shard (the router is per token, so ``logits`` --
    e.g. the device's -- may be given for all T tokens at once), applies the
    capacity rule to its shard alone, sends its kept slots to the experts'
    owners, the owners run their experts on the rows they received, the
    outputs return, and each rank combines its tokens.  ``tokens`` limits the
    expert work and y to the listed tokens (None: all)."""
    xa, _ = _as_array(x)
    T = xa.shape[0]
    if logits is None:
        la = router_logits(x, Wg, bg)
        if noise is not None:
            Wn, bn, eps, min_std = noise
            la = noisy_logits(la, router_logits(x, Wn, bn), eps, min_std)
    else:
        la = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    probs = softmax(la)
    idx = topk(la, k)
    g = gates(probs, idx, renormalize)
    b = shard_bounds(T, G)
    C_rank = [capacity(b[r + 1] - b[r], E, cf) for r in range(G)]
    ex = ep_exchange(idx, E, G, C_rank)
    tok = np.arange(T, dtype=np.int32) if tokens is None else _i32(tokens)
    # the owners compute the received rows that the listed tokens need
    rows_needed = ex.recv_row[tok].reshape(-1)
    rows_needed = np.unique(rows_needed[rows_needed >= 0])
    o = np.zeros((max(int(ex.recv_rows.sum()), 1), xa.shape[1]), dtype=np.float64)
    if rows_needed.size:
        slot = ex.recv_slot[rows_needed]
        o[rows_needed] = expert_apply(x, W1, W3, W2, b1, b2, slot // k, idx.reshape(-1)[slot],
                                      act_name=act_name)
    ys = None
    if S > 0:  # each rank applies the shared experts to its own tokens
        ys = np.zeros((S, T, xa.shape[1]), dtype=np.float64)
        for sh in range(S):
            ys[sh, tok] = expert_apply(x, W1, W3, W2, b1, b2, tok, np.full(tok.shape, E + sh),
                                       act_name=act_name)
    xa2, xc = _as_array(x)
    y = np.empty((tok.shape[0], xa.shape[1]), dtype=np.float64)
    ga = np.ascontiguousarray(g, dtype=np.float64)
    _lib().orc_ep_combine(T, xa.shape[1], k, S, int(residual_mode), _ptr(xa2), xc, _ptr(ga),
                          _ptr(ex.dropped), _ptr(ex.recv_row), _ptr(o),
                          _ptr(ys) if ys is not None else None, tok.shape[0], _ptr(tok), _ptr(y))
    counts = ex.counts_rank.sum(axis=0).astype(np.int32)
    return EPResult(la, probs, idx, g, counts, ex, C_rank, ep_aux(ex.counts_rank, probs, k), y)
