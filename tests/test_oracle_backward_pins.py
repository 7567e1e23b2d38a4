"""Pins for the oracle's backward pass (CPU only).

The analytic gradients are checked against central finite differences of the
oracle's forward (itself pinned in test_oracle_pins.py), taken in fp64 with the
routing decisions verified unchanged at every perturbed point; against the
dense-MLP special case written with numpy matmuls; and against invariants of
the softmax Jacobian.  Shapes are small and non-square so that a transposed
operand, a dropped term or a wrong index fails.
"""
import numpy as np
import pytest

from oracle import moe_oracle as orc


def _layer(seed, *, T, d, E, k, F, S, act, bias, noisy, bg=True):
    rng = np.random.default_rng(seed)
    ES = E + S
    L = {
        "x": rng.standard_normal((T, d)),
        "Wg": rng.standard_normal((E, d)) * 0.7,
        "bg": rng.standard_normal(E) * 0.3 if bg else None,
        "W1": rng.standard_normal((ES, F, d)) * 0.5,
        "W3": rng.standard_normal((ES, F, d)) * 0.5 if act == "swiglu" else None,
        "W2": rng.standard_normal((ES, d, F)) * 0.5,
        "b1": rng.standard_normal((ES, F)) * 0.2 if bias else None,
        "b2": rng.standard_normal((ES, d)) * 0.2 if bias else None,
        "noise": ((rng.standard_normal((E, d)) * 0.5, rng.standard_normal(E), rng.standard_normal((T, E)), 0.01)
                  if noisy else None),
    }
    return L


def _loss(L, dy, d_aux, *, E, S, k, act, renorm, cf, mode, ref=None):
    y, r = orc.forward(L["x"], L["Wg"], L["bg"], L["W1"], L["W3"], L["W2"], L["b1"], L["b2"], E=E, S=S, k=k,
                       act_name=act, renormalize=renorm, cf=cf, residual_mode=mode, noise=L["noise"])
    if ref is not None:  # the discrete decisions must not move under the perturbation
        assert np.array_equal(r.idx, ref.idx) and np.array_equal(r.dropped, ref.dropped)
    return float((dy * y).sum() + d_aux * r.aux), r


def _fd(L, name, dy, d_aux, ref, kw, h=1e-6):
    """Central differences of the loss in every element of input `name`."""
    if name.startswith("noise."):
        j = {"W": 0, "b": 1}[name[6:]]
        arr = np.array(L["noise"][j], dtype=np.float64)

        def setter(a):
            n = list(L["noise"])
            n[j] = a
            return {**L, "noise": tuple(n)}
    else:
        arr = np.array(L[name], dtype=np.float64)

        def setter(a):
            return {**L, name: a}
    g = np.empty_like(arr)
    for i in np.ndindex(arr.shape):
        a = arr.copy()
        a[i] += h
        lp, _ = _loss(setter(a), dy, d_aux, ref=ref, **kw)
        a[i] -= 2 * h
        lm, _ = _loss(setter(a), dy, d_aux, ref=ref, **kw)
        g[i] = (lp - lm) / (2 * h)
    return g


CASES = {
    # name: (shape/act kwargs, routing kwargs)
    "gelu_tanh_noisy_renorm": (dict(T=7, d=5, E=4, k=2, F=3, S=0, act="gelu_tanh", bias=True, noisy=True),
                               dict(renorm=True, cf=None, mode=1)),
    "swiglu_shared_capacity": (dict(T=8, d=4, E=4, k=2, F=3, S=1, act="swiglu", bias=False, noisy=False),
                               dict(renorm=False, cf=0.75, mode=0)),
    "gelu_erf_top1_drops": (dict(T=9, d=3, E=3, k=1, F=4, S=0, act="gelu_erf", bias=True, noisy=False),
                            dict(renorm=False, cf=0.7, mode=0)),
    "relu_k3": (dict(T=5, d=4, E=5, k=3, F=6, S=0, act="relu", bias=True, noisy=True),
                dict(renorm=True, cf=None, mode=0)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_finite_differences(case):
    shape, route = CASES[case]
    L = _layer(3, **shape)
    E, S, k, act = shape["E"], shape["S"], shape["k"], shape["act"]
    kw = dict(E=E, S=S, k=k, act=act, **route)
    rng = np.random.default_rng(4)
    dy = rng.standard_normal((shape["T"], shape["d"]))
    d_aux = 0.37
    _, r = _loss(L, dy, d_aux, **kw)
    if act == "relu":  # stay away from the kink: every pre-activation is far from 0
        for t in range(shape["T"]):
            for e in list(r.idx[t]) + list(range(E, E + S)):
                z = L["W1"][e] @ L["x"][t] + (L["b1"][e] if L["b1"] is not None else 0)
                assert np.abs(z).min() > 1e-3
    if route["cf"] is not None:
        assert r.dropped.any() and not r.dropped.all()  # the case exercises drops
    g = orc.backward(L["x"], L["Wg"], L["bg"], L["W1"], L["W3"], L["W2"], L["b1"], L["b2"], idx=r.idx,
                     dropped=r.dropped, dy=dy, d_aux=d_aux, E=E, S=S, act_name=act,
                     renormalize=route["renorm"], residual_mode=route["mode"], noise=L["noise"])
    names = {"dx": "x", "dW_gate": "Wg", "db_gate": "bg", "dW1": "W1", "dW3": "W3", "dW2": "W2",
             "db1": "b1", "db2": "b2", "dW_noise": "noise.W", "db_noise": "noise.b"}
    checked = 0
    for gname, pname in names.items():
        if g[gname] is None:
            continue
        num = _fd(L, pname, dy, d_aux, r, kw)
        np.testing.assert_allclose(g[gname], num, rtol=1e-6, atol=1e-7, err_msg=gname)
        checked += 1
    assert checked >= 6


def test_backward_single_expert_is_the_dense_mlp_gradient():
    # E = 1, k = 1, no capacity: the gate is softmax of one logit = 1, so y = W2 relu(W1 x + b1) + b2
    # and the router gets no gradient; the expert gradients are the textbook MLP ones
    rng = np.random.default_rng(5)
    T, d, F = 6, 5, 7
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((1, d))
    W1 = rng.standard_normal((1, F, d))
    W2 = rng.standard_normal((1, d, F))
    b1 = rng.standard_normal((1, F))
    b2 = rng.standard_normal((1, d))
    dy = rng.standard_normal((T, d))
    idx = np.zeros((T, 1), dtype=np.int32)
    g = orc.backward(x, Wg, None, W1, None, W2, b1, b2, idx=idx, dropped=np.zeros((T, 1), np.uint8), dy=dy,
                     d_aux=2.5, E=1, S=0, act_name="relu", renormalize=False, residual_mode=0)
    z = x @ W1[0].T + b1[0]
    h = np.maximum(z, 0)
    dh = dy @ W2[0]
    dz = dh * (z > 0)
    np.testing.assert_allclose(g["dW2"][0], dy.T @ h, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["db2"][0], dy.sum(0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW1"][0], dz.T @ x, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["db1"][0], dz.sum(0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dx"], dz @ W1[0], rtol=1e-12, atol=1e-12)
    assert np.abs(g["dW_gate"]).max() == 0.0


def test_router_bias_gradient_sums_to_zero_per_batch():
    # each token's logit gradient is p * (dp - <p, dp>), which sums to 0 over experts
    L = _layer(6, T=11, d=6, E=5, k=2, F=4, S=0, act="gelu_tanh", bias=True, noisy=True)
    y, r = orc.forward(L["x"], L["Wg"], L["bg"], L["W1"], None, L["W2"], L["b1"], L["b2"], E=5, S=0, k=2,
                       act_name="gelu_tanh", renormalize=True, cf=None, noise=L["noise"])
    dy = np.random.default_rng(7).standard_normal(y.shape)
    g = orc.backward(L["x"], L["Wg"], L["bg"], L["W1"], None, L["W2"], L["b1"], L["b2"], idx=r.idx,
                     dropped=r.dropped, dy=dy, d_aux=1.0, E=5, S=0, act_name="gelu_tanh", renormalize=True,
                     residual_mode=0, noise=L["noise"])
    assert abs(g["db_gate"].sum()) < 1e-12 * max(1.0, np.abs(g["db_gate"]).max())
    # and sum_e dW_gate[e] = 0 likewise (x factors out of the sum over experts)
    assert np.abs(g["dW_gate"].sum(0)).max() < 1e-12 * max(1.0, np.abs(g["dW_gate"]).max())


@pytest.mark.parametrize("act", ["relu", "gelu_tanh", "gelu_erf", "swiglu"])
def test_activation_derivatives(act):
    # central differences of the pinned activation functions
    for z in (-2.3, -0.4, 0.3, 1.7):
        h = 1e-6
        num = (orc.act(act, z + h) - orc.act(act, z - h)) / (2 * h)
        assert orc.act_grad(act, z) == pytest.approx(num, rel=1e-7, abs=1e-9)
