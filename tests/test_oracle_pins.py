"""Pins for the fp64 CPU oracle (CPU only).

Each test ties an oracle step to something other than the oracle itself: the
values the pages print, closed forms evaluated with mpmath, invariants,
brute-force enumeration, or an independent library routine (numpy matmul) on a
special case that reduces to plain linear algebra.  The cases use non-square
shapes so that a transposed operand, a dropped term or a wrong index fails.
"""
import itertools
import json
import os

import mpmath as mp
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
mp.mp.dps = 40


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _worked(k, renorm):
    """The 3-expert example embedded in the layer: d=1, x=[1], W_g=[[1],[2],[3]]
    gives logits [1,2,3]; expert e is ReLU(1*x)*10(e+1), i.e. outputs 10/20/30."""
    x = np.array([[1.0]])
    Wg = np.array([[1.0], [2.0], [3.0]])
    W1 = np.ones((3, 1, 1))
    W2 = np.array([10.0, 20.0, 30.0]).reshape(3, 1, 1)
    return orc.forward(x, Wg, None, W1, None, W2, None, None, E=3, S=0, k=k,
                       act_name="relu", renormalize=renorm, cf=None)


# ---------------------------------------------------------------- worked example

def test_worked_example_matches_page_numbers():
    g = _gold("worked_example.json")
    y, r = _worked(k=3, renorm=True)
    np.testing.assert_array_equal(r.logits[0], g["logits"])
    p = r.probs[0]
    # the page rounds each gate to two decimals and checks they sum to 1.00
    assert [round(v, 2) for v in p] == g["page_gates"]
    assert round(float(p.sum()), 2) == g["page_gate_sum"]
    # the page's denominator adds e^1, e^2, e^3 already rounded to 2 decimals
    den = float(mp.e ** 3) / p[2]
    assert abs(den - g["page_denominator"]) < 0.015
    assert [round(float(mp.e ** v), 2) for v in g["logits"]] == g["page_exp_terms"]
    # y = sum g_i e_i: the page's 25.8 is the exact value rounded to one decimal
    assert round(float(y[0, 0]), 1) == g["page_y"]
    # and the gates the oracle used are the full probabilities (k = E, renormalised)
    np.testing.assert_allclose(r.gates[0], p[r.idx[0]], rtol=0, atol=1e-15)


@pytest.mark.parametrize("k,renorm,expect", [
    # closed forms of the worked example (logits 1,2,3; outputs 10,20,30)
    (3, True, lambda E: (10 * E(1) + 20 * E(2) + 30 * E(3)) / (E(1) + E(2) + E(3))),
    (1, False, lambda E: 30 * E(3) / (E(1) + E(2) + E(3))),
    (1, True, lambda E: mp.mpf(30)),
    (2, True, lambda E: (30 * E(3) + 20 * E(2)) / (E(2) + E(3))),
    (2, False, lambda E: (30 * E(3) + 20 * E(2)) / (E(1) + E(2) + E(3))),
])
def test_worked_example_closed_forms(k, renorm, expect):
    y, _ = _worked(k=k, renorm=renorm)
    exact = float(expect(mp.exp))
    assert abs(y[0, 0] - exact) <= 1e-12 * abs(exact)


def test_worked_example_known_digits():
    # 25.752104 (exact, 6 decimals) is what the page's 25.8 rounds from
    y, _ = _worked(k=3, renorm=True)
    assert abs(y[0, 0] - 25.7521038) < 1e-6


# ---------------------------------------------------------------- softmax

def test_softmax_invariants():
    rng = np.random.default_rng(1)
    l = rng.normal(size=(50, 7)) * 3
    p = orc.softmax(l)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-12)
    # ratios are exp of logit differences (closed form, mpmath)
    for t in range(5):
        for i, j in [(0, 1), (2, 6), (5, 3)]:
            want = float(mp.exp(mp.mpf(l[t, i]) - mp.mpf(l[t, j])))
            assert abs(p[t, i] / p[t, j] - want) <= 1e-13 * want
    # shift invariance and the one-expert case
    np.testing.assert_allclose(orc.softmax(l + 123.0), p, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(orc.softmax(np.zeros((3, 1))), np.ones((3, 1)))


def test_softmax_large_logits_no_overflow():
    p = orc.softmax(np.array([[1000.0, 1000.0, 0.0]]))
    np.testing.assert_allclose(p[0, :2], 0.5, atol=1e-15)
    assert p[0, 2] < 1e-300


# ---------------------------------------------------------------- top-k

def _brute_topk(row, k):
    """Max-sum k-subset; among equal sums the lexicographically smallest index
    tuple (combinations() enumerates in that order and max() keeps the first);
    slots ordered by score descending, equal scores by index."""
    best = max(itertools.combinations(range(len(row)), k), key=lambda c: sum(row[i] for i in c))
    return sorted(best, key=lambda i: (-row[i], i))


def test_topk_all_tie_patterns_small():
    for E in range(1, 5):
        for vals in itertools.product([0.0, 1.0, 2.0], repeat=E):
            row = np.array(vals)
            for k in range(1, E + 1):
                got = orc.topk(row[None, :], k)[0].tolist()
                assert got == _brute_topk(list(vals), k), (vals, k)


def test_topk_random_fp32_scores():
    rng = np.random.default_rng(2)
    s = rng.normal(size=(64, 9)).astype(np.float32)
    s[::3, 4] = s[::3, 7]  # exact ties between experts 4 and 7
    for k in (1, 2, 5, 9):
        idx = orc.topk(s, k)
        for t in range(s.shape[0]):
            assert idx[t].tolist() == _brute_topk(s[t].astype(np.float64).tolist(), k)


def test_topk_on_probs_equals_on_logits():
    # softmax is monotone: selecting on p or on logits picks the same experts
    rng = np.random.default_rng(3)
    l = rng.normal(size=(40, 16))
    np.testing.assert_array_equal(orc.topk(l, 4), orc.topk(orc.softmax(l), 4))


# ---------------------------------------------------------------- gates

def test_renormalised_gates_equal_softmax_of_topk_logits():
    # [Intro] renormalises top-k of softmax; [Arch]/[Sparse] take softmax of the
    # top-k logits.  They are the same function.
    rng = np.random.default_rng(4)
    l = rng.normal(size=(30, 8)) * 2
    p = orc.softmax(l)
    idx = orc.topk(l, 3)
    g = orc.gates(p, idx, True)
    top = np.take_along_axis(l, idx, 1)
    ex = np.exp(top - top.max(1, keepdims=True))
    np.testing.assert_allclose(g, ex / ex.sum(1, keepdims=True), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-15)


def test_raw_gates_are_probabilities():
    rng = np.random.default_rng(5)
    l = rng.normal(size=(30, 8))
    p = orc.softmax(l)
    idx = orc.topk(l, 1)
    g = orc.gates(p, idx, False)
    np.testing.assert_array_equal(g[:, 0], p.max(1))
    idx6 = orc.topk(l, 6)
    g6 = orc.gates(p, idx6, False)
    np.testing.assert_array_equal(g6, np.take_along_axis(p, idx6, 1))
    assert np.all(g6.sum(1) < 1.0)


# ---------------------------------------------------------------- capacity

def test_capacity_page_example_and_configs():
    ex = _gold("capacity_examples.json")["page_example"]
    assert orc.capacity(ex["T"], ex["E"], ex["cf"]) == ex["C"]
    assert orc.capacity(8192, 128, 1.25) == 80     # Switch layer
    assert orc.capacity(4096, 256, 1.0) == 16      # skewed layer
    assert orc.capacity(64, 256, 1.0) == 0         # decode batch
    assert orc.capacity(100, 8, None) == -1        # no limit
    assert orc.capacity(100, 8, 0.0) == -1


def _brute_dispatch(idx, E, C):
    """Kept slots of expert e = the C earliest tokens (ascending) that chose e;
    perm rows list experts in order, each expert's kept tokens ascending."""
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E)
    dropped = np.zeros((T, k), np.uint8)
    perm = -np.ones((T, k), np.int64)
    row = 0
    for e in range(E):
        toks = sorted(t for t in range(T) if e in idx[t])
        kept = toks if C < 0 else toks[:C]
        for t in toks:
            j = list(idx[t]).index(e)
            if t in kept:
                perm[t, j] = row + kept.index(t)
            else:
                dropped[t, j] = 1
        row += len(kept)
    return counts, dropped, perm


def test_dispatch_bruteforce():
    rng = np.random.default_rng(6)
    for trial in range(300):
        E = int(rng.integers(1, 5))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 9))
        C = int(rng.integers(-1, 4))
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        got = orc.dispatch(idx, E, C)
        counts, dropped, perm = _brute_dispatch(idx, E, C)
        np.testing.assert_array_equal(got.counts, counts)
        np.testing.assert_array_equal(got.dropped, dropped)
        np.testing.assert_array_equal(got.perm_row, perm)
        kept = np.bincount(idx[dropped == 0].ravel(), minlength=E)
        np.testing.assert_array_equal(kept, counts if C < 0 else np.minimum(counts, C))


# ---------------------------------------------------------------- aux statistic

@pytest.mark.parametrize("E,k", [(8, 1), (8, 2), (64, 6), (5, 5)])
def test_aux_uniform_router_is_one(E, k):
    # W_g = 0: p = 1/E everywhere, so N * sum f_i P_i = sum f_i = 1 whatever is picked
    x = np.random.default_rng(7).normal(size=(37, 6))
    r = orc.route(x, np.zeros((E, 6)), None, k=k, renormalize=True, cf=None)
    assert abs(r.aux - 1.0) < 1e-12


def test_aux_collapse_is_E():
    E, T = 16, 40
    l = np.zeros((T, E))
    l[:, 3] = 60.0  # every token sends (almost) all probability to expert 3
    r = orc.route_from_logits(l, k=1, renormalize=False, cf=None)
    assert (r.idx[:, 0] == 3).all()
    assert abs(r.aux - E) < 1e-9


def test_aux_balanced_round_robin_is_one():
    E, T = 8, 64
    l = np.zeros((T, E))
    l[np.arange(T), np.arange(T) % E] = 1e-9
    r = orc.route_from_logits(l, k=1, renormalize=False, cf=None)
    np.testing.assert_array_equal(r.counts, T // E)
    assert abs(r.aux - 1.0) < 1e-8


def test_aux_counts_before_drops():
    # f_i is the router's hard assignment, not what survives the capacity
    l = np.zeros((10, 2))
    l[:, 0] = 5.0
    a = orc.route_from_logits(l, k=1, renormalize=False, cf=None)
    b = orc.route_from_logits(l, k=1, renormalize=False, cf=0.2)  # C = 1
    assert b.C == 1 and b.dropped.sum() == 9
    assert a.aux == b.aux


# ---------------------------------------------------------------- activations

@pytest.mark.parametrize("z", [-3.0, -1.0, -0.25, 0.0, 0.5, 1.0, 2.5])
def test_activations_against_mpmath(z):
    zz = mp.mpf(z)
    gt = 0.5 * zz * (1 + mp.tanh(mp.sqrt(2 / mp.pi) * (zz + mp.mpf("0.044715") * zz ** 3)))
    assert abs(orc.act("gelu_tanh", z) - float(gt)) < 1e-15
    assert abs(orc.act("gelu_erf", z) - float(zz * mp.ncdf(zz))) < 1e-15
    assert abs(orc.act("swiglu", z) - float(zz / (1 + mp.exp(-zz)))) < 1e-15
    assert orc.act("relu", z) == max(z, 0.0)


def test_activation_textbook_constants():
    assert abs(orc.act("gelu_erf", 1.0) - 0.8413447460685429) < 1e-15   # Phi(1)
    assert abs(orc.act("gelu_erf", -1.0) + 0.15865525393145707) < 1e-15
    assert abs(orc.act("swiglu", 1.0) - 0.7310585786300049) < 1e-15     # sigmoid(1)


# ---------------------------------------------------------------- expert FFN

def _rand(rng, *shape, scale=1.0):
    return rng.normal(size=shape) * scale


def test_single_expert_layer_is_plain_mlp_relu_with_bias():
    # E=1, k=1, renormalised, no capacity: the layer is one 2-layer MLP
    rng = np.random.default_rng(8)
    T, d, F = 9, 6, 11
    x, Wg = _rand(rng, T, d), _rand(rng, 1, d)
    W1, W2 = _rand(rng, 1, F, d), _rand(rng, 1, d, F)
    b1, b2 = _rand(rng, 1, F), _rand(rng, 1, d)
    y, r = orc.forward(x, Wg, None, W1, None, W2, b1, b2, E=1, S=0, k=1, act_name="relu",
                       renormalize=True, cf=None)
    np.testing.assert_array_equal(r.gates, 1.0)
    want = np.maximum(x @ W1[0].T + b1[0], 0) @ W2[0].T + b2[0]
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


def test_single_expert_layer_is_plain_mlp_swiglu():
    rng = np.random.default_rng(9)
    T, d, F = 7, 5, 13
    x, Wg = _rand(rng, T, d), _rand(rng, 1, d)
    W1, W3, W2 = _rand(rng, 1, F, d), _rand(rng, 1, F, d), _rand(rng, 1, d, F)
    y, _ = orc.forward(x, Wg, None, W1, W3, W2, None, None, E=1, S=0, k=1, act_name="swiglu",
                       renormalize=True, cf=None)
    a, b = x @ W1[0].T, x @ W3[0].T
    want = (a / (1 + np.exp(-a)) * b) @ W2[0].T
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


def test_dense_soft_moe_with_linear_experts():
    # [Basic] formulas: g = softmax(W_g x), e_i(x) = A_i x + b_i, y = sum_i g_i e_i(x).
    # A linear expert is a ReLU MLP with W1 = [I; -I], W2 = [A, -A], b2 = b.
    rng = np.random.default_rng(10)
    T, d, E = 6, 4, 3
    x, Wg = _rand(rng, T, d), _rand(rng, E, d)
    A, b = _rand(rng, E, d, d), _rand(rng, E, d)
    W1 = np.stack([np.vstack([np.eye(d), -np.eye(d)])] * E)
    W2 = np.stack([np.hstack([A[e], -A[e]]) for e in range(E)])
    y, _ = orc.forward(x, Wg, None, W1, None, W2, None, b, E=E, S=0, k=E, act_name="relu",
                       renormalize=True, cf=None)
    z = x @ Wg.T
    g = np.exp(z - z.max(1, keepdims=True))
    g /= g.sum(1, keepdims=True)
    want = sum(g[:, i:i + 1] * (x @ A[i].T + b[i]) for i in range(E))
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def test_topk_layer_sums_selected_experts_only():
    rng = np.random.default_rng(11)
    T, d, F, E, k = 12, 6, 9, 5, 2
    x, Wg = _rand(rng, T, d), _rand(rng, E, d)
    W1, W2 = _rand(rng, E, F, d), _rand(rng, E, d, F)
    y, r = orc.forward(x, Wg, None, W1, None, W2, None, None, E=E, S=0, k=k, act_name="relu",
                       renormalize=True, cf=None)
    for t in range(T):
        want = sum(r.gates[t, j] * (np.maximum(W1[e] @ x[t], 0) @ W2[e].T)
                   for j, e in enumerate(r.idx[t]))
        np.testing.assert_allclose(y[t], want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- drops, residual, shared

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_all_dropped_tokens_return_x_exactly(dtype):
    # [Switch] capacity: a dropped token's expert output is 0, and 0 + x = x
    g = torch.Generator().manual_seed(0)
    T, d, F, E = 10, 8, 16, 4
    x = torch.randn(T, d, generator=g).to(dtype)
    Wg = torch.randn(E, d, generator=g)
    W1 = torch.randn(E, F, d, generator=g).to(dtype)
    W2 = torch.randn(E, d, F, generator=g).to(dtype)
    y, r = orc.forward(x, Wg, None, W1, None, W2, None, None, E=E, S=0, k=2,
                       act_name="relu", renormalize=True, cf=0.1)  # C = floor(0.25) = 0
    assert r.C == 0 and r.dropped.all()
    np.testing.assert_array_equal(y, x.double().numpy())


def test_partially_dropped_token_keeps_its_kept_slots_without_x():
    l = np.zeros((4, 3))
    l[:, 0], l[:, 1] = 3.0, 2.0  # every token picks experts 0 then 1
    x = np.arange(4 * 2, dtype=np.float64).reshape(4, 2) + 1
    W1 = np.stack([np.eye(2)] * 3)
    W2 = np.stack([np.eye(2) * (e + 1) for e in range(3)])
    r = orc.route_from_logits(l, k=2, renormalize=True, cf=1.0)  # C = floor(4/3) = 1
    assert r.C == 1
    y = orc.output_rows(x, W1, None, W2, None, None, r.idx, r.gates, r.dropped, E=3, S=0,
                        act_name="relu", residual_mode=0)
    # token 0 keeps both slots; the others keep none and pass x through
    np.testing.assert_allclose(y[0], r.gates[0, 0] * 1 * x[0] + r.gates[0, 1] * 2 * x[0])
    np.testing.assert_array_equal(y[1:], x[1:])


def test_residual_modes_differ_by_x():
    rng = np.random.default_rng(12)
    T, d, F, E = 8, 4, 6, 3
    x, Wg = _rand(rng, T, d), _rand(rng, E, d)
    W1, W2 = _rand(rng, E, F, d), _rand(rng, E, d, F)
    r = orc.route(x, Wg, None, k=2, renormalize=True, cf=None)
    kw = dict(E=E, S=0, act_name="relu")
    y0 = orc.output_rows(x, W1, None, W2, None, None, r.idx, r.gates, r.dropped,
                         residual_mode=0, **kw)
    y1 = orc.output_rows(x, W1, None, W2, None, None, r.idx, r.gates, r.dropped,
                         residual_mode=1, **kw)
    np.testing.assert_array_equal(y1, y0 + x)


def test_shared_experts_always_on_with_gate_one():
    # [Switch] DeepSeekMoE: K_s shared experts are applied to every token
    rng = np.random.default_rng(13)
    T, d, F, E, S = 6, 4, 5, 3, 2
    x, Wg = _rand(rng, T, d), _rand(rng, E, d)
    W1, W3, W2 = _rand(rng, E + S, F, d), _rand(rng, E + S, F, d), _rand(rng, E + S, d, F)
    y_s, r = orc.forward(x, Wg, None, W1, W3, W2, None, None, E=E, S=S, k=2,
                         act_name="swiglu", renormalize=False, cf=None)
    y_r = orc.output_rows(x, W1, W3, W2, None, None, r.idx, r.gates, r.dropped, E=E, S=0,
                          act_name="swiglu", residual_mode=0)

    def ffn(e):
        a, b = x @ W1[e].T, x @ W3[e].T
        return (a / (1 + np.exp(-a)) * b) @ W2[e].T

    np.testing.assert_allclose(y_s, y_r + ffn(E) + ffn(E + 1), rtol=1e-12, atol=1e-12)


def test_shared_experts_equal_one_wide_swiglu():
    # S shared SwiGLU experts of hidden F = one SwiGLU of hidden S*F with the
    # weights concatenated along the hidden dimension
    rng = np.random.default_rng(14)
    T, d, F, E, S = 5, 4, 3, 2, 2
    x = _rand(rng, T, d)
    W1, W3, W2 = _rand(rng, E + S, F, d), _rand(rng, E + S, F, d), _rand(rng, E + S, d, F)
    none = np.zeros((T, 1), np.int32)
    drop = np.ones((T, 1), np.uint8)
    g0 = np.zeros((T, 1))
    y_sep = orc.output_rows(x, W1, W3, W2, None, None, none, g0, drop, E=E, S=S,
                            act_name="swiglu", residual_mode=0) - x
    W1c = np.concatenate([W1[E], W1[E + 1]])[None]
    W3c = np.concatenate([W3[E], W3[E + 1]])[None]
    W2c = np.concatenate([W2[E], W2[E + 1]], axis=1)[None]
    y_cat = orc.output_rows(x, W1c, W3c, W2c, None, None, none, g0, drop, E=0, S=1,
                            act_name="swiglu", residual_mode=0) - x
    np.testing.assert_allclose(y_sep, y_cat, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- router + storage

def test_router_logits_match_numpy_matmul_with_bias():
    rng = np.random.default_rng(15)
    x, Wg, bg = _rand(rng, 17, 12), _rand(rng, 5, 12), _rand(rng, 5)
    np.testing.assert_allclose(orc.router_logits(x, Wg, bg), x @ Wg.T + bg, rtol=1e-13,
                               atol=1e-13)


def test_bf16_inputs_are_widened_exactly():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(9, 16, generator=g).to(torch.bfloat16)
    Wg = torch.randn(4, 16, generator=g)
    a = orc.router_logits(x, Wg)
    b = orc.router_logits(x.float(), Wg)
    c = orc.router_logits(x.double().numpy(), Wg.double().numpy())
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_route_from_fp32_logits_is_selection_on_those_values():
    rng = np.random.default_rng(16)
    l32 = rng.normal(size=(50, 6)).astype(np.float32)
    l32[::4, 1] = l32[::4, 2]
    r = orc.route_from_logits(l32, k=2, renormalize=True, cf=None)
    for t in range(50):
        assert r.idx[t].tolist() == _brute_topk(l32[t].astype(np.float64).tolist(), 2)


# ---------------------------------------------------------------- noisy top-k gating

@pytest.mark.parametrize("z", [-700.0, -50.0, -3.5, -1e-3, 0.0, 0.7, 5.0, 40.0, 700.0])
def test_softplus_closed_form(z):
    # softplus(z) = ln(1 + e^z), evaluated at 40 digits
    ref = float(mp.log(1 + mp.e ** mp.mpf(z)))
    got = orc.softplus(z)
    if ref == 0.0:
        assert got == 0.0 or abs(got) < 1e-300
    else:
        assert abs(got - ref) <= 2e-16 * abs(ref)


def test_softplus_identities():
    assert orc.softplus(0.0) == pytest.approx(float(mp.log(2)), rel=1e-16, abs=0)
    for z in (-9.25, -0.5, 0.125, 3.0, 31.0):
        # softplus(z) - softplus(-z) = z;  softplus'(z) = sigmoid(z) via a central difference
        assert orc.softplus(z) - orc.softplus(-z) == pytest.approx(z, rel=1e-14, abs=1e-14)
        h = 1e-6
        deriv = (orc.softplus(z + h) - orc.softplus(z - h)) / (2 * h)
        assert deriv == pytest.approx(1.0 / (1.0 + np.exp(-z)), rel=1e-7)


def test_noisy_logits_zero_draws_is_clean():
    rng = np.random.default_rng(11)
    clean = rng.standard_normal((5, 7))
    nl = rng.standard_normal((5, 7)) * 4
    out = orc.noisy_logits(clean, nl, np.zeros((5, 7)), 0.01)
    np.testing.assert_array_equal(out, clean)


def test_noisy_logits_constant_noise_map_closed_form():
    # W_noise = 0 and a bias b: the noise scale of expert e is softplus(b_e) + min_std,
    # the same for every token; distinct eps values catch a transposed index
    T, E, d = 3, 5, 4
    rng = np.random.default_rng(12)
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, d))
    b = np.array([-2.0, -0.5, 0.0, 1.5, 6.0])
    eps = (np.arange(T * E, dtype=np.float64).reshape(T, E) - 7.0) / 3.0
    min_std = 0.01
    clean = orc.router_logits(x, Wg)
    noise_logits = orc.router_logits(x, np.zeros((E, d)), b)
    out = orc.noisy_logits(clean, noise_logits, eps, min_std)
    for t in range(T):
        for e in range(E):
            scale = float(mp.log(1 + mp.e ** mp.mpf(b[e]))) + min_std
            assert out[t, e] == pytest.approx(clean[t, e] + eps[t, e] * scale, rel=1e-14, abs=1e-14)


def test_noisy_route_row_constant_shift_leaves_softmax_and_choice():
    # W_noise = 0, b_noise = 0, min_std = 0: the shift of token t is eps[t] * ln 2 on every
    # expert; softmax is invariant to a per-row constant, so probs, top-k and aux equal the
    # clean routing's, while the logits move by exactly eps[t] * ln 2
    T, E, d, k = 9, 6, 5, 2
    rng = np.random.default_rng(13)
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, d))
    c = np.linspace(-3.0, 4.0, T)
    eps = np.repeat(c[:, None], E, axis=1)
    base = orc.route(x, Wg, None, k=k, renormalize=True, cf=1.0)
    noisy = orc.route(x, Wg, None, k=k, renormalize=True, cf=1.0,
                      noise=(np.zeros((E, d)), None, eps, 0.0))
    np.testing.assert_allclose(noisy.logits - base.logits,
                               np.repeat((c * float(mp.log(2)))[:, None], E, axis=1), rtol=0, atol=1e-13)
    np.testing.assert_allclose(noisy.probs, base.probs, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(noisy.idx, base.idx)
    np.testing.assert_array_equal(noisy.dropped, base.dropped)
    assert noisy.aux == pytest.approx(base.aux, rel=1e-13)


def test_noisy_route_flips_choice_by_hand():
    # one token, logits [1, 0, -1]; noise scale softplus(-40) + 0.01 ~= 0.01 on every expert.
    # eps = [0, 0, 250] lifts expert 2 to -1 + 2.5 = 1.5 > 1: it wins and expert 0 is second;
    # eps = [0, 0, 150] gives 0.5 < 1: the clean order [0, 1] stays
    x = np.array([[1.0]])
    Wg = np.array([[1.0], [0.0], [-1.0]])
    Wn = np.zeros((3, 1))
    bn = np.full(3, -40.0)
    r = orc.route(x, Wg, None, k=2, renormalize=False, cf=None,
                  noise=(Wn, bn, np.array([[0.0, 0.0, 250.0]]), 0.01))
    assert r.idx.tolist() == [[2, 0]]
    assert r.logits[0, 2] == pytest.approx(-1.0 + 250.0 * (0.01 + float(mp.log(1 + mp.e ** -40))), rel=1e-14)
    r = orc.route(x, Wg, None, k=2, renormalize=False, cf=None,
                  noise=(Wn, bn, np.array([[0.0, 0.0, 150.0]]), 0.01))
    assert r.idx.tolist() == [[0, 2]]
    # the second slot is expert 2 (0.5) ahead of expert 1 (0.0)


# ---------------------------------------------------------------- int8 expert weights

def test_quantize_int8_closed_form():
    # amax 127 gives scale 1 exactly, so q = round-half-even(w); the all-zero row gets
    # scale 0; a row with amax 0.5 gets scale 0.5/127 and its largest element maps to 127
    w = np.array([[127.0, -63.5, 2.5, -0.49, 0.5, 1.5],
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
                  [0.5, -0.5, 0.25, 0.0, -0.125, 0.0625]], dtype=np.float32)
    q, s = orc.quantize_int8(w)
    assert s[0] == 1.0 and s[1] == 0.0 and s[2] == np.float32(np.float32(0.5) / np.float32(127.0))
    assert q[0].tolist() == [127, -64, 2, 0, 0, 2]
    assert q[1].tolist() == [0] * 6
    assert q[2, 0] == 127 and q[2, 1] == -127 and q[2, 3] == 0


def test_quantize_int8_error_bound_and_range():
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((37, 53)) * rng.uniform(0.01, 3.0, size=(37, 1))).astype(np.float32)
    q, s = orc.quantize_int8(w)
    assert q.dtype == np.int8 and np.abs(q.astype(int)).max() == 127
    assert (np.abs(q.astype(int)).max(axis=1) == 127).all()  # every row reaches its scale
    deq = orc.dequantize_int8(q, s)
    # round to nearest: |w - q s| <= s / 2, with fp32 division slack
    err = np.abs(w.astype(np.float64) - deq)
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    # scale is max|w| / 127 in fp32
    np.testing.assert_array_equal(s, (np.abs(w).max(axis=1) / np.float32(127.0)).astype(np.float32))


# ---------------------------------------------------------------- 4-bit expert weights

def test_quantize_int4_closed_form_and_packing():
    # group 0 (8 columns, group size 8 here) has amax 7: scale 1, q = round-half-even(w);
    # group 1 is all zero (scale 0, q 0); in row 1, group 0 is tiny and group 1 large, so the
    # two groups get independent scales (a per-row scale would round group 0 to zero)
    w = np.array([[7.0, -2.5, 2.5, -3.5, 0.5, 1.5, -0.49, 6.5, 0, 0, 0, 0, 0, 0, 0, 0],
                  [0.07, -0.035, 0.0, 0.01, 0, 0, 0, 0, 70.0, -35.0, 10.0, 5.0, 0, 0, 0, -70.0]],
                 dtype=np.float32)
    packed, s = orc.quantize_int4(w, group=8)
    assert packed.shape == (2, 8) and s.shape == (2, 2)
    assert s[0, 0] == 1.0 and s[0, 1] == 0.0
    assert s[1, 0] == np.float32(np.float32(0.07) / np.float32(7.0)) and s[1, 1] == 10.0
    q = orc.unpack_int4(packed)
    assert q[0].tolist() == [7, -2, 2, -4, 0, 2, 0, 6] + [0] * 8
    assert q[1].tolist() == [7, -4, 0, 1, 0, 0, 0, 0, 7, -4, 1, 0, 0, 0, 0, -7]
    # nibble order and two's complement by hand: (7, -2) -> 0x7 | 0xE << 4 = 0xE7; (2, -4) -> 0xC2
    assert packed[0, 0] == 0xE7 and packed[0, 1] == 0xC2 and packed[0, 3] == 0x60
    np.testing.assert_array_equal(orc.dequantize_int4(packed, s, group=8)[1, 8:],
                                  [70.0, -40.0, 10.0, 0.0, 0.0, 0.0, 0.0, -70.0])


def test_quantize_int4_error_bound_and_range():
    rng = np.random.default_rng(22)
    w = (rng.standard_normal((19, 512)) * rng.uniform(0.01, 3.0, size=(19, 1))).astype(np.float32)
    w[3, 128:256] = 0.0  # one all-zero group
    packed, s = orc.quantize_int4(w)
    assert s.shape == (19, 4)
    q = orc.unpack_int4(packed).astype(int)
    assert np.abs(q).max() == 7
    per_group = np.abs(q).reshape(19, 4, 128).max(axis=2)
    assert per_group[3, 1] == 0 and s[3, 1] == 0.0
    assert (np.delete(per_group.reshape(-1), 3 * 4 + 1) == 7).all()  # every other group reaches +-7
    deq = orc.dequantize_int4(packed, s)
    err = np.abs(w.astype(np.float64) - deq)
    assert (err <= np.repeat(s, 128, axis=1).astype(np.float64) * (0.5 + 1e-5)).all()
    np.testing.assert_array_equal(
        s, (np.abs(w).reshape(19, 4, 128).max(axis=2) / np.float32(7.0)).astype(np.float32))
