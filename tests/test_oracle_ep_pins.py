"""Pins of the oracle's expert-parallel layer (orc.ep_forward, orc.ep_exchange).

Expert parallelism places the experts on different devices and shards the
tokens over the workers, which exchange tokens with an AllToAll ("MoE架构解析"
§3.2 分布式训练优化 and §5 问题3; "MoE混合专家模型原理与实战" §4.2 专家分片).
The pins tie the rank-by-rank computation to the single-rank oracle (itself
pinned by the pages' worked example, closed forms and brute force) and to the
readings of the layout:
  - without a capacity limit, G ranks compute exactly the single-rank layer,
    and the receive order of all ranks' buffers, concatenated, is the
    single-rank expert-contiguous token order (perm_row);
  - with a capacity limit, each shard is exactly a single-rank layer over its
    own tokens with C_r = floor(T_r cf / E), and the balance statistic is
    still the global one (uniform router -> 1, collapsed router -> E);
  - brute force on tiny layers: every kept slot is received exactly once, by
    the owner of its expert, in (expert, source rank, token) order;
  - a hand-worked case of the per-shard capacity rule.
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from sparse_mixture_experts_scan_b300 import config, make_inputs


def _layer(cfg, seed=0):
    inp = make_inputs(cfg, seed)
    return {k: (None if v is None else v) for k, v in inp.items()}


def _args(cfg):
    return dict(E=cfg.E, S=cfg.S, k=cfg.k, act_name=cfg.act, renormalize=cfg.renormalize,
                cf=cfg.cf, residual_mode=cfg.residual_mode)


def _single(inp, cfg, **kw):
    a = _args(cfg)
    a.update(kw)
    return orc.forward(inp["x"], inp["W_gate"], inp["b_gate"], inp["W1"], inp["W3"], inp["W2"],
                       inp["b1"], inp["b2"], **a)


def _ep(inp, cfg, G, **kw):
    a = _args(cfg)
    a.update(kw)
    return orc.ep_forward(inp["x"], inp["W_gate"], inp["b_gate"], inp["W1"], inp["W3"], inp["W2"],
                          inp["b1"], inp["b2"], G=G, **a)


CASES = [
    config("tiny", T=203),                                              # GELU, biases, ragged shards
    config("deepseek", T=157, d=32, E=16, k=3, F=24, S=2),              # shared experts, raw gates
    config("mixtral", T=96, d=32, E=8, k=2, F=40, residual_mode=1),     # residual on every token
]


@pytest.mark.parametrize("cfg", CASES, ids=["tiny", "shared", "residual1"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_without_capacity_ranks_compute_the_single_rank_layer(cfg, G):
    if cfg.E % G:
        pytest.skip("E not a multiple of G")
    inp = _layer(cfg)
    y1, r1 = _single(inp, cfg, cf=None)
    ep = _ep(inp, cfg, G, cf=None)
    np.testing.assert_array_equal(ep.idx, r1.idx)
    np.testing.assert_array_equal(ep.counts, r1.counts)
    np.testing.assert_array_equal(ep.ex.dropped, r1.dropped)
    # the concatenated receive buffers are the single-rank expert-contiguous token order
    np.testing.assert_array_equal(ep.ex.recv_row, r1.perm_row)
    assert np.abs(ep.y - y1).max() <= 1e-12 * max(1.0, np.abs(y1).max())
    assert abs(ep.aux - r1.aux) <= 1e-13 * max(1.0, r1.aux)
    b = orc.shard_bounds(cfg.T, G)
    for r in range(G):  # per-rank counts add up and cover only the rank's tokens
        want = np.bincount(r1.idx[b[r]:b[r + 1]].reshape(-1), minlength=cfg.E)
        np.testing.assert_array_equal(ep.ex.counts_rank[r], want)


@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("cf", [0.5, 1.0, 1.25])
def test_with_capacity_each_shard_is_a_single_rank_layer(G, cf):
    cfg = config("tiny", T=203, cf=cf)
    inp = _layer(cfg)
    ep = _ep(inp, cfg, G)
    b = orc.shard_bounds(cfg.T, G)
    kept_total = 0
    for r in range(G):
        sub = {k_: v for k_, v in inp.items()}
        sub["x"] = inp["x"][b[r]:b[r + 1]]
        T_r = b[r + 1] - b[r]
        y_r, r_r = _single(sub, config("tiny", T=T_r, cf=cf))
        assert ep.C_rank[r] == orc.capacity(T_r, cfg.E, cf) == int(np.floor(T_r * cf / cfg.E))
        np.testing.assert_array_equal(ep.ex.dropped[b[r]:b[r + 1]], r_r.dropped)
        np.testing.assert_array_equal(ep.ex.counts_rank[r], r_r.counts)
        assert np.abs(ep.y[b[r]:b[r + 1]] - y_r).max() <= 1e-12 * max(1.0, np.abs(y_r).max())
        kept_total += int(np.minimum(r_r.counts, ep.C_rank[r]).sum())
    assert int((ep.ex.dropped == 0).sum()) == kept_total == int(ep.ex.recv_rows.sum())


def test_one_rank_with_capacity_is_the_single_rank_layer():
    cfg = config("tiny", T=150, cf=1.0)
    inp = _layer(cfg)
    y1, r1 = _single(inp, cfg)
    ep = _ep(inp, cfg, 1)
    np.testing.assert_array_equal(ep.ex.dropped, r1.dropped)
    np.testing.assert_array_equal(ep.ex.recv_row, r1.perm_row)
    assert np.abs(ep.y - y1).max() <= 1e-12 * max(1.0, np.abs(y1).max())
    assert abs(ep.aux - r1.aux) <= 1e-13


def test_per_shard_capacity_by_hand():
    # T = 8 tokens, E = 2, k = 1, G = 2, cf = 1: every token chooses expert 0.
    # Per shard C_r = floor(4 * 1 / 2) = 2: tokens 0, 1 (rank 0) and 4, 5 (rank 1) are kept.
    # (The whole batch on one rank would have C = 4 and keep tokens 0..3.)
    idx = np.zeros((8, 1), dtype=np.int32)
    ex = orc.ep_exchange(idx, 2, 2, [orc.capacity(4, 2, 1.0)] * 2)
    assert orc.capacity(4, 2, 1.0) == 2
    np.testing.assert_array_equal(ex.dropped[:, 0], [0, 0, 1, 1, 0, 0, 1, 1])
    np.testing.assert_array_equal(ex.recv_row[:, 0], [0, 1, -1, -1, 2, 3, -1, -1])
    np.testing.assert_array_equal(ex.recv_rows, [4, 0])  # rank 0 owns expert 0
    np.testing.assert_array_equal(ex.recv_slot, [0, 1, 4, 5])
    np.testing.assert_array_equal(ex.counts_rank, [[4, 0], [4, 0]])
    one = orc.dispatch(idx, 2, orc.capacity(8, 2, 1.0))
    np.testing.assert_array_equal(one.dropped[:, 0], [0, 0, 0, 0, 1, 1, 1, 1])


def _brute_force_layout(idx, E, G, C_rank):
    """Kept slots of each rank by enumeration; received rows listed by sorting on
    (owner, expert, source rank, token, slot)."""
    T, k = idx.shape
    b = orc.shard_bounds(T, G)
    kept = []
    for r in range(G):
        seen = {}
        for t in range(b[r], b[r + 1]):
            for j in range(k):
                e = int(idx[t, j])
                p = seen.get(e, 0)
                seen[e] = p + 1
                if C_rank[r] < 0 or p < C_rank[r]:
                    kept.append((e // (E // G), e, r, t, j))
    return sorted(kept)


def test_exchange_layout_brute_force():
    rng = np.random.default_rng(5)
    n = 0
    for E, G in [(2, 1), (2, 2), (4, 2), (4, 4), (6, 3)]:
        for k in range(1, min(E, 3) + 1):
            for T in (1, 3, 5, 8, 9):
                for cf in (None, 0.5, 1.0, 2.0):
                    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
                    b = orc.shard_bounds(T, G)
                    C_rank = [orc.capacity(b[r + 1] - b[r], E, cf) for r in range(G)]
                    ex = orc.ep_exchange(idx, E, G, C_rank)
                    want = _brute_force_layout(idx, E, G, C_rank)
                    got_slots = [int(s) for s in ex.recv_slot]
                    assert got_slots == [t * k + j for (_, _, _, t, j) in want]
                    owners = [q for (q, *_) in want]
                    assert list(ex.recv_rows) == [owners.count(q) for q in range(G)]
                    for s in range(T * k):
                        row = ex.recv_row.reshape(-1)[s]
                        assert (row < 0) == bool(ex.dropped.reshape(-1)[s])
                        if row >= 0:
                            assert ex.recv_slot[row] == s
                    n += 1
    assert n == 260  # (2 + 2 + 3 + 3 + 3) top-k values x 5 batch sizes x 4 capacity factors


@pytest.mark.parametrize("G", [1, 2, 4])
def test_balance_statistic_is_global(G):
    cfg = config("tiny", T=96, cf=1.0)
    inp = _layer(cfg)
    # uniform router: p = 1/E for every token, so E sum f P = sum f = 1 whatever the ties select
    uni = dict(inp)
    uni["W_gate"] = torch.zeros_like(inp["W_gate"])
    uni["b_gate"] = torch.zeros_like(inp["b_gate"])
    assert abs(_ep(uni, cfg, G).aux - 1.0) <= 1e-14
    # collapsed router: every token sends (almost) all probability to expert 3 -> aux -> E
    col = dict(uni)
    col["b_gate"] = torch.zeros_like(inp["b_gate"])
    col["b_gate"][3] = 60.0
    col["b_gate"][5] = 30.0  # the second choice of every token (k = 2)
    ep = _ep(col, cfg, G)
    assert abs(ep.aux - cfg.E / 2.0) <= 1e-9  # f_3 = f_5 = 1/2, P_3 -> 1
    np.testing.assert_array_equal(ep.counts, np.eye(cfg.E, dtype=np.int32)[[3, 5]].sum(0) * cfg.T)
