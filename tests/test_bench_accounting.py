"""The bench's roofline arithmetic on hand-built routings (CPU).

The algorithmic bytes and flops of the expert stage and the minimum bytes of the memory
stages are counted here tensor by tensor for tiny layers whose routing is written out,
and compared with what bench.py reports for the same routing.
"""
import torch

import bench
from sparse_mixture_experts_scan_b300 import config


def _out(idx, dropped):
    return {"expert_idx": torch.tensor(idx, dtype=torch.int32),
            "dropped": torch.tensor(dropped, dtype=torch.uint8)}


def test_expert_stage_bytes_and_flops_relu_top1():
    # 4 tokens, experts 0, 2, 2, 3; token 3's slot dropped: experts 0 and 2 are touched
    cfg = config("switch", T=4, d=8, E=4, k=1, F=16)
    out = _out([[0], [2], [2], [3]], [[0], [0], [0], [1]])
    got = bench.algorithmic_gemm_work(cfg, out)
    w1 = cfg.F * cfg.d * 2  # one expert's W1 in bf16
    w2 = cfg.d * cfg.F * 2
    weights = 2 * (w1 + w2)  # experts 0 and 2
    per_row = (cfg.d + cfg.F + cfg.F + cfg.d) * 2  # Xp read, H written, H read, Yp written
    assert got["touched_experts"] == 2 and got["kept_rows"] == 3
    assert got["weight_bytes"] == weights
    assert got["bytes"] == weights + 3 * per_row
    assert got["flops"] == 3 * (2 * cfg.d * cfg.F) * 2  # two GEMMs, 2 flops per multiply-add
    # the combine finished in the expert stage adds each kept row's token and gate
    assert bench.algorithmic_gemm_work(cfg, out, direct=True)["bytes"] == weights + 3 * per_row + 3 * 8


def test_expert_stage_bytes_with_shared_experts_and_quantised_weights():
    cfg = config("deepseek", T=2, d=128, E=2, k=1, F=256, S=2)
    out = _out([[1], [1]], [[0], [0]])
    got = bench.algorithmic_gemm_work(cfg, out)
    one = 3 * cfg.d * cfg.F * 2  # W1, W3, W2 of one expert, bf16
    assert got["touched_experts"] == 1 + cfg.S
    assert got["weight_bytes"] == (1 + cfg.S) * one
    routed = 2 * (cfg.d + 2 * cfg.F + cfg.d) * 2
    # shared: x read once, S * F hidden columns per token written and read, one output row
    shared = (cfg.T * cfg.d + cfg.T * cfg.S * cfg.F * 2 + cfg.T * cfg.d) * 2
    assert got["bytes"] == (1 + cfg.S) * one + routed + shared
    assert got["flops"] == (2 + cfg.S * cfg.T) * 2 * cfg.d * cfg.F * 3

    q8 = bench.algorithmic_gemm_work(config("switch", T=2, d=128, E=2, k=1, F=256, weights="int8"),
                                     _out([[0], [1]], [[0], [0]]))
    # per expert: 1-byte W1 and W2 plus one fp32 scale per row of each
    assert q8["weight_bytes"] == 2 * (2 * 128 * 256 + 4 * (256 + 128))
    q4 = bench.algorithmic_gemm_work(config("switch", T=2, d=128, E=2, k=1, F=256, weights="int4"),
                                     _out([[0], [0]], [[0], [0]]))
    # one expert: half-byte W1 and W2 plus one fp32 scale per 128 inputs of every row
    assert q4["weight_bytes"] == (256 * 128 + 128 * 256) // 2 + 4 * (256 * 1 + 128 * 2)


def test_memory_stage_bytes():
    cfg = config("switch", T=4, d=8, E=4, k=1, F=16)
    out = _out([[0], [2], [2], [3]], [[0], [0], [0], [1]])
    gemm = bench.algorithmic_gemm_work(cfg, out)
    got = bench.stage_bytes(cfg, out, gemm)
    s, T, d, k, E = 2, cfg.T, cfg.d, cfg.k, cfg.E
    # router: x read, fp32 W_gate read, expert index and gate written per slot
    assert got["moe_router"] == T * d * s + E * d * 4 + T * k * (4 + 4)
    # dispatch: indices read, 3 kept rows copied (read + write), per slot dropped flag,
    # permutation row and padded row written
    assert got["moe_dispatch"] == T * k * 4 + 3 * d * s * 2 + T * k * (1 + 4 + 4)
    # combine: kept expert rows read, y written, the dropped token's x read, gates read
    assert got["moe_combine"] == 3 * d * s + T * d * s + 1 * d * s + T * k * 8
    # top-1 direct combine: the dispatch also copies the dropped token's row into y and
    # records each kept row's token and gate; no combine stage
    direct = bench.stage_bytes(cfg, out, gemm, direct=True)
    assert direct["moe_combine"] == 0
    assert direct["moe_dispatch"] == got["moe_dispatch"] + 2 * d * s + 3 * 8
