"""How many MMA rows the CTA-pair GEMMs spend on padding, from each workload's
routing counts: an expert's rows fill 256-row pair blocks, and its partial
last block cost a full tile before swap tiles (an M = 128 half tile costs as
many cycles) and costs its rows rounded up to 16 as a swap tile.  The routing
here is torch's fp32 top-k on the CPU (the counts' spread, not the exact
fixed-order ties, sets these shares)."""
import numpy as np
import pytest
import torch

from dispatch_ffn_combine_gb300.workloads import CONFIGS, make_inputs


def _counts(name):
    cfg = CONFIGS[name]
    g = make_inputs(cfg, seed=0, experts=False)
    logits = g["x"].float() @ g["wg"].t()
    if g["bias"] is not None:
        logits += g["bias"]
    ids = torch.topk(logits, cfg.k, dim=1).indices
    return torch.bincount(ids.flatten(), minlength=cfg.E).numpy().astype(np.int64)


def _padding(counts):
    rows = int(counts.sum())
    full, tail = counts // 256, counts % 256
    before = int((full * 256 + np.where(tail > 0, 256, 0)).sum())
    after = int((full * 256 + (tail + 15) // 16 * 16).sum())
    return 1 - rows / before, 1 - rows / after


@pytest.mark.parametrize("name,before,after", [("large", 0.104, 0.0075), ("mid", 0.210, 0.015), ("skewed", 0.061, 0.004)])
def test_padding_share_before_and_after_swap_tiles(name, before, after):
    b, a = _padding(_counts(name))
    assert b == pytest.approx(before, abs=0.005)
    assert a == pytest.approx(after, abs=0.002)
