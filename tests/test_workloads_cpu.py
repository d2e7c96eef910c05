"""The synthetic input recipe: shapes and dtypes, the variance reading of
N(0, 1/d), the Zipf router offset of the skewed workload, and seeding."""
import math

import torch

from dispatch_ffn_combine_gb300.workloads import CONFIGS, make_inputs, zipf_bias


def test_shapes_dtypes_and_scales():
    cfg = CONFIGS["ragged"]  # T 1000, d 384, E 12, k 3, f 320
    g = make_inputs(cfg, seed=0)
    assert g["x"].shape == (1000, 384) and g["x"].dtype == torch.bfloat16
    assert g["wg"].shape == (12, 384) and g["wg"].dtype == torch.float32
    assert g["w1"].shape == g["w3"].shape == (12, 320, 384) and g["w1"].dtype == torch.bfloat16
    assert g["w2"].shape == (12, 384, 320) and g["w2"].dtype == torch.bfloat16
    assert g["bias"] is None
    # 1/d and 1/ffn are variances: standard deviations d^-1/2 and f^-1/2
    assert abs(g["x"].float().std().item() - 1.0) < 0.02
    assert abs(g["wg"].std().item() * math.sqrt(384) - 1.0) < 0.05
    assert abs(g["w1"].float().std().item() * math.sqrt(384) - 1.0) < 0.02
    assert abs(g["w3"].float().std().item() * math.sqrt(384) - 1.0) < 0.02
    assert abs(g["w2"].float().std().item() * math.sqrt(320) - 1.0) < 0.02


def test_seeding_is_deterministic_and_per_tensor():
    cfg = CONFIGS["tiny"]
    a, b = make_inputs(cfg, seed=0), make_inputs(cfg, seed=0)
    c = make_inputs(cfg, seed=1)
    for name in ("x", "wg", "w1", "w3", "w2"):
        assert torch.equal(a[name], b[name])
        assert not torch.equal(a[name], c[name])
    assert not torch.equal(a["w1"], a["w3"])  # separate streams per tensor


def test_token_override_keeps_weights():
    cfg = CONFIGS["tiny"]
    a, b = make_inputs(cfg, seed=0), make_inputs(cfg, seed=0, T=37)
    assert b["x"].shape == (37, cfg.d)
    for name in ("wg", "w1", "w3", "w2"):
        assert torch.equal(a[name], b[name])


def test_zipf_offset_skews_routing():
    bias = zipf_bias(64, 1.2)
    assert bias[0].item() == 0.0
    assert abs(bias[9].item() + 1.2 * math.log(10.0)) < 1e-6
    assert torch.all(bias[1:] < bias[:-1])
    cfg = CONFIGS["skewed"]  # E 64, k 8, bias = -1.2 ln(e + 1)
    g = make_inputs(cfg, seed=0, T=2048, experts=False)
    assert torch.equal(g["bias"], bias)
    logits = g["x"].float() @ g["wg"].t() + g["bias"]
    ids = torch.topk(logits, cfg.k, dim=1).indices
    counts = torch.bincount(ids.flatten(), minlength=64).float()
    assert counts[0] / 2048 > 0.9  # nearly every token picks expert 0
    assert counts.max() / counts.mean() > 5  # strongly imbalanced
