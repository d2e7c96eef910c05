"""Shared helpers for the GPU parity tests (host-side marshalling only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dispatch_ffn_combine_gb300.workloads import CONFIGS, bf16_bits, bits_to_float, make_inputs

# Layer output tolerance: max|g - o| <= 1e-2 * max|o| + 1e-3 and
# sum|g - o| / sum|o| <= 5e-3 (mean relative error over all elements).
MAX_REL = 1e-2
MAX_ABS = 1e-3
MEAN_REL = 5e-3


def check_output(got, ref, what=""):
    """got: bf16 torch tensor or float array; ref: fp64 array (the oracle)."""
    if isinstance(got, torch.Tensor):
        got = bits_to_float(bf16_bits(got)).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    max_err = float(err.max()) if err.size else 0.0
    bound = MAX_REL * float(np.abs(ref).max()) + MAX_ABS
    mean_rel = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    assert max_err <= bound, f"{what}: max|err| {max_err:.3e} > {bound:.3e}"
    assert mean_rel <= MEAN_REL, f"{what}: mean relative error {mean_rel:.3e} > {MEAN_REL}"
    return max_err, mean_rel


class Workload:
    """One config's inputs on the GPU plus host copies for the oracle."""

    def __init__(self, name: str, seed: int = 0, T: int | None = None, experts: bool = True):
        self.cfg = CONFIGS[name]
        self.dev = torch.device("cuda:0")
        gen_dev = "cpu" if self.cfg.E * self.cfg.f * self.cfg.d <= (1 << 26) else self.dev
        inp = make_inputs(self.cfg, seed=seed, device=gen_dev, T=T, experts=experts)
        self.T = inp["x"].shape[0]
        self.g = {k: (v.to(self.dev) if v is not None else None) for k, v in inp.items()}
        self.h = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
        self._bits = {}

    def bits(self, name):
        if name not in self._bits:
            self._bits[name] = bf16_bits(self.h[name])
        return self._bits[name]

    @property
    def wg(self):
        return self.h["wg"].numpy()

    @property
    def bias(self):
        b = self.h["bias"]
        return None if b is None else b.numpy()

    def oracle_routing(self):
        logits = oracle.router_logits(self.bits("x"), self.wg, self.bias)
        ids, w = oracle.topk(logits, self.cfg.k)
        return logits, ids, w

    def oracle_layer(self, tokens=None):
        return oracle.layer(self.bits("x"), self.wg, self.bias, self.bits("w1"), self.bits("w3"), self.bits("w2"),
                            self.cfg.k, tokens=tokens)

    def near_ties(self, ids, rel=1e-5):
        """Tokens whose k-th and (k+1)-th fp64 logits are closer than rel*|l| (diagnostic)."""
        if self.cfg.k >= self.cfg.E:
            return 0
        l64 = oracle.router_logits_f64(self.bits("x"), self.wg, self.bias)
        s = -np.sort(-l64, axis=1)
        gap = s[:, self.cfg.k - 1] - s[:, self.cfg.k]
        return int(np.sum(gap < rel * np.maximum(np.abs(s[:, self.cfg.k - 1]), 1.0)))


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """A fixed sample: first and last tokens plus a seeded random spread."""
    if n >= T:
        return np.arange(T, dtype=np.int64)
    rs = np.random.RandomState(seed)
    mid = rs.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid])).astype(np.int64)
