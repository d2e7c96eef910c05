"""Seeded synthetic workloads for the MoE layer.

This module only draws random inputs with the shapes and distributions of the
layer's workloads; it holds none of the layer's arithmetic.  Both the CUDA path
and the CPU oracle consume the tensors it returns.

Recipe (one fixed reading, stated once):
  x   ~ N(0, 1) drawn in fp32, rounded to bf16 (round-to-nearest-even)   [T, d]
  Wg  ~ N(0, 1/d) fp32 (1/d is the variance)                             [E, d]
  W1, W3 ~ N(0, 1/d) drawn in fp32, rounded to bf16                      [E, f, d]
  W2  ~ N(0, 1/f) drawn in fp32, rounded to bf16                         [E, d, f]
  bias: none, except for the skewed workload, where expert e's gate logit
        is offset by -s * ln(e + 1) with s = 1.2 (the log of an unnormalised
        Zipf(s) weight of rank e + 1), so the routing prior follows Zipf.
Every tensor (and every expert's slice of a weight tensor) has its own seed,
derived from the workload seed and the tensor's name, so a slice can be
regenerated alone and the draw does not depend on the device's memory size.
"""
from __future__ import annotations

import dataclasses
import math
import zlib

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int      # tokens
    d: int      # model dim
    E: int      # experts
    k: int      # experts per token
    f: int      # FFN (intermediate) dim
    zipf_s: float = 0.0   # > 0: gate logits biased by -zipf_s * ln(e + 1)

    @property
    def S(self) -> int:
        """Routed rows T*k."""
        return self.T * self.k

    @property
    def expert_flops(self) -> int:
        """FLOPs of the expert GEMMs: gemm1 (gate and up) + gemm2 = 6*T*k*d*f."""
        return 6 * self.T * self.k * self.d * self.f

    @property
    def router_flops(self) -> int:
        return 2 * self.T * self.d * self.E

    def describe(self) -> str:
        b = f", zipf bias s={self.zipf_s}" if self.zipf_s else ""
        return f"{self.name}: T={self.T} d={self.d} E={self.E} k={self.k} ffn={self.f}{b}"


# The five layer workloads, and small test shapes with ragged tiles.
CONFIGS = {
    "tiny": MoEConfig("tiny", 256, 256, 8, 2, 512),
    "mid": MoEConfig("mid", 4096, 2048, 32, 4, 1408),
    "skewed": MoEConfig("skewed", 16384, 4096, 64, 8, 1536, zipf_s=1.2),
    "decode": MoEConfig("decode", 128, 7168, 256, 8, 2048),
    "large": MoEConfig("large", 32768, 7168, 256, 8, 2048),
    # test shapes: several M/N/K tiles, ragged in every dimension
    "ragged": MoEConfig("ragged", 1000, 384, 12, 3, 320),
    "ragged_skew": MoEConfig("ragged_skew", 777, 512, 20, 5, 192, zipf_s=1.2),
    "single": MoEConfig("single", 300, 256, 1, 1, 384),
    # ~500 rows per expert: several row blocks per expert, ragged in every tile dimension
    "ragged_pair": MoEConfig("ragged_pair", 1500, 384, 6, 2, 320),
    # edge shapes: the smallest d and ffn with k = E (every expert takes every
    # token), and 256 experts at k = 1 with most experts empty or single-row
    "edge_min": MoEConfig("edge_min", 50, 64, 3, 3, 64),
    "many_experts": MoEConfig("many_experts", 300, 128, 256, 1, 128),
    # profiling shape: the large layer's d and ffn with 16 experts (about 2.5 GB
    # on the device), small enough for multi-pass counter captures
    "prof": MoEConfig("prof", 4096, 7168, 16, 8, 2048),
}


def tensor_seed(seed: int, name: str, index: int = 0) -> int:
    h = zlib.crc32(f"{name}:{index}".encode())
    return (int(seed) * 1_000_003 + h * 65_537 + int(index)) % (2 ** 62)


def _normal(shape, std, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def zipf_bias(E: int, s: float) -> torch.Tensor:
    return torch.tensor([-s * math.log(e + 1.0) for e in range(E)], dtype=torch.float32)


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", T: int | None = None, experts: bool = True) -> dict:
    """Draw one workload.  Returns a dict of torch tensors on ``device``:
    x [T,d] bf16, wg [E,d] f32, bias [E] f32 or None, w1/w3 [E,f,d] bf16,
    w2 [E,d,f] bf16.  ``T`` overrides the token count (weights unchanged);
    ``experts=False`` skips the expert weights (router-only uses)."""
    T = cfg.T if T is None else T
    d, E, f = cfg.d, cfg.E, cfg.f
    dev = torch.device(device)
    x = _normal((T, d), 1.0, tensor_seed(seed, "x"), dev).to(torch.bfloat16)
    wg = _normal((E, d), d ** -0.5, tensor_seed(seed, "wg"), dev)
    bias = zipf_bias(E, cfg.zipf_s).to(dev) if cfg.zipf_s else None
    if not experts:
        return {"x": x, "wg": wg, "bias": bias, "w1": None, "w3": None, "w2": None}
    w1 = torch.empty((E, f, d), dtype=torch.bfloat16, device=dev)
    w3 = torch.empty((E, f, d), dtype=torch.bfloat16, device=dev)
    w2 = torch.empty((E, d, f), dtype=torch.bfloat16, device=dev)
    for e in range(E):
        w1[e].copy_(_normal((f, d), d ** -0.5, tensor_seed(seed, "w1", e), dev))
        w3[e].copy_(_normal((f, d), d ** -0.5, tensor_seed(seed, "w3", e), dev))
        w2[e].copy_(_normal((d, f), f ** -0.5, tensor_seed(seed, "w2", e), dev))
    return {"x": x, "wg": wg, "bias": bias, "w1": w1, "w3": w3, "w2": w2}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_float(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp32 values."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
