"""Seeded synthetic workloads for the DSpark draft-head round.

This module is the one piece shared by the CUDA path's tests/benchmarks and the
CPU oracle.  It draws random tensors and builds the profiled steps-per-second
tables; it holds none of the method's arithmetic (no logits, no sampling, no
confidences, no scheduling, no verification).

The five workload shapes follow the draft-head configurations the method is
exercised on: a tiny instance, a Qwen3-4B-shaped and a Qwen3-8B-shaped draft
head, the DeepSeek-V4-shaped DSpark-5 (block size 5, Markov rank 512, noise
token id 128799, per the DeepSeek-V4-Pro-0813 DSpark configuration), and a
high-concurrency scheduler stress case.  The trained checkpoints, target models
and benchmark suites are not available, so every tensor here is synthetic:

* backbone hidden states h ~ N(0, 1)
* shared LM head W_lm ~ N(0, 1/sqrt(d))   (so base logits are ~N(0, 1))
* Markov factors W1 ~ N(0, 1/sqrt(r)), W2 ~ N(0, 2/sqrt(r))
* confidence head w ~ N(0, 1/sqrt(d + r))
* Sequential-Temperature-Scaling temperatures T_k
* anchors uniform over the vocabulary (below the noise token id for V4 shapes)
* target-logit noise N(0, sigma) (std = sigma), per request where stated
* a monotone, concave or stair-stepped SPS(B) table

"N(0, s)" is read as standard deviation s throughout.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

BASE_SEED = 0x5EED


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int          # requests in the batch
    gamma: int      # draft positions per request
    V: int          # vocabulary
    r: int          # Markov-head rank
    d: int          # backbone hidden size
    dtype: str      # "fp32" (values bf16-representable) or "bf16"
    tau: float      # sampling temperature for draft and verify; 0 = greedy
    temps: str      # "uniform12" (T_k ~ U[1,2]) or "linear" (T_k = 1 + 0.1 k)
    sigma: str      # target noise: "const:<s>" or "uniform:<lo>:<hi>" per request
    anchor_hi: int  # anchors uniform in [0, anchor_hi)
    sps: str        # SPS(B) table kind, see sps_table()
    n_sps: int
    index: int      # position in the workload list (seed offset)

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index

    @property
    def M(self) -> int:
        return self.R * self.gamma

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 4, 5, 1024, 64, 256, "fp32", 0.0, "uniform12",
                     "const:1.0", 1024, "linear", 64, 0),
    "qwen3_4b": Workload("qwen3_4b", 1, 8, 151936, 256, 2560, "bf16", 0.0, "uniform12",
                         "const:0.5", 151936, "linear", 64, 1),
    "qwen3_8b": Workload("qwen3_8b", 64, 8, 151936, 256, 4096, "bf16", 1.0, "linear",
                         "const:0.5", 151936, "concave", 1024, 2),
    "v4_dspark5": Workload("v4_dspark5", 256, 5, 129280, 512, 7168, "bf16", 1.0, "uniform12",
                           "uniform:0.2:2.0", 128799, "stair", 2048, 3),
    "stress": Workload("stress", 1024, 7, 129280, 512, 7168, "bf16", 0.0, "uniform12",
                       "uniform:0.2:2.0", 128799, "stair", 8192, 4),
}


def sps_table(kind: str, n: int) -> torch.Tensor:
    """Synthetic engine-profiled steps/s for verify batch sizes B = 1..n (entry B-1).

    linear : 1000 (1 - (B-1)/128)                  monotone decreasing
    concave: 1000 (1 - 0.75 ((B-1)/(n-1))^2)         smooth, concave
    stair  : 1000 / (1 + 0.15 floor((B-1)/64))      plateaus every 64 tokens
    """
    B = torch.arange(1, n + 1, dtype=torch.float64)
    if kind == "linear":
        s = 1000.0 * (1.0 - (B - 1.0) / 128.0)
    elif kind == "concave":
        s = 1000.0 * (1.0 - 0.75 * ((B - 1.0) / max(n - 1, 1)) ** 2)
    elif kind == "stair":
        s = 1000.0 / (1.0 + 0.15 * torch.floor((B - 1.0) / 64.0))
    else:
        raise ValueError(kind)
    return s.to(torch.float32)


def _round_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, device: str = "cpu", seed: Optional[int] = None,
                with_target_noise: bool = True) -> Dict[str, torch.Tensor]:
    """Draw every random input of one round of workload `w`.

    Returned tensors (weights/activations in bf16; for dtype "fp32" they are
    returned as float32 tensors holding bf16-representable values):
      h [R, gamma, d], anchor [R] int32, W_lm [V, d], W1 [V, r], W2 [r, V],
      w_conf [d + r], T [gamma] fp32, sps [n_sps] fp32, sigma [R] fp32,
      noise [R, gamma + 1, V] (target-logit noise, std sigma_r; bf16),
      h_next [R, d] (hidden state that makes target row gamma + 1),
      draft_seed, verify_seed (python ints).
    """
    seed = w.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    R, G, V, r, d = w.R, w.gamma, w.V, w.r, w.d

    def normal(shape, std):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        return _round_bf16(t)

    out: Dict[str, torch.Tensor] = {}
    out["h"] = normal((R, G, d), 1.0)
    out["W_lm"] = normal((V, d), 1.0 / math.sqrt(d))
    out["W1"] = normal((V, r), 1.0 / math.sqrt(r))
    out["W2"] = normal((r, V), 2.0 / math.sqrt(r))
    out["w_conf"] = normal((d + r,), 1.0 / math.sqrt(d + r))
    out["h_next"] = normal((R, d), 1.0)
    out["anchor"] = torch.randint(0, w.anchor_hi, (R,), generator=g, device=device,
                                  dtype=torch.int64).to(torch.int32)
    if w.temps == "uniform12":
        T = 1.0 + torch.rand((G,), generator=g, device=device, dtype=torch.float32)
    elif w.temps == "linear":
        T = 1.0 + 0.1 * torch.arange(1, G + 1, device=device, dtype=torch.float32)
    else:
        raise ValueError(w.temps)
    out["T"] = T
    kind, *args = w.sigma.split(":")
    if kind == "const":
        sigma = torch.full((R,), float(args[0]), device=device, dtype=torch.float32)
    else:
        lo, hi = float(args[0]), float(args[1])
        sigma = lo + (hi - lo) * torch.rand((R,), generator=g, device=device,
                                            dtype=torch.float32)
    out["sigma"] = sigma
    if with_target_noise:
        n = torch.randn((R, G + 1, V), generator=g, device=device, dtype=torch.float32)
        n.mul_(sigma.view(R, 1, 1))
        out["noise"] = _round_bf16(n)
        del n
    out["sps"] = sps_table(w.sps, w.n_sps).to(device)
    if w.dtype == "fp32":
        for k in ("h", "W_lm", "W1", "W2", "w_conf", "h_next", "noise"):
            if k in out:
                out[k] = out[k].to(torch.float32)
    out["draft_seed"] = (seed * 0x9E3779B97F4A7C15 + 1) & 0xFFFFFFFFFFFFFFFF
    out["verify_seed"] = (seed * 0xC2B2AE3D27D4EB4F + 7) & 0xFFFFFFFFFFFFFFFF
    return out


def random_confidences(R: int, gamma: int, seed: int, device: str = "cpu",
                       ones_frac: float = 0.0) -> torch.Tensor:
    """Confidences in (0, 1] for scheduler-only tests; a fraction can be exactly 1."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    c = torch.rand((R, gamma), generator=g, device=device, dtype=torch.float32)
    c = 0.02 + 0.98 * c
    if ones_frac > 0:
        m = torch.rand((R, gamma), generator=g, device=device) < ones_frac
        c = torch.where(m, torch.ones_like(c), c)
    return c


def random_tokens(R: int, gamma: int, V: int, seed: int, device: str = "cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, V, (R, gamma), generator=g, device=device,
                         dtype=torch.int64).to(torch.int32)


def random_lengths(R: int, gamma: int, seed: int, device: str = "cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, gamma + 1, (R,), generator=g, device=device,
                         dtype=torch.int64).to(torch.int32)


def random_normal(shape, std: float, seed: int, device: str = "cpu",
                  dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std) samples rounded to `dtype` (e.g. stand-alone logits for stage tests)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return t.mul_(std).to(dtype)
