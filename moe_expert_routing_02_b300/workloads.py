"""Seeded synthetic inputs for the MoE routing-and-expert step.

This module only draws random inputs; it holds none of the step's arithmetic
(no top-k, no counting, no GEMM).  Both the CUDA path and the CPU oracle take
their inputs from here, so a parity test always feeds the two sides the very
same numbers.

The pages measure on trained models and text corpora (MoE-GPT/MoE-BERT on
OpenWebText/PILE/OSCAR in the PopFetcher review; DeepSeekV2, Mixtral and DBRX
in the EPS-MoE review).  None of those are available, so seeded synthetic
tensors of the same shapes stand in for them:

* router logits  g = N(0,1) + b_e with a Zipf bias  b_e = -alpha * ln(e+1)
  (expert 0 hottest), fp32.  The skew follows the PopFetcher review's first
  observation (few experts receive most tokens, settling after a transient).
* inter-layer correlation: layer j+1 logits get +gamma on expert
  pi_j(argmax_e g_j[t]) for a seeded permutation pi_j (PopFetcher review,
  second observation: consecutive layers' choices are correlated).
* X ~ N(0,1) and weights ~ N(0, 0.02), both rounded to bf16.

Logits are drawn with NumPy's PCG64 from the seed tuple
(seed, config id, iteration, layer, stream); X and weights are drawn with a
torch generator on the device that will hold them (values therefore depend on
the device; tests hand the oracle a host copy of the same tensor).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = ["MoEConfig", "CONFIGS", "config_by_name", "alpha_at", "make_logits",
           "make_layer_logits", "make_x", "make_weights", "bf16_bits"]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    cid: int          # config id folded into every seed
    T: int            # tokens per iteration
    L: int            # MoE layers
    E: int            # experts
    k: int            # top-k
    H: int            # hidden size
    F: int            # expert FFN width
    act: str          # "gelu" | "swiglu"
    alpha: float      # Zipf exponent of the logit bias (final value)
    gamma: float      # inter-layer correlation boost
    iters: int        # iterations of the routing stream
    window: int = 10  # sliding window s (PopFetcher review, s = 10)
    alpha_ramp: int = 0      # iterations over which alpha ramps up linearly (0 = fixed)
    replicate: bool = False  # hot-expert replication on

    @property
    def A(self) -> int:
        return self.T * self.k

    def describe(self) -> dict:
        return {k: v for k, v in dataclasses.asdict(self).items()}


# The five workloads.  Shapes follow the models the pages name: MoE-GPT
# (12 layers, H=1024, alpha=F/H=2; PopFetcher review), Mixtral-8x7B (8 experts,
# top-2), DeepSeekV2 (160 experts, top-6) and DBRX (16 experts, top-4) from the
# EPS-MoE review's experiment set-up.
CONFIGS = [
    MoEConfig("tiny", 1, T=256, L=2, E=8, k=2, H=64, F=128, act="gelu",
              alpha=1.0, gamma=2.0, iters=10),
    MoEConfig("moe_gpt_stream", 2, T=16384, L=12, E=16, k=2, H=1024, F=2048, act="gelu",
              alpha=1.2, gamma=1.5, iters=200, alpha_ramp=50),
    MoEConfig("mixtral_layer", 3, T=8192, L=1, E=8, k=2, H=4096, F=14336, act="swiglu",
              alpha=1.0, gamma=0.0, iters=1),
    MoEConfig("deepseekv2_layer", 4, T=4096, L=1, E=160, k=6, H=5120, F=1536, act="swiglu",
              alpha=1.1, gamma=0.0, iters=1),
    MoEConfig("dbrx_replicated_layer", 5, T=4096, L=1, E=16, k=4, H=6144, F=10752, act="swiglu",
              alpha=1.5, gamma=0.0, iters=1, replicate=True),
]


def config_by_name(name: str) -> MoEConfig:
    for c in CONFIGS:
        if c.name == name or str(c.cid) == str(name):
            return c
    raise KeyError(name)


def alpha_at(cfg: MoEConfig, it: int) -> float:
    """Zipf exponent at iteration `it`: ramps linearly over the first
    `alpha_ramp` iterations, then stays fixed (the transient-then-stable load
    pattern of "Prediction Is All MoE Needs")."""
    if cfg.alpha_ramp <= 0:
        return cfg.alpha
    return cfg.alpha * min(it + 1, cfg.alpha_ramp) / cfg.alpha_ramp


def _perm(cfg: MoEConfig, layer: int, seed: int) -> np.ndarray:
    return np.random.default_rng([seed, cfg.cid, 0xFFFF, layer, 1]).permutation(cfg.E)


def make_logits(T: int, E: int, alpha: float, *, seed_key, prev: Optional[np.ndarray] = None,
                perm: Optional[np.ndarray] = None, gamma: float = 0.0) -> np.ndarray:
    """One layer's fp32 router logits [T, E].

    prev/perm/gamma add the inter-layer correlation: +gamma on expert
    perm[argmax_e prev[t]] (first maximum on ties)."""
    rng = np.random.default_rng(list(seed_key))
    g = rng.standard_normal((T, E))
    g += -alpha * np.log(np.arange(1, E + 1, dtype=np.float64))[None, :]
    if prev is not None and gamma != 0.0:
        top1 = np.argmax(prev, axis=1)
        g[np.arange(T), perm[top1]] += gamma
    out = g.astype(np.float32)
    # the gate's contract takes finite logits (the kernels do not check each
    # element), so the generator checks what it hands out
    if not np.isfinite(out).all():
        raise ValueError("non-finite logits")
    return out


def make_layer_logits(cfg: MoEConfig, it: int, *, seed: int = 0, T: Optional[int] = None,
                      layers: Optional[int] = None) -> list:
    """Router logits of every layer at iteration `it` (list of [T, E] fp32).

    `T` may be lowered to draw a prefix-sized sample with the same recipe."""
    T = cfg.T if T is None else T
    L = cfg.L if layers is None else layers
    out = []
    a = alpha_at(cfg, it)
    for j in range(L):
        prev = out[-1] if j > 0 else None
        perm = _perm(cfg, j - 1, seed) if j > 0 else None
        out.append(make_logits(T, cfg.E, a, seed_key=(seed, cfg.cid, it, j, 0),
                               prev=prev, perm=perm, gamma=cfg.gamma))
    return out


def _torch_gen(device, key):
    import torch
    g = torch.Generator(device=device)
    # fold the key tuple into one 63-bit seed
    h = 1469598103934665603
    for v in key:
        h = ((h ^ (int(v) & 0xFFFFFFFFFFFF)) * 1099511628211) & ((1 << 63) - 1)
    g.manual_seed(h)
    return g


def make_x(cfg: MoEConfig, it: int, layer: int, *, device="cpu", seed: int = 0, T: Optional[int] = None):
    """Token activations X [T, H] in bf16, N(0,1)."""
    import torch
    T = cfg.T if T is None else T
    g = _torch_gen(device, (seed, cfg.cid, it, layer, 2))
    return torch.randn((T, cfg.H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_weights(cfg: MoEConfig, layer: int, *, device="cpu", seed: int = 0, E: Optional[int] = None,
                 H: Optional[int] = None, F: Optional[int] = None):
    """Expert weights (w1 [E,H,F], w3 [E,H,F] or None, w2 [E,F,H]) in bf16, N(0, 0.02).

    w1 is the gate projection (GeLU: the only first projection), w3 the up
    projection of SwiGLU, w2 the down projection.  Drawn one expert at a time
    so the fp32 temporary stays one expert large."""
    import torch
    E = cfg.E if E is None else E
    H = cfg.H if H is None else H
    F = cfg.F if F is None else F
    g = _torch_gen(device, (seed, cfg.cid, 0, layer, 3))
    names = ["w1", "w3", "w2"] if cfg.act == "swiglu" else ["w1", "w2"]
    out = {}
    for nm in names:
        shape = (E, F, H) if nm == "w2" else (E, H, F)
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for e in range(E):
            t[e] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
        out[nm] = t
    return out["w1"], out.get("w3"), out["w2"]


def bf16_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a bf16 torch tensor (for the oracle)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
