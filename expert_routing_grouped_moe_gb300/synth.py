"""Seeded synthetic inputs for the MoE-LoRA expert layer.

This module only draws random numbers and rounds them to the storage types
(bf16 by round-to-nearest-even, fp32, int32).  It holds none of the layer's
arithmetic: no routing, no softmax, no top-k over router logits, no GEMM.
Both the CPU oracle (through the tests) and the CUDA path consume what it
returns, so the two sides always see identical bits.

Workload shapes follow the layer configurations the pages benchmark
(Unsloth "faster MoE" page, sections on gpt-oss, Qwen3 and GLM benchmarks):

* ``tiny``            T=256,  d=128,  f=64,   E=8,   k=2, r=8,  alpha=16
* ``qwen3_30b_a3b``   T=4096, d=2048, f=768,  E=128, k=8, r=64, alpha=128
* ``gpt_oss_20b``     T=8192, d=2880, f=2880, E=32,  k=4, r=8,  alpha=16
* ``skewed_shared``   T=16384, d=2048, f=1536, E=64 routed + 1 shared, k=4,
                      r=16, alpha=32, router bias following a Zipf ranking

Value distributions: X ~ N(0,1); base weights W and LoRA A ~ N(0, 1/d)
(variance 1/d, i.e. std 1/sqrt(d), for gate_up and down alike); LoRA B ~
N(0, 0.02^2) (std 0.02, nonzero); router logits fp32 ~ N(0,1) (+ bias for the
skewed workload); upstream gradient dY ~ N(0,1).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # tokens
    d: int          # hidden size
    f: int          # expert intermediate size
    E: int          # routed experts
    k: int          # experts per token
    r: int          # LoRA rank
    alpha: float    # LoRA alpha; scale s = alpha / r
    shared: bool = False   # one always-active shared expert (weight 1)
    zipf_bias: float = 0.0  # >0: per-expert router bias = zipf_bias * rank^-1.2
    n_blocked: int = 0      # experts whose router bias is -inf (never picked)

    @property
    def scale(self) -> float:
        return self.alpha / self.r

    @property
    def groups(self) -> int:
        """Expert groups with weights: routed experts plus the shared one."""
        return self.E + (1 if self.shared else 0)

    @property
    def slots(self) -> int:
        """Expert slots per token: top-k plus the shared expert."""
        return self.k + (1 if self.shared else 0)

    @property
    def rows(self) -> int:
        """Routed (token, expert) rows N."""
        return self.T * self.slots


CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, d=128, f=64, E=8, k=2, r=8, alpha=16),
    "qwen3_30b_a3b": LayerConfig("qwen3_30b_a3b", T=4096, d=2048, f=768, E=128,
                                 k=8, r=64, alpha=128),
    "gpt_oss_20b": LayerConfig("gpt_oss_20b", T=8192, d=2880, f=2880, E=32, k=4,
                               r=8, alpha=16),
    "skewed_shared": LayerConfig("skewed_shared", T=16384, d=2048, f=1536, E=64,
                                 k=4, r=16, alpha=32, shared=True,
                                 zipf_bias=3.0, n_blocked=4),
}


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """A copy of ``cfg`` with some fields replaced (used for edge cases)."""
    return dataclasses.replace(cfg, **kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype=torch.bfloat16):
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)  # torch's float->bf16 cast rounds to nearest even


def router_bias(cfg: LayerConfig, seed: int) -> torch.Tensor:
    """Per-expert router logit bias of the skewed workload (fp32, [E]).

    bias_e = zipf_bias * rank_e^-1.2 with rank a seeded permutation of 1..E;
    the ``n_blocked`` experts with the largest ranks get -inf so that empty
    experts occur.  Zero bias when ``zipf_bias`` is 0.
    """
    if cfg.zipf_bias == 0.0 and cfg.n_blocked == 0:
        return torch.zeros(cfg.E, dtype=torch.float32)
    g = _gen(seed * 7919 + 17, "cpu")
    rank = torch.randperm(cfg.E, generator=g) + 1
    bias = cfg.zipf_bias * rank.to(torch.float64).pow(-1.2)
    if cfg.n_blocked:
        bias[rank > cfg.E - cfg.n_blocked] = -math.inf
    return bias.to(torch.float32)


def layer_weights(cfg: LayerConfig, seed: int, device="cpu") -> dict:
    """Frozen base weights and LoRA adapters, one group per expert.

    Layout (row-major, bf16): W_gu [G,2f,d] (rows [0,f) gate, [f,2f) up),
    A_gu [G,r,d], B_gu [G,2f,r], W_dn [G,d,f], A_dn [G,r,f], B_dn [G,d,r];
    G = E (+1 for the shared expert, stored last).
    """
    G, d, f, r = cfg.groups, cfg.d, cfg.f, cfg.r
    g = _gen(seed * 1000003 + 1, device)
    sd = 1.0 / math.sqrt(d)
    return {
        "W_gu": _normal((G, 2 * f, d), sd, g, device),
        "A_gu": _normal((G, r, d), sd, g, device),
        "B_gu": _normal((G, 2 * f, r), 0.02, g, device),
        "W_dn": _normal((G, d, f), sd, g, device),
        "A_dn": _normal((G, r, f), sd, g, device),
        "B_dn": _normal((G, d, r), 0.02, g, device),
    }


def layer_activations(cfg: LayerConfig, seed: int, device="cpu") -> dict:
    """Token rows X [T,d] bf16, router logits [T,E] fp32, upstream grad dY [T,d] bf16."""
    g = _gen(seed * 1000003 + 2, device)
    X = _normal((cfg.T, cfg.d), 1.0, g, device)
    logits = torch.randn(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float32)
    logits += router_bias(cfg, seed).to(device)
    dY = _normal((cfg.T, cfg.d), 1.0, g, device)
    return {"X": X, "logits": logits, "dY": dY}


# ---------------------------------------------------------------------------
# Routing / permute sweep: top-k ids drawn directly (the layer's input), with
# distinct ids per token, uniform or Zipf(1.2) expert popularity.
# ---------------------------------------------------------------------------

ROUTE_SWEEP = [(T, E, k, dist)
               for T in (1 << 10, 1 << 14, 1 << 18, 1 << 20)
               for E in (8, 32, 64, 128)
               for k in (2, 4, 8)
               for dist in ("uniform", "zipf")
               if k <= E]


def topk_ids(T: int, E: int, k: int, dist: str, seed: int, device="cpu") -> torch.Tensor:
    """Distinct expert ids per token, [T,k] int32.

    Drawn without replacement with probability p_e (uniform, or proportional
    to rank_e^-1.2 with rank a seeded permutation of 1..E) by perturbing
    log p_e with Gumbel noise and keeping the k largest keys (a standard way
    to sample k items without replacement).  This is data synthesis only.
    """
    g = _gen(seed * 1000003 + 3, device)
    if dist == "uniform":
        logp = torch.zeros(E, device=device)
    elif dist == "zipf":
        gr = _gen(seed * 7919 + 29, "cpu")
        rank = (torch.randperm(E, generator=gr) + 1).to(torch.float64)
        logp = (-1.2 * rank.log()).to(torch.float32).to(device)
    else:
        raise ValueError(dist)
    ids = torch.empty(T, k, dtype=torch.int32, device=device)
    chunk = 1 << 16
    for t0 in range(0, T, chunk):
        n = min(chunk, T - t0)
        u = torch.rand(n, E, generator=g, device=device).clamp_(min=1e-20)
        keys = logp - torch.log(-torch.log(u))
        ids[t0:t0 + n] = torch.topk(keys, k, dim=1).indices.to(torch.int32)
    return ids


def combine_weights(T: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    """Per-slot combine weights [T,k] fp32: U(0,1) normalised per token."""
    g = _gen(seed * 1000003 + 4, device)
    w = torch.rand(T, k, generator=g, device=device, dtype=torch.float64) + 1e-3
    return (w / w.sum(dim=1, keepdim=True)).to(torch.float32)


def hidden_rows(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 token rows [T,d] ~ N(0,1)."""
    g = _gen(seed * 1000003 + 5, device)
    return _normal((T, d), 1.0, g, device)
