"""Seeded synthetic inputs shaped like the pages' workload.

This module holds no arithmetic of the method: it only draws random tensors
(router logits, the initial selection bias, score gradients, hidden states and
router weights) with torch generators.  Both the CUDA path and the CPU oracle
are fed from here, the oracle through a host copy of the very same tensors.

Workload shapes follow "Exact Quantile Balancing and Load-Error Injection for
Mixture-of-Experts" (testbed paragraph: 256 routed experts, top-6, 48 MoE
layers; LEI paragraph and results: eta = 8e-5) and "[Dev] Add global-batch
quantile balancing" ("Quantile estimator": 1000 uniform bins over
[min b - 1, max b + 1]).  Distribution N(m, s) means mean m, standard
deviation s, except the router weight, whose 1/2048 is a variance (fan-in
initialisation, so logits come out about unit scale).

Draw order inside one layer: per-expert offsets, bias, then each microbatch
in turn (logits, then its skew subset and skewed tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    E: int
    k: int
    n_micro: int
    n_tokens: int  # tokens per microbatch
    logits_dtype: torch.dtype = torch.float32
    logit_std: float = 1.0
    offset_std: float = 0.5
    bias_range: float = 0.1
    skew: bool = False
    nbins: int = 0  # K3 only
    layers: int = 1
    eta: float = 0.0  # LEI only
    grad_std: float = 1e-3
    hidden: int = 0  # router GEMM only
    extra: dict = field(default_factory=dict)

    @property
    def n_pool(self) -> int:
        return self.n_micro * self.n_tokens


# The five workloads.  Seeds: workload c, layer l -> 1000*c + l, except the tiny
# EQB case which uses seed 0.
WORKLOADS = {
    "eqb_tiny": Workload("eqb_tiny", E=64, k=6, n_micro=1, n_tokens=4096),
    "eqb_pooled": Workload("eqb_pooled", E=256, k=6, n_micro=8, n_tokens=16384, skew=True),
    "k3": Workload("k3", E=256, k=8, n_micro=4, n_tokens=65536, logits_dtype=torch.bfloat16,
                   logit_std=1.5, offset_std=0.3, bias_range=0.2, nbins=1000),
    "full_step": Workload("full_step", E=256, k=6, n_micro=16, n_tokens=32768, skew=True,
                          layers=48, eta=8e-5),
    "router_gemm": Workload("router_gemm", E=256, k=6, n_micro=4, n_tokens=32768, hidden=2048),
}

_WORKLOAD_INDEX = {"eqb_tiny": 1, "eqb_pooled": 2, "k3": 3, "full_step": 4, "router_gemm": 5}


def seed_for(name: str, layer: int = 0) -> int:
    if name == "eqb_tiny":
        return layer
    return 1000 * _WORKLOAD_INDEX[name] + layer


def scaled(w: Workload, **changes) -> Workload:
    """Same recipe, other sizes (used for the small parity cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(changes)
    return Workload(**d)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def router_layer(w: Workload, seed: int, device="cpu", out=None):
    """Bias and per-microbatch logits of one router layer.

    Returns (bias [E] fp32, [logits [n_tokens, E]] * n_micro).  When ``out`` is
    a preallocated tensor [n_micro * n_tokens, E] the microbatches are written
    into it and returned as views (the bench keeps 48 layers resident this way).
    """
    g = _gen(seed, device)
    E = w.E
    off = torch.randn(E, generator=g, device=device, dtype=torch.float32) * w.offset_std
    bias = (torch.rand(E, generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0) * w.bias_range
    mbs = []
    for m in range(w.n_micro):
        x = torch.randn(w.n_tokens, E, generator=g, device=device, dtype=torch.float32)
        x.mul_(w.logit_std).add_(off)
        if w.skew:
            subset = torch.randperm(E, generator=g, device=device)[:16]
            n_sk = (w.n_tokens * 10) // 100
            toks = torch.randperm(w.n_tokens, generator=g, device=device)[:n_sk]
            x[toks.unsqueeze(1), subset.unsqueeze(0)] += 1.0
        x = x.to(w.logits_dtype)
        if out is not None:
            dst = out[m * w.n_tokens:(m + 1) * w.n_tokens]
            dst.copy_(x)
            mbs.append(dst)
        else:
            mbs.append(x.contiguous())
    return bias, mbs


def k3_initial_bounds(bias: torch.Tensor):
    """[min b - 1, max b + 1] of the initial bias, in fp32 ("Quantile estimator")."""
    b = bias.detach().float().cpu()
    lo = (b.min() - 1.0).to(torch.float32)
    hi = (b.max() + 1.0).to(torch.float32)
    return torch.stack([lo, hi])


def score_grad(w: Workload, seed: int, n_tokens: int | None = None, device="cpu", out=None):
    """fp32 score gradient [n_tokens, E] ~ N(0, grad_std)."""
    g = _gen(seed + 500_000, device)
    n = w.n_tokens if n_tokens is None else n_tokens
    if out is not None:
        out.normal_(0.0, w.grad_std, generator=g)
        return out
    return torch.randn(n, w.E, generator=g, device=device, dtype=torch.float32) * w.grad_std


def gemm_layer(w: Workload, seed: int, device="cpu"):
    """Router GEMM inputs: bias [E], W [H, E] bf16 (variance 1/H), hidden states per microbatch."""
    g = _gen(seed, device)
    H, E = w.hidden, w.E
    bias = (torch.rand(E, generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0) * w.bias_range
    W = (torch.randn(H, E, generator=g, device=device, dtype=torch.float32) * (1.0 / H) ** 0.5)
    W = W.to(torch.bfloat16)
    hs = [torch.randn(w.n_tokens, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
          for _ in range(w.n_micro)]
    return bias, W, hs


def random_topk(n_tokens: int, E: int, k: int, seed: int, device="cpu"):
    """k distinct experts per token drawn uniformly (for LEI cases without routing)."""
    g = _gen(seed, device)
    r = torch.rand(n_tokens, E, generator=g, device=device)
    return torch.topk(r, k, dim=1).indices.to(torch.int32)
