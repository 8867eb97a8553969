"""Seeded synthetic inputs for the MXFP4 MoE expert layer.

This module draws the tensors a verify-block MoE layer consumes and nothing
else: hidden states, router weights and bias, RMSNorm weights and the fp32
master copies of the expert weights (which a quantizer then turns into MXFP4).
It holds none of the layer's arithmetic.  The one place it evaluates anything
is the routing-margin condition that the workload definition puts on the
inputs ("router ... so the top-k logit margin is at least 1e-3"): rows of x are
re-drawn until the gaps between the top-(k+1) router logits, computed with a
library fp64 matmul, are all at least ``margin``.  That only *selects* inputs;
both the CUDA path and the oracle receive the same selected tensors.  A caller
may add its own condition on a row (``make_inputs(accept_row=...)``), bringing
whatever arithmetic that condition needs.

Workloads (one MoE verify block of T tokens; page 3 "DFlash: block-level
masked parallel draft" fixes 8 positions per stream):

=========  ====  =====  =====  ===  ==  ======  =========================
name        T     H      I      E   k  layers  routing
=========  ====  =====  =====  ===  ==  ======  =========================
tiny        8     256    128     8   2    1    uniform
mid         8    4096   1536    64   8    1    uniform
large       8    7168   2048   384   8    1    uniform
batched   256    7168   2048   384   8    1    Zipf(1.1) expert popularity
stack       8    4096   1536    64   8    8    uniform, RMSNorm + residual
=========  ====  =====  =====  ===  ==  ======  =========================

Distributions: x ~ N(0, 1) -> bf16 (RNE); router W ~ N(0, 0.02) -> bf16;
expert weights fp32 ~ N(0, 1/sqrt(fan_in)) (fan_in = H for gate/up, I for
down); RMSNorm weight ~ N(1, 0.1) -> bf16.  The second argument of N is the
standard deviation.

Every tensor has its own sub-stream: a splitmix64 chain over
(workload seed, tensor tag, layer, index, attempt) seeds a torch generator.
Expert weights are drawn per (layer, expert, matrix) so any subset of experts
can be regenerated alone, on any device (the CPU and CUDA generators give
different streams, so a caller picks one device per tensor and keeps it).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def splitmix64(z: int) -> int:
    """One splitmix64 output step (Steele, Lea, Flood 2014) on a 64-bit state."""
    z = (z + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


_TAGS = {"x": 1, "router_w": 2, "norm_w": 3, "gate": 4, "up": 5, "down": 6, "zipf": 7}


def derive_seed(base: int, tag: str, layer: int = 0, index: int = 0, attempt: int = 0) -> int:
    """Seed of one sub-stream; a pure function of its arguments."""
    z = splitmix64(base & _MASK64)
    for part in (_TAGS[tag], layer, index, attempt):
        z = splitmix64(z ^ (part & _MASK64))
    return z & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    layers: int = 1
    routing: str = "uniform"  # or "zipf"
    norm: bool = False
    seed: int = 0
    margin: float = 1e-3
    rms_eps: float = 1e-6
    zipf_s: float = 1.1
    # > 0: every element of x is also multiplied by 2^u, u a uniform integer in
    # [-x_spread, x_spread] (drawn from the row's stream after the normal values), so
    # that one 32-element block of x spans up to 2^(2 x_spread) in magnitude
    x_spread: int = 0

    @property
    def expert_bytes(self) -> int:
        """Packed bytes of one expert: 3 matrices of H*I nibbles + one scale byte per 32."""
        return 3 * (self.H * self.I // 2 + self.H * self.I // 32)

    def scaled(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", T=8, H=256, I=128, E=8, k=2, seed=0x5EED0000),
    "mid": Workload("mid", T=8, H=4096, I=1536, E=64, k=8, seed=0x5EED0001),
    "large": Workload("large", T=8, H=7168, I=2048, E=384, k=8, seed=0x5EED0002),
    "batched": Workload("batched", T=256, H=7168, I=2048, E=384, k=8, routing="zipf", seed=0x5EED0003),
    "stack": Workload("stack", T=8, H=4096, I=1536, E=64, k=8, layers=8, norm=True, seed=0x5EED0004),
}


@dataclass
class LayerTensors:
    router_w: torch.Tensor            # bf16 [E, H]
    router_b: torch.Tensor            # fp32 [E]
    norm_w: torch.Tensor | None       # bf16 [H] or None


@dataclass
class Inputs:
    wl: Workload
    x: torch.Tensor                   # bf16 [T, H] (CPU)
    layers: list = field(default_factory=list)   # list[LayerTensors] (CPU)
    redraws: dict = field(default_factory=dict)  # token -> attempts used by the margin rule

    def expert_weight(self, layer: int, e: int, which: str, device="cpu") -> torch.Tensor:
        """fp32 master weight of one expert matrix: gate/up [I, H], down [H, I]."""
        return expert_weight(self.wl, layer, e, which, device)


def expert_weight(wl: Workload, layer: int, e: int, which: str, device="cpu") -> torch.Tensor:
    if which in ("gate", "up"):
        shape, fan_in = (wl.I, wl.H), wl.H
    elif which == "down":
        shape, fan_in = (wl.H, wl.I), wl.I
    else:
        raise ValueError(which)
    g = _gen(derive_seed(wl.seed, which, layer, e), device)
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return w * torch.tensor(1.0 / math.sqrt(fan_in), dtype=torch.float32, device=device)


def _zipf_bias(wl: Workload, H: int) -> torch.Tensor:
    """Per-expert router bias that makes expert popularity roughly Zipf(s).

    Ranks 1..E are randomly permuted over the experts; p_e is proportional to
    rank_e^-s and b_e = beta * ln p_e.  With Gaussian router logits of std
    sigma = 0.02 * sqrt(H) (x ~ N(0,1)), beta = sigma * sqrt(6) / pi makes the
    logit noise roughly Gumbel of scale beta, so the top-1 choice is roughly
    Categorical(p) and top-k roughly sampling without replacement.
    """
    g = _gen(derive_seed(wl.seed, "zipf"), "cpu")
    ranks = torch.randperm(wl.E, generator=g).to(torch.float64) + 1.0
    logp = -wl.zipf_s * torch.log(ranks)
    logp = logp - torch.logsumexp(logp, 0)
    sigma = 0.02 * math.sqrt(H)
    beta = sigma * math.sqrt(6.0) / math.pi
    return (beta * logp).to(torch.float32)


def _row_ok(logits_row: torch.Tensor, k: int, margin: float) -> bool:
    top = torch.sort(logits_row, descending=True).values[: min(k + 1, logits_row.numel())]
    return bool(torch.all(top[:-1] - top[1:] >= margin))


def _draw_row(wl: Workload, t: int, attempt: int) -> torch.Tensor:
    """Row t of x, attempt `attempt`: N(0, 1) values (times 2^u with x_spread), bf16 (RNE)."""
    g = _gen(derive_seed(wl.seed, "x", 0, t, attempt), "cpu")
    row = torch.randn(wl.H, generator=g, dtype=torch.float64)
    if wl.x_spread > 0:
        u = torch.randint(-wl.x_spread, wl.x_spread + 1, (wl.H,), generator=g, dtype=torch.int64)
        row = row * torch.exp2(u.to(torch.float64))
    return row.to(torch.bfloat16)


def make_inputs(wl: Workload, max_attempts: int = 64, accept_row=None) -> Inputs:
    """Draw x, router and norm weights (all on CPU) for a workload.

    accept_row(t, row) -> bool, when given, is a further condition on row t of x
    (bf16 [H]) after the first-layer margin rule: a row it rejects is re-drawn like
    one that fails the margin rule.  The caller brings the arithmetic it needs (for
    example the margins of every layer of a stack along a reference trajectory);
    this module only draws and selects."""
    layers = []
    for l in range(wl.layers):
        g = _gen(derive_seed(wl.seed, "router_w", l), "cpu")
        wr = (torch.randn((wl.E, wl.H), generator=g, dtype=torch.float64) * 0.02).to(torch.bfloat16)
        if wl.routing == "zipf" and l == 0:
            b = _zipf_bias(wl, wl.H)
        else:
            b = torch.zeros(wl.E, dtype=torch.float32)
        nw = None
        if wl.norm:
            g = _gen(derive_seed(wl.seed, "norm_w", l), "cpu")
            nw = (1.0 + 0.1 * torch.randn(wl.H, generator=g, dtype=torch.float64)).to(torch.bfloat16)
        layers.append(LayerTensors(router_w=wr, router_b=b, norm_w=nw))

    # Margin rule on the first layer's router (the one that sees x directly).
    wr0 = layers[0].router_w.to(torch.float64)
    b0 = layers[0].router_b.to(torch.float64)
    rows, redraws = [], {}
    for t in range(wl.T):
        for a in range(max_attempts):
            row = _draw_row(wl, t, a)
            if wl.margin <= 0 and accept_row is None:
                break
            xin = row.to(torch.float64)
            if wl.norm:
                # the first layer routes the RMS-normalised row; the norm only
                # rescales per element, so evaluate it with a library routine.
                xin = torch.nn.functional.rms_norm(xin[None], (wl.H,), layers[0].norm_w.to(torch.float64),
                                                   eps=wl.rms_eps)[0]
            if (wl.margin <= 0 or _row_ok(xin @ wr0.T + b0, wl.k, wl.margin)) and \
                    (accept_row is None or accept_row(t, row)):
                break
        else:
            raise RuntimeError(f"margin rule failed for token {t} after {max_attempts} draws")
        if a:
            redraws[t] = a
        rows.append(row)
    x = torch.stack(rows)
    return Inputs(wl=wl, x=x, layers=layers, redraws=redraws)
