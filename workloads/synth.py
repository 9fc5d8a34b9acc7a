"""Seeded input generators and the five workload definitions.

Every tensor is drawn on the host with ``torch.Generator('cpu')`` from a fixed
seed, so the oracle and the CUDA path see identical bytes. Shapes and value
distributions follow the BitLinear workloads:

* weights W [N][K] fp32, N(0, 0.02^2), or 0.02 * Student-t(nu=4) for the
  7B-class stack;
* activations x [M][K], N(0, 1), cast to bf16 (fp32 for the small CPU-scale
  case); the batched-decode case scales 1% of the channels by 20 (outlier
  channels, the failure mode per-token absmax must survive).

Nothing here quantises, rounds to a code or scales by a statistic of the data:
the generators only draw numbers.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

WEIGHT_STD = 0.02


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def gaussian_weights(n: int, k: int, seed: int, std: float = WEIGHT_STD) -> torch.Tensor:
    """W ~ N(0, std^2), fp32 [n][k], row-major (nn.Linear layout: out x in)."""
    w = torch.randn((n, k), generator=_gen(seed), dtype=torch.float32)
    return (w * std).contiguous()


def student_t_weights(n: int, k: int, seed: int, nu: int = 4, std: float = WEIGHT_STD) -> torch.Tensor:
    """W = std * T_nu, with T = Z / sqrt(V/nu), V a sum of nu squared normals."""
    g = _gen(seed)
    z = torch.randn((n, k), generator=g, dtype=torch.float64)
    v = torch.zeros((n, k), dtype=torch.float64)
    for _ in range(nu):
        v += torch.randn((n, k), generator=g, dtype=torch.float64) ** 2
    t = z / torch.sqrt(v / nu)
    return (t * std).to(torch.float32).contiguous()


def student_t_weights_on(device, n: int, k: int, seed: int, nu: int = 4, std: float = WEIGHT_STD) -> torch.Tensor:
    """The Student-t recipe drawn by a seeded generator on ``device`` (fast for
    multi-GB weight stacks; same distribution, different draws from the CPU
    generator, so only for timing)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    z = torch.randn((n, k), generator=g, dtype=torch.float32, device=device)
    v = torch.zeros((n, k), dtype=torch.float32, device=device)
    for _ in range(nu):
        v += torch.randn((n, k), generator=g, dtype=torch.float32, device=device) ** 2
    return (z / torch.sqrt(v / nu) * std).contiguous()


def gaussian_activations_on(device, m: int, k: int, seed: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """x ~ N(0, 1) drawn by a seeded generator on ``device``, then cast (timing only)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn((m, k), generator=g, dtype=torch.float32, device=device).to(dtype).contiguous()


def gaussian_activations(m: int, k: int, seed: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """x ~ N(0, 1) drawn in fp32, then cast to ``dtype``."""
    x = torch.randn((m, k), generator=_gen(seed), dtype=torch.float32)
    return x.to(dtype).contiguous()


def outlier_activations(m: int, k: int, seed: int, frac: float = 0.01, gain: float = 20.0,
                        dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """x ~ N(0, 1) with round(frac*K) channels multiplied by ``gain``.

    The channel set is ``randperm(K)[:round(frac*K)]`` from the same generator,
    the same channels for every token; the gain is applied in fp32 before the
    cast to ``dtype``.
    """
    g = _gen(seed)
    x = torch.randn((m, k), generator=g, dtype=torch.float32)
    n_out = int(round(frac * k))
    idx = torch.randperm(k, generator=g)[:n_out]
    x[:, idx] *= gain
    return x.to(dtype).contiguous()


@dataclass(frozen=True)
class Projection:
    """One BitLinear projection: x [m][k] against W [n][k]."""

    name: str
    m: int
    k: int
    n: int
    w_seed: int
    x_seed: int
    w_dist: str = "gauss"          # "gauss" | "t4"
    x_dist: str = "gauss"          # "gauss" | "outlier"
    x_dtype: str = "bf16"          # "bf16" | "f32"


def make_projection_inputs(p: Projection):
    """Returns (W fp32 [n][k], x [m][k]) for a projection, on the CPU."""
    if p.w_dist == "gauss":
        w = gaussian_weights(p.n, p.k, p.w_seed)
    elif p.w_dist == "t4":
        w = student_t_weights(p.n, p.k, p.w_seed)
    else:
        raise ValueError(p.w_dist)
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[p.x_dtype]
    if p.x_dist == "gauss":
        x = gaussian_activations(p.m, p.k, p.x_seed, dt)
    elif p.x_dist == "outlier":
        x = outlier_activations(p.m, p.k, p.x_seed, dtype=dt)
    else:
        raise ValueError(p.x_dist)
    return w, x


@dataclass
class Workload:
    name: str
    description: str
    projections: List[Projection] = field(default_factory=list)
    layers: int = 1                  # >1: the projection list is one layer, repeated with new weights


def _stack_layer_projections(m: int, layer: int) -> List[Projection]:
    shapes = [("qkv", 4096, 12288), ("o", 4096, 4096), ("up", 4096, 11008), ("down", 11008, 4096)]
    out = []
    for j, (nm, k, n) in enumerate(shapes):
        out.append(Projection(f"L{layer}.{nm}", m, k, n, w_seed=1000 + 4 * layer + j, x_seed=5000 + j,
                              w_dist="t4", x_dist="gauss"))
    return out


def stack_projections(m: int, layers: int = 32) -> List[Projection]:
    out: List[Projection] = []
    for layer in range(layers):
        out.extend(_stack_layer_projections(m, layer))
    return out


WORKLOADS = {
    # CPU-oracle scale: every output is checked element by element.
    "cpu_small": Workload(
        "cpu_small", "single BitLinear M=4 K=256 N=256, fp32 activations",
        [Projection("p", 4, 256, 256, w_seed=0, x_seed=1, x_dtype="f32")]),
    # Decode GEMV at 2B-class shapes (the benchmark's default step).
    "decode_2b": Workload(
        "decode_2b", "decode GEMV M=1, K=2560->N=6912 and K=6912->N=2560, bf16 activations",
        [Projection("up", 1, 2560, 6912, w_seed=10, x_seed=20),
         Projection("down", 1, 6912, 2560, w_seed=11, x_seed=21)]),
    # Batched decode with outlier channels.
    "skinny_2b": Workload(
        "skinny_2b", "batched decode M in {8,32,64}, K=2560, N in {2560,6912}, 1% channels x20",
        [Projection(f"m{m}_n{n}", m, 2560, n, w_seed=30 + ni, x_seed=40 + mi, x_dist="outlier")
         for mi, m in enumerate((8, 32, 64)) for ni, n in enumerate((2560, 6912))]),
    # Prefill.
    "prefill_2b": Workload(
        "prefill_2b", "prefill GEMM M=2048, K=2560->N=6912 and K=6912->N=2560",
        [Projection("up", 2048, 2560, 6912, w_seed=50, x_seed=60),
         Projection("down", 2048, 6912, 2560, w_seed=51, x_seed=61)]),
    # 7B-class stack: 32 layers x 4 projections, each layer packed once.
    "stack_7b_decode": Workload(
        "stack_7b_decode", "7B-class stack, 32 layers x {qkv,o,up,down}, M=1, Student-t(4) weights",
        stack_projections(1), layers=32),
    "stack_7b_prefill": Workload(
        "stack_7b_prefill", "7B-class stack, 32 layers x {qkv,o,up,down}, M=2048, Student-t(4) weights",
        stack_projections(2048), layers=32),
}


def workload(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def describe(name: Optional[str] = None) -> str:
    names = [name] if name else sorted(WORKLOADS)
    return "\n".join(f"{n}: {WORKLOADS[n].description}" for n in names)
