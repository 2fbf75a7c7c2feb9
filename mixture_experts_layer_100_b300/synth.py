"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module draws inputs only: token activations, router and expert weights,
the routing bias, and stand-alone affinity scores or expert choices for the
routing and permutation checks. It holds none of the layer's arithmetic, so
both the CUDA path and the CPU oracle may take their inputs from it.

Shapes and value distributions follow the DeepSeek-V3 pages:
  * 256 routed experts + 1 shared expert, top-8, width 7168
    ("Deepseek-v3技术报告简报", p2hp.com, section 2 Pretraining);
  * parameter init std 0.006 (same page, section 3 Training Hyperparameters);
  * the per-token group ("node") limit of 4
    ("DeepSeek-V3技术报告" digest, mpbf.cn, section 2.2 and section 3.3).
The pages publish no dataset or checkpoint for this layer, so every tensor
here is random and seeded.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

INIT_STD = 0.006  # parameter init std (p2hp.com digest, section 3)

# Strength of the rank-8 routing-skew component of the V3-shaped workloads.
# Picked once with oracle/calibrate_zipf.py (seed 0): the log-log slope of
# the sorted raw expert load (bias 0) over its top ranks steepens with alpha
# and levels off near -0.91 (the other K-2 picks of every token add a flat
# floor), so alpha = 5 is the value closest to the -1.1 aimed at; the
# hottest expert then carries about 12x the mean load.
ZIPF_ALPHA = 5.0
ZIPF_EXPONENT = 1.1
ZIPF_COMPONENTS = 8


@dataclasses.dataclass(frozen=True)
class Preset:
    """Shape, dtype and input recipe of one workload."""

    name: str
    T: int            # tokens
    d: int            # hidden width
    E: int            # routed experts
    G: int            # expert groups (the pages' "nodes")
    K: int            # routed experts per token
    M: int            # groups a token may use
    I: int            # expert intermediate width
    S: int            # shared experts
    dtype: str        # "f32" or "bf16": activations, master weights, output
    expert_dtype: str  # "f32", "bf16", "e4m3" or "e4m3_ue8m0" (power-of-two scales): expert GEMM operands
    bias: str         # "zeros", "u0.01" or "u0.02"
    zipf: bool        # add the rank-8 routing-skew component to x
    steps: int        # forward + bias-update steps the workload runs
    gamma: float = 1e-3
    group_topk: int = 2
    seed: int = 0
    combine: str = "gather"  # how the layer call combines the routed rows: "gather" or "scatter_add"

    def replace(self, **kw) -> "Preset":
        return dataclasses.replace(self, **kw)


PRESETS = {
    p.name: p
    for p in [
        Preset("tiny_t256_d512_e16_fp32", T=256, d=512, E=16, G=4, K=4, M=2,
               I=256, S=1, dtype="f32", expert_dtype="f32", bias="zeros",
               zipf=False, steps=10),
        Preset("mid_t4096_d2048_e64_bf16", T=4096, d=2048, E=64, G=8, K=6,
               M=3, I=1408, S=2, dtype="bf16", expert_dtype="bf16",
               bias="u0.01", zipf=False, steps=1),
        Preset("v3_t16384_d7168_e256_bf16", T=16384, d=7168, E=256, G=8, K=8,
               M=4, I=2048, S=1, dtype="bf16", expert_dtype="bf16",
               bias="zeros", zipf=True, steps=1),
        Preset("v3_decode_t64_bf16", T=64, d=7168, E=256, G=8, K=8, M=4,
               I=2048, S=1, dtype="bf16", expert_dtype="bf16", bias="u0.02",
               zipf=False, steps=1),
        Preset("v3_decode_t512_bf16", T=512, d=7168, E=256, G=8, K=8, M=4,
               I=2048, S=1, dtype="bf16", expert_dtype="bf16", bias="u0.02",
               zipf=False, steps=1),
        Preset("v3_t32768_d7168_e256_fp8", T=32768, d=7168, E=256, G=8, K=8,
               M=4, I=2048, S=1, dtype="bf16", expert_dtype="e4m3",
               bias="zeros", zipf=True, steps=50),
        # the same workload with power-of-two (UE8M0) tile scales
        Preset("v3_t32768_d7168_e256_fp8_ue8m0", T=32768, d=7168, E=256, G=8, K=8,
               M=4, I=2048, S=1, dtype="bf16", expert_dtype="e4m3_ue8m0",
               bias="zeros", zipf=True, steps=50),
    ]
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + tensor_id)
    return g


@dataclasses.dataclass
class Weights:
    w_router: torch.Tensor  # [E, d]
    w13: torch.Tensor       # [E, 2I, d]: rows 0..I-1 gate (W1), I..2I-1 up (W3)
    w2: torch.Tensor        # [E, d, I]
    ws13: torch.Tensor      # [S, 2I, d]
    ws2: torch.Tensor       # [S, d, I]


def _normal(shape, std, seed, tid, device, dtype):
    g = _gen(seed, tid, device)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(dtype)


def make_weights(p: Preset, device="cpu", zero_routed: bool = False) -> Weights:
    """Router and expert weights ~ N(0, 0.006^2), cast to the preset dtype."""
    dt = torch_dtype(p.dtype)
    w_router = _normal((p.E, p.d), INIT_STD, p.seed, 1, device, dt)
    if zero_routed:
        w13 = torch.zeros((p.E, 2 * p.I, p.d), dtype=dt, device=device)
        w2 = torch.zeros((p.E, p.d, p.I), dtype=dt, device=device)
    else:
        w13 = _normal((p.E, 2 * p.I, p.d), INIT_STD, p.seed, 2, device, dt)
        w2 = _normal((p.E, p.d, p.I), INIT_STD, p.seed, 3, device, dt)
    ws13 = _normal((p.S, 2 * p.I, p.d), INIT_STD, p.seed, 4, device, dt)
    ws2 = _normal((p.S, p.d, p.I), INIT_STD, p.seed, 5, device, dt)
    return Weights(w_router, w13, w2, ws13, ws2)


def zipf_directions(p: Preset, w_router: torch.Tensor):
    """The rank-8 skew component: unit directions aligned with 16 router rows.

    Direction j is the normalised sum of router rows e_{2j} and e_{2j+1} for
    16 seeded distinct experts. Returns (directions [8, d] fp32, experts [16]).
    """
    g = _gen(p.seed, 6, "cpu")
    experts = torch.randperm(p.E, generator=g)[: 2 * ZIPF_COMPONENTS]
    w = w_router.float().cpu()
    v = w[experts[0::2]] + w[experts[1::2]]
    v = v / v.norm(dim=1, keepdim=True)
    return v, experts


def zipf_component_choice(p: Preset, T: Optional[int] = None) -> torch.Tensor:
    """Per token, the skew direction j drawn with P(j) proportional to (j+1)^-1.1."""
    T = p.T if T is None else T
    probs = torch.tensor([(j + 1) ** -ZIPF_EXPONENT for j in range(ZIPF_COMPONENTS)],
                         dtype=torch.float64)
    g = _gen(p.seed, 7, "cpu")
    return torch.multinomial(probs, T, replacement=True, generator=g)


def make_x(p: Preset, w_router: torch.Tensor, device="cpu",
           alpha: Optional[float] = None) -> torch.Tensor:
    """Token activations x [T, d]: z ~ N(0,1), plus alpha * v_j(t) when skewed."""
    z = _normal((p.T, p.d), 1.0, p.seed, 8, device, torch.float32)
    if p.zipf:
        a = ZIPF_ALPHA if alpha is None else alpha
        v, _ = zipf_directions(p, w_router)
        j = zipf_component_choice(p)
        z += a * v.to(device)[j.to(device)]
    return z.to(torch_dtype(p.dtype))


def make_bias(p: Preset, device="cpu") -> torch.Tensor:
    """Initial routing bias b [E] fp32."""
    if p.bias == "zeros":
        return torch.zeros(p.E, dtype=torch.float32, device=device)
    lim = {"u0.01": 0.01, "u0.02": 0.02}[p.bias]
    g = _gen(p.seed, 9, "cpu")
    b = (torch.rand(p.E, generator=g, dtype=torch.float32) * 2 - 1) * lim
    return b.to(device)


def make_scores(T: int, E: int, seed: int, kind: str = "uniform") -> torch.Tensor:
    """Stand-alone fp32 affinity scores in (0, 1) for the routing checks.

    kinds:
      "uniform"  - U(0.05, 0.95);
      "dyadic"   - multiples of 1/64, so that many values tie exactly;
      "const"    - every score 0.5 (everything ties);
      "skewed"   - U(0.2, 0.6) plus a per-expert offset that falls off as
                   rank^-1.1, so that raw loads are uneven and the bias has
                   something to balance.
    """
    g = _gen(seed, 10, "cpu")
    if kind == "uniform":
        s = torch.rand((T, E), generator=g) * 0.9 + 0.05
    elif kind == "dyadic":
        s = torch.randint(1, 64, (T, E), generator=g).float() / 64.0
    elif kind == "const":
        s = torch.full((T, E), 0.5)
    elif kind == "skewed":
        perm = torch.randperm(E, generator=g)
        off = torch.empty(E)
        off[perm] = 0.3 * torch.arange(1, E + 1, dtype=torch.float32) ** -ZIPF_EXPONENT
        s = torch.rand((T, E), generator=g) * 0.4 + 0.2 + off
    else:
        raise ValueError(kind)
    return s.float().contiguous()


def make_topk_idx(T: int, E: int, K: int, seed: int) -> torch.Tensor:
    """Random expert choices [T, K] int32, K distinct experts per token."""
    g = _gen(seed, 11, "cpu")
    keys = torch.rand((T, E), generator=g)
    return keys.argsort(dim=1)[:, :K].to(torch.int32).contiguous()
