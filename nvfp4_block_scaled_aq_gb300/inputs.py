"""Seeded synthetic inputs for the NVFP4 decode-projection path.

This module only draws random numbers of the shapes and distributions of the
workloads; it holds none of the method's arithmetic.  Both the CUDA path
(through the tests and the benchmark) and the CPU oracle consume the exact
tensors produced here, so the two sides see identical bytes.

Distributions (shapes of the Gemma-3-1B and Gemma-4-31B decoder projections
the AttnQuant docs benchmark, "Throughput" and landing page "What's
supported today"):
  * weights  W ~ N(0, 0.02^2) in bf16, each entry independently (p = 0.001)
    multiplied by 20 to plant outliers;
  * theta    W0 ~ N(0, 0.02^2), s = exp(0.1 z) with z ~ N(0, 1) (per-row
    lognormal(0, 0.1)), U [N, R] and V [K, R] ~ N(0, 0.01^2);
  * tokens   x ~ N(0, 1) in bf16.
Every draw uses its own torch.Generator seeded from (seed, layer, proj) as
seed + 1000 * layer + proj, so a tensor does not depend on what was drawn
before it.
"""
from dataclasses import dataclass

import torch

OUTLIER_P = 0.001
OUTLIER_SCALE = 20.0
W_STD = 0.02
UV_STD = 0.01
S_LOG_STD = 0.1


def seed_of(seed: int, layer: int = 0, proj: int = 0) -> int:
    return int(seed) + 1000 * int(layer) + int(proj)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weight(n: int, k: int, seed: int, device="cpu", outliers: bool = True,
           std: float = W_STD) -> torch.Tensor:
    """bf16 [n, k] ~ N(0, std^2), optionally with 0.1% x20 outliers."""
    g = _gen(seed, device)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    if outliers:
        mask = torch.rand((n, k), generator=g, device=device) < OUTLIER_P
        w[mask] *= OUTLIER_SCALE
        del mask
    return w.to(torch.bfloat16)


def tokens(m: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 activations [m, k] ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((m, k), generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


@dataclass
class Theta:
    W0: torch.Tensor  # bf16 [n, k]
    s: torch.Tensor   # fp32 [n]
    U: torch.Tensor   # bf16 [n, r]
    V: torch.Tensor   # bf16 [k, r]


def theta(n: int, k: int, r: int, seed: int, device="cpu",
          passthrough: bool = False) -> Theta:
    """Theta bundle of one projection; passthrough gives s = 1, U = V = 0."""
    W0 = weight(n, k, seed, device=device, outliers=False)
    if passthrough:
        s = torch.ones(n, device=device, dtype=torch.float32)
        U = torch.zeros((n, r), device=device, dtype=torch.bfloat16)
        V = torch.zeros((k, r), device=device, dtype=torch.bfloat16)
        return Theta(W0, s, U, V)
    g = _gen(seed + 7, device)
    s = torch.exp(S_LOG_STD * torch.randn(n, generator=g, device=device,
                                          dtype=torch.float32))
    U = (UV_STD * torch.randn((n, r), generator=g, device=device)).to(torch.bfloat16)
    V = (UV_STD * torch.randn((k, r), generator=g, device=device)).to(torch.bfloat16)
    return Theta(W0, s, U, V)


# Projection shapes (N, K) per decoder layer: fused QKV, o_proj, fused
# gate+up, down.  The 1B-shaped stack has 26 layers, the 31B-shaped 60.
LAYER_1B = ((1536, 1152), (1152, 1024), (13824, 1152), (1152, 6912))
LAYER_31B = ((8192, 5376), (5376, 4096), (43008, 5376), (5376, 21504))
# bf16 tied lm_head / embedding [vocab, hidden] of the ~31B and ~1B shapes
LM_HEAD_31B = (262144, 5376)
LM_HEAD_1B = (262144, 1152)
LAYERS_1B = 26
LAYERS_31B = 60
PROJ_NAMES = ("qkv", "o_proj", "gate_up", "down")


def bits_u16(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (copied to host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def from_bits_u16(a, device="cpu") -> torch.Tensor:
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
