"""Seeded synthetic inputs for the five workloads, shared by tests and bench.

This module holds no arithmetic of the FP8 method: it only draws tensors.
The CUDA library and the CPU oracle both receive the very bytes drawn here.
Tensors are bf16 torch tensors (or fp32 router logits).  Draw order and
seeds are fixed per workload:

  tiny dense      seed 0: X [128,512] ~ N(0,1), columns 5 and 260 scaled x100;
                  W [256,512] ~ N(0, 0.02^2)
  dense linear    seed 0: X [4096,7168] ~ 0.5 * Student-t(3); W [7168,7168] ~ N(0, 0.02^2)
  MoE up-proj     seed 0: X [4096,7168] ~ N(0,1); logits [4096,256] ~ N(0,1);
                  W [256][4096][7168] ~ N(0, 0.02^2), drawn expert by expert
  MoE down-proj   seed 1: logits [4096,256] ~ N(0,1); g, u [32768,2048] ~ N(0,1),
                  h = bf16(silu(g) * u); W [256][7168][2048] ~ N(0, 0.02^2)
  Wgrad           seed 0: dY [8192,7168] ~ N(0, 1e-3^2); X [8192,7168] ~ N(0,1)

Everything is drawn with torch's CPU generator except the two expert weight
stacks, which are too large for host memory at full size: each expert's
matrix is drawn with a generator seeded (seed, 1000 + e) on the device that
will hold it, so a test can redraw any single expert on the same device.
Student-t(3) is drawn as Z / sqrt(V / 3) with V the sum of three squared
standard normals.  Each tensor is rounded to bf16 once.
"""
from __future__ import annotations

import torch

HIDDEN = 7168
EXPERTS = 256
TOPK = 8
INTER = 2048

# name -> shapes (for reporting only)
CONFIGS = {
    "tiny_dense": dict(M=128, N=256, K=512),
    "dense_linear": dict(M=4096, N=7168, K=7168),
    "moe_up": dict(T=4096, E=EXPERTS, topk=TOPK, N=2 * INTER, K=HIDDEN),
    "moe_down": dict(T=4096, E=EXPERTS, topk=TOPK, N=HIDDEN, K=INTER),
    "wgrad": dict(T=8192, H=HIDDEN),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device) * std


def _student_t3(shape, g) -> torch.Tensor:
    z = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.zeros(shape, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(shape, generator=g, dtype=torch.float32)
        v += n * n
    return z / torch.sqrt(v / 3.0)


def tiny_dense(seed: int = 0, M: int = 128, N: int = 256, K: int = 512,
               outlier_cols=(5, 260)):
    g = _gen(seed)
    x = _normal((M, K), 1.0, g)
    for c in outlier_cols:
        if c < K:
            x[:, c] *= 100.0
    w = _normal((N, K), 0.02, g)
    return dict(x=x.to(torch.bfloat16), w=w.to(torch.bfloat16))


def dense_linear(seed: int = 0, M: int = 4096, N: int = HIDDEN, K: int = HIDDEN):
    g = _gen(seed)
    x = 0.5 * _student_t3((M, K), g)
    w = _normal((N, K), 0.02, g)
    return dict(x=x.to(torch.bfloat16), w=w.to(torch.bfloat16))


def expert_weight(seed: int, e: int, N: int, K: int, device="cpu") -> torch.Tensor:
    """One expert's bf16 [N, K] weight, redrawable on its own."""
    g = _gen(seed * 1_000_003 + 1000 + e, device)
    return _normal((N, K), 0.02, g, device).to(torch.bfloat16)


def expert_weights(seed: int, E: int, N: int, K: int, device="cpu") -> torch.Tensor:
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    for e in range(E):
        out[e] = expert_weight(seed, e, N, K, device)
    return out


def moe_up(seed: int = 0, T: int = 4096, E: int = EXPERTS, N: int = 2 * INTER,
           K: int = HIDDEN, weights_device="cpu", with_weights=True):
    g = _gen(seed)
    x = _normal((T, K), 1.0, g).to(torch.bfloat16)
    logits = _normal((T, E), 1.0, g)
    out = dict(x=x, logits=logits)
    if with_weights:
        out["w"] = expert_weights(seed, E, N, K, weights_device)
    return out


def moe_down(seed: int = 1, T: int = 4096, E: int = EXPERTS, topk: int = TOPK,
             N: int = HIDDEN, K: int = INTER, weights_device="cpu", with_weights=True):
    g = _gen(seed)
    logits = _normal((T, E), 1.0, g)
    gate_in = _normal((T * topk, K), 1.0, g)
    up = _normal((T * topk, K), 1.0, g)
    h = (torch.nn.functional.silu(gate_in) * up).to(torch.bfloat16)
    out = dict(logits=logits, h=h)
    if with_weights:
        out["w"] = expert_weights(seed, E, N, K, weights_device)
    return out


def wgrad(seed: int = 0, T: int = 8192, H: int = HIDDEN):
    g = _gen(seed)
    dy = _normal((T, H), 1e-3, g).to(torch.bfloat16)
    x = _normal((T, H), 1.0, g).to(torch.bfloat16)
    return dict(dy=dy, x=x)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its raw bits (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(a) -> torch.Tensor:
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
