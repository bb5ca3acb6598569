"""Seeded synthetic inputs for the five Muon-step workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no momentum, normalisation, iteration or update), so both
the CUDA path and the float64 oracle can be fed from it.

Workloads (shapes are [rows, cols] of the stored parameter):

* ``c1`` -- 4 fp32 gradients [64,256] then one [256,64], N(0,1) from NumPy
  ``default_rng(0)`` in that order; fp32 weights N(0, 0.02) from
  ``default_rng(1)``; zero momentum.
* ``c2`` -- 74 bf16 gradients [24,10240], N(0,1)*1e-3; fp32 weights N(0,0.02).
* ``c3`` -- MoE expert tensors, bf16 gradients [128,2048,768] and
  [128,768,2048]; every expert e has entries N(0, s_e^2) with
  s_e = 10**U(-4,-2) (log-uniform, geometric centre 1e-3); fp32 weights.
* ``c4`` -- Llama-3-8B parameter shapes, 32 layers x {q,o [4096,4096];
  k,v [1024,4096]; gate,up [14336,4096]; down [4096,14336]}: bf16 weights
  N(0,0.02), bf16 gradients N(0,1)*1e-3, fp32 momentum; 224 separate tensors.
* ``c5`` -- 8 x [8192,28672], 8 x [8192,8192], 4 x [16384,16384] bf16
  gradients N(0,1), plus 2 x [8192,8192] low-rank-plus-noise gradients
  U_r diag(s) V_r^T + N(0, 1e-3^2) with r = 64, s = 10**U(0,3) and U_r, V_r
  the Q factors of Gaussian matrices; fp32 weights.

Momentum always starts at zero.  Values are drawn in fp32 and rounded to
the stated storage dtype by ``Tensor.to`` (round to nearest even).
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

MU, NESTEROV, LR, WD = 0.95, True, 0.02, 0.01


def config_c1_numpy() -> List[Dict[str, np.ndarray]]:
    """The small fp32 case as NumPy arrays (two groups)."""
    rg = np.random.default_rng(0)
    rw = np.random.default_rng(1)
    g_a = np.stack([rg.standard_normal((64, 256)) for _ in range(4)]).astype(np.float32)
    g_b = rg.standard_normal((1, 256, 64)).astype(np.float32)
    w_a = np.stack([rw.standard_normal((64, 256)) * 0.02 for _ in range(4)]).astype(np.float32)
    w_b = (rw.standard_normal((1, 256, 64)) * 0.02).astype(np.float32)
    return [
        {"W": w_a, "G": g_a, "Mom": np.zeros_like(g_a)},
        {"W": w_b, "G": g_b, "Mom": np.zeros_like(g_b)},
    ]


def _torch():
    import torch
    return torch


def _gen(device, seed: int):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, device, seed, scale=1.0, dtype=None):
    torch = _torch()
    t = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    return t if dtype is None else t.to(dtype)


def _group(W, G, Mom, name):
    return {"W": W, "G": G, "Mom": Mom, "name": name}


def config_c1(device) -> List[dict]:
    torch = _torch()
    out = []
    for i, g in enumerate(config_c1_numpy()):
        out.append(_group(torch.from_numpy(g["W"]).to(device),
                          torch.from_numpy(g["G"]).to(device),
                          torch.zeros(g["G"].shape, dtype=torch.float32, device=device),
                          f"c1_g{i}"))
    return out


def config_c2(device, count: int = 74, seed: int = 2) -> List[dict]:
    torch = _torch()
    shape = (count, 24, 10240)
    G = _randn(shape, device, seed * 1000 + 1, 1e-3, torch.bfloat16)
    W = _randn(shape, device, seed * 1000 + 2, 0.02)
    return [_group(W, G, torch.zeros(shape, dtype=torch.float32, device=device), "c2")]


def config_c3(device, experts: int = 128, seed: int = 3) -> List[dict]:
    torch = _torch()
    out = []
    for gi, (r, c) in enumerate(((2048, 768), (768, 2048))):
        shape = (experts, r, c)
        sig_gen = np.random.default_rng(seed * 100 + gi)
        sig = 10.0 ** sig_gen.uniform(-4.0, -2.0, size=experts)
        G = _randn(shape, device, seed * 1000 + 10 * gi + 1)
        G.mul_(torch.tensor(sig, dtype=torch.float32, device=device).view(-1, 1, 1))
        G = G.to(torch.bfloat16)
        W = _randn(shape, device, seed * 1000 + 10 * gi + 2, 0.02)
        out.append(_group(W, G, torch.zeros(shape, dtype=torch.float32, device=device),
                          f"c3_{'gate_up' if gi == 0 else 'down'}"))
    return out


C4_LAYER = (("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
            ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336))


def config_c4(device, layers: int = 32, seed: int = 4,
              only: Optional[List[str]] = None) -> List[dict]:
    """224 separate [rows, cols] tensors (one group each, B = 1)."""
    torch = _torch()
    out = []
    for l in range(layers):
        for pi, (name, r, c) in enumerate(C4_LAYER):
            if only is not None and name not in only:
                continue
            s = seed * 100000 + l * 100 + pi * 2
            G = _randn((1, r, c), device, s + 1, 1e-3, torch.bfloat16)
            W = _randn((1, r, c), device, s + 2, 0.02, torch.bfloat16)
            out.append(_group(W, G, torch.zeros((1, r, c), dtype=torch.float32, device=device),
                              f"L{l}.{name}"))
    return out


def _qr_q(a, device):
    """Q factor of a tall Gaussian matrix, taken on the host in float64 (the
    factors are r x 64; this also keeps the generator free of the GPU's
    linear-algebra library)."""
    torch = _torch()
    q, _ = torch.linalg.qr(a.to("cpu", torch.float64))
    return q.to(device, torch.float32)


def lowrank_plus_noise(r_dim, c_dim, rank, device, seed):
    """U_r diag(s) V_r^T + N(0, 1e-3^2), s = 10**U(0,3)."""
    torch = _torch()
    U = _qr_q(_randn((r_dim, rank), device, seed + 1), device)
    V = _qr_q(_randn((c_dim, rank), device, seed + 2), device)
    sig_gen = np.random.default_rng(seed)
    s = torch.tensor(10.0 ** sig_gen.uniform(0.0, 3.0, size=rank), dtype=torch.float32,
                     device=device)
    G = (U * s) @ V.T
    G.add_(_randn((r_dim, c_dim), device, seed + 3, 1e-3))
    return G


def config_c5(device, seed: int = 5, scale_down: int = 1) -> List[dict]:
    """The large compute-bound sweep.  ``scale_down`` divides every dimension
    (for a smaller stand-in of the same structure)."""
    torch = _torch()
    d = lambda x: x // scale_down  # noqa: E731
    specs = [(8, d(8192), d(28672)), (8, d(8192), d(8192)), (4, d(16384), d(16384))]
    out = []
    for gi, (b, r, c) in enumerate(specs):
        G = _randn((b, r, c), device, seed * 1000 + 10 * gi + 1, 1.0, torch.bfloat16)
        W = _randn((b, r, c), device, seed * 1000 + 10 * gi + 2, 0.02)
        out.append(_group(W, G, torch.zeros((b, r, c), dtype=torch.float32, device=device),
                          f"c5_{b}x{r}x{c}"))
    out.append(config_c5_lowrank(device, seed, scale_down))
    return out


def config_c5_lowrank(device, seed: int = 5, scale_down: int = 1) -> dict:
    """The large sweep's last group alone: 2 low-rank-plus-noise gradients
    [8192, 8192] (same values as in ``config_c5``), fp32 weights."""
    torch = _torch()
    r = 8192 // scale_down
    lr_g = torch.stack([lowrank_plus_noise(r, r, max(1, 64 // scale_down), device,
                                           seed * 1000 + 100 + 10 * i) for i in range(2)])
    W = _randn((2, r, r), device, seed * 1000 + 99, 0.02)
    return _group(W, lr_g.to(torch.bfloat16),
                  torch.zeros((2, r, r), dtype=torch.float32, device=device), "c5_lowrank")


CONFIGS = {"c1": config_c1, "c2": config_c2, "c3": config_c3, "c4": config_c4, "c5": config_c5}

WORKLOAD_NAMES = {
    "c1": "4x[64,256]+1x[256,64] fp32, mu=0.95 nesterov, 5 NS steps",
    "c2": "74x[24,10240] bf16 grads, fp32 W/mom, 5 NS steps (tall-skinny, split-K)",
    "c3": "MoE experts bf16 [128,2048,768]+[128,768,2048], fp32 W/mom, 5 NS steps",
    "c4": "Llama-3-8B shapes x32 layers (224 tensors) bf16 W/G, fp32 mom, 5 NS steps",
    "c5": "8x[8192,28672]+8x[8192,8192]+4x[16384,16384]+2 low-rank [8192,8192], 5 NS steps",
}


def random_group(shape, g_dtype, w_dtype, device, seed, g_scale=1.0, mom_scale=0.0):
    """A generic seeded group for parity tests: G ~ N(0, g_scale^2) in g_dtype,
    W ~ N(0, 0.02^2) in w_dtype, Mom ~ N(0, mom_scale^2) fp32."""
    torch = _torch()
    G = _randn(shape, device, seed * 7 + 1, g_scale, g_dtype)
    W = _randn(shape, device, seed * 7 + 2, 0.02, w_dtype)
    if mom_scale:
        Mom = _randn(shape, device, seed * 7 + 3, mom_scale)
    else:
        Mom = torch.zeros(shape, dtype=torch.float32, device=device)
    return _group(W, G, Mom, f"rand{tuple(shape)}")
