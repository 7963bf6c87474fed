"""Seeded synthetic workloads of the optimizer step (random draws only).

This module holds the workload definitions (shapes, dtypes, hyper-parameters)
and draws their inputs. It contains none of the method's arithmetic, so both the
CUDA path and the fp64 oracle can take their inputs from it.

Draws: one torch.Generator per workload on the target device, seeded with the
workload index minus one unless a seed is given; normal draws in fp32, then cast
(round-to-nearest-even) to the storage dtype.
"""

import dataclasses
from typing import List, Optional, Tuple

import torch

QUINTIC = (3.4445, -4.7750, 2.0315)


@dataclasses.dataclass
class Workload:
    index: int
    name: str
    kind: str                    # "sign" (Sign-Muon over simulated workers), "muon" or "dion"
    shapes: List[Tuple[int, int]]
    workers: int = 1             # Sign-Muon: simulated workers
    m_dtype: torch.dtype = torch.bfloat16
    g_dtype: torch.dtype = torch.bfloat16
    w_dtype: torch.dtype = torch.bfloat16
    compute: str = "bf16"
    g_std: float = 1.0
    m0_std: float = 0.0
    w_std: float = 0.0
    expert_scales: bool = False  # per-matrix gradient scale 10**U(-3, 0) (MoE experts)
    mu: float = 0.95
    lr: float = 0.02
    steps: int = 5
    coeffs: Tuple[float, float, float] = QUINTIC
    eps: float = 1e-7
    rank: int = 0                # Dion: rank r of the low-rank factors

    @property
    def elements(self):
        return sum(r * c for r, c in self.shapes)


def _gpt12():
    return [s for _ in range(12) for s in ((768, 2304), (768, 768), (768, 3072), (3072, 768))]


def _dense32():
    layer = [(4096, 4096)] * 4 + [(4096, 14336), (14336, 4096), (4096, 14336)]
    return [s for _ in range(32) for s in layer]


def _moe128():
    return [s for _ in range(128) for s in ((2048, 768), (2048, 768), (768, 2048))] + [(2048, 2048)]


WORKLOADS = {
    1: Workload(1, "signmuon_64x128_f32_w4", "sign", [(64, 128)], workers=4,
                m_dtype=torch.float32, g_dtype=torch.float32, w_dtype=torch.float32,
                compute="f32", g_std=1.0, m0_std=0.0, w_std=0.0, mu=0.95, lr=0.02),
    2: Workload(2, "muon_gpt12_d768_bf16", "muon", _gpt12(), g_std=0.02, m0_std=0.01,
                w_std=0.02, mu=0.95, lr=0.02),
    3: Workload(3, "signmuon_4096sq_bf16_w8", "sign", [(4096, 4096)], workers=8, g_std=1.0,
                m0_std=1.0, w_std=0.02, mu=0.95, lr=1e-3),
    4: Workload(4, "muon_dense32_4096_14336_f32m", "muon", _dense32(), m_dtype=torch.float32,
                g_std=0.01, m0_std=0.01, w_std=0.02, mu=0.95, lr=0.02),
    5: Workload(5, "muon_moe128_2048x768_bf16", "muon", _moe128(), g_std=0.02, m0_std=0.01,
                w_std=0.02, expert_scales=True, mu=0.95, lr=0.02),
    # Dion on the same 12-layer d = 768 shapes with r = d / 4 (the page's rank sweep uses
    # d / 4, d / 8 and d / 16 at d = 768)
    6: Workload(6, "dion_gpt12_d768_r192", "dion", _gpt12(), g_std=0.02, m0_std=0.01,
                w_std=0.02, mu=0.95, lr=0.02, rank=192),
}


def workload(index):
    return WORKLOADS[index]


def _normal(gen, shape, std, dtype, device):
    if std == 0.0:
        return torch.zeros(shape, dtype=dtype, device=device)
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def generate(wl: Workload, device, seed: Optional[int] = None, shapes=None):
    """Inputs of one step: dict with lists W, M, G (Sign-Muon: one W, W_n of M and G;
    Dion adds Q, the previous right factors: n x r float32 standard normal draws).

    `shapes` replaces the workload's shape list (smaller parity cases of the same recipe).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.index - 1 if seed is None else seed)
    shapes = list(shapes) if shapes is not None else list(wl.shapes)
    if wl.kind == "sign":
        (R, C), = shapes
        W = [_normal(gen, (R, C), wl.w_std, wl.w_dtype, device)]
        M0 = _normal(gen, (R, C), wl.m0_std, wl.m_dtype, device)   # shared initial momentum
        M = [M0.clone() for _ in range(wl.workers)]
        G = [_normal(gen, (R, C), wl.g_std, wl.g_dtype, device) for _ in range(wl.workers)]
        return {"W": W, "M": M, "G": G}
    W, M, G = [], [], []
    if wl.expert_scales:
        # one scale per expert (three matrices each); the trailing dense block keeps scale 1
        n_exp = (len(shapes) - 1) // 3
        u = torch.rand(n_exp, generator=gen, dtype=torch.float32, device=device).cpu()
        scales = [10.0 ** (-3.0 + 3.0 * float(v)) for v in u for _ in range(3)] + [1.0]
    else:
        scales = [1.0] * len(shapes)
    for (R, C), sc in zip(shapes, scales):
        W.append(_normal(gen, (R, C), wl.w_std, wl.w_dtype, device))
        M.append(_normal(gen, (R, C), wl.m0_std, wl.m_dtype, device))
        G.append(_normal(gen, (R, C), wl.g_std * sc, wl.g_dtype, device))
    if wl.kind == "dion":
        Q = [_normal(gen, (C, wl.rank), 1.0, torch.float32, device) for (R, C) in shapes]
        return {"W": W, "M": M, "G": G, "Q": Q}
    return {"W": W, "M": M, "G": G}
