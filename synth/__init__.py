"""Seeded synthetic inputs for the owner-side Muon update.

This module holds only random-number recipes and shape lists.  It contains
none of the update's arithmetic, so the CPU oracle (``oracle/``) and the CUDA
path can both draw their inputs from it without sharing any of the method.

Every tensor is drawn with a ``torch.Generator`` seeded explicitly: fp32 normal
samples first, then scaled, then cast to the storage dtype (bf16 by rounding to
nearest even, which is what ``Tensor.to(torch.bfloat16)`` does).

Workloads (sizes follow the Llama-style and synthetic shapes the DMuon
technical summary's evaluation stands in for; the pages publish no dataset or
weights we could use):

* ``c1``  one 128x256 fp32 matrix, N(0,1), seed 0.
* ``c2``  16 square 1024x1024 bf16 gradients, N(0, 0.02^2), seed 1.
* ``c3``  a 32-layer d=4096, ffn=14336 transformer: per layer q,k,v,o 4096x4096,
          gate/up 4096x14336, down 14336x4096; bf16 grads N(0, (1e-3)^2), seed 2.
* ``c4``  512 matrices whose shape is drawn uniformly from
          {256x1024, 512x2048, 768x3072}; grad = rank-8 Gaussian product / sqrt(8)
          plus N(0, (1e-4)^2) noise, summed in fp32 then cast to bf16, seed 3.
* ``c5``  aspect-ratio sweep: m=1024, n in {1024..16384}, 8 matrices per shape,
          N(0,1) with row 0 scaled by 100, seed 4.

Weights W0 are N(0, 0.02^2) with seed 1000 + config number.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch

QUINTIC = (3.4445, -4.7750, 2.0315)
BETA = 0.95
LR = 0.02

C3_LAYERS = 32
C3_D = 4096
C3_FFN = 14336
C4_SHAPES = ((256, 1024), (512, 2048), (768, 3072))
C5_M = 1024
C5_NS = (1024, 2048, 4096, 8192, 16384)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def sha256_of(t: torch.Tensor) -> str:
    """SHA-256 of a tensor's raw bytes (CPU copy, contiguous)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return hashlib.sha256(t.numpy().tobytes()).hexdigest()


@dataclass
class Workload:
    """A list of matrices (shapes in input order) plus their tensors."""
    name: str
    shapes: list
    grads: list = field(default_factory=list)
    weights: list = field(default_factory=list)
    dtype: torch.dtype = torch.bfloat16
    steps: int = 5
    coeffs: tuple = QUINTIC
    beta: float = BETA
    lr: float = LR

    def flop_count(self) -> float:
        """Symmetric Gram-space count 3 s^2 l + (4T-3) s^3 per matrix."""
        tot = 0.0
        for (m, n) in self.shapes:
            s, l = min(m, n), max(m, n)
            t = self.steps
            tot += 3.0 * s * s * l + (4 * t - 3) * float(s) ** 3 if t > 0 else 3.0 * s * s * l
        return tot


def normal(shape, std, seed, device="cpu", dtype=torch.float32):
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def c1(device="cpu") -> Workload:
    g = normal((128, 256), 1.0, 0, device)
    w = normal((128, 256), 0.02, 1001, device)
    return Workload("c1", [(128, 256)], [g], [w], dtype=torch.float32)


def c2(device="cpu", batch=16, size=1024) -> Workload:
    g = normal((batch, size, size), 0.02, 1, device, torch.bfloat16)
    w = normal((batch, size, size), 0.02, 1002, device, torch.bfloat16)
    return Workload("c2", [(size, size)] * batch, list(g.unbind(0)), list(w.unbind(0)))


def c3_shapes(layers=C3_LAYERS, d=C3_D, ffn=C3_FFN):
    out = []
    for _ in range(layers):
        out += [(d, d)] * 4 + [(d, ffn), (d, ffn), (ffn, d)]
    return out


def c3(device="cpu", layers=C3_LAYERS, d=C3_D, ffn=C3_FFN) -> Workload:
    """Grads and weights of the Llama-style model, one generator stream per
    tensor kind (seed 2 for grads, 1003 for weights), drawn in shape order."""
    shapes = c3_shapes(layers, d, ffn)
    gg, gw = _gen(2, device), _gen(1003, device)
    grads, ws = [], []
    for (m, n) in shapes:
        x = torch.randn(m, n, generator=gg, device=device)
        grads.append(x.mul_(1e-3).to(torch.bfloat16))
        y = torch.randn(m, n, generator=gw, device=device)
        ws.append(y.mul_(0.02).to(torch.bfloat16))
    return Workload("c3", shapes, grads, ws)


def c4_shapes(count=512, seed=3):
    g = _gen(seed)
    idx = torch.randint(0, len(C4_SHAPES), (count,), generator=g)
    return [C4_SHAPES[int(i)] for i in idx]


def c4(device="cpu", count=512) -> Workload:
    shapes = c4_shapes(count)
    g = _gen(3 + 100, device)
    gw = _gen(1004, device)
    grads, ws = [], []
    for (m, n) in shapes:
        a = torch.randn(m, 8, generator=g, device=device)
        b = torch.randn(n, 8, generator=g, device=device)
        noise = torch.randn(m, n, generator=g, device=device).mul_(1e-4)
        grads.append(((a @ b.T) / (8 ** 0.5) + noise).to(torch.bfloat16))
        ws.append(torch.randn(m, n, generator=gw, device=device).mul_(0.02).to(torch.bfloat16))
    return Workload("c4", shapes, grads, ws)


def c5(device="cpu", n=4096, batch=8, dtype=torch.bfloat16, steps=5, m=C5_M) -> Workload:
    """One shape of the aspect-ratio sweep (seed 4 + n so shapes are independent)."""
    g = normal((batch, m, n), 1.0, 4 + n, device)
    g[:, 0, :] *= 100.0
    g = g.to(dtype)
    w = normal((batch, m, n), 0.02, 1005 + n, device, dtype)
    return Workload(f"c5_n{n}", [(m, n)] * batch, list(g.unbind(0)), list(w.unbind(0)),
                    dtype=dtype, steps=steps)


def random_matrix(m, n, seed, dtype=torch.float32, std=1.0, device="cpu"):
    return normal((m, n), std, seed, device, dtype)


def low_rank(m, n, rank, noise, seed, dtype=torch.float32, device="cpu"):
    g = _gen(seed, device)
    a = torch.randn(m, rank, generator=g, device=device)
    b = torch.randn(n, rank, generator=g, device=device)
    x = (a @ b.T) / (rank ** 0.5) + torch.randn(m, n, generator=g, device=device) * noise
    return x.to(dtype)
