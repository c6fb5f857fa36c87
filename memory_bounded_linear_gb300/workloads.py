"""Seeded synthetic workloads for the fused linear cross-entropy path.

This module only *draws inputs*: hidden states H [N, d], the vocabulary projection W [V, d]
and integer labels y [N].  It holds none of the method's arithmetic (no logits, no
log-softmax, no gradients), so that the CUDA path and the float64 oracle can both be fed
from it without sharing any code that computes the loss.

The five workloads are language-model-head shapes (hidden size d, vocabulary V, tokens N):

* ``tiny-fp32``                      N=256,    d=256,  V=4096,   strip 512, fp32, uniform labels
* ``n4096-d2048-v151936``            N=4096,   d=2048, V=151936, strip 8192, Zipf(1.1) labels
* ``n16384-d4096-v131072-ignore10``  N=16384,  d=4096, V=131072, strip 16384, W~N(0, 0.02^2),
                                     uniform labels, 10% of rows set to ignore_index=-100
* ``n65536-d2048-v151936``           N=65536,  d=2048, V=151936, strips {4096, 8192, 16384, 32768}
* ``n32768-d6144-v151552-outliers``  N=32768,  d=6144, V=151552, strip 16384, H~0.5*N(0,1),
                                     1% of W rows scaled x8, Zipf(1.1) labels, sum reduction

Draw recipe (fixed order, one ``torch.Generator`` per tensor, seeded ``seed + k``):
  k=0 H ~ N(0,1) * h_scale;  k=1 W ~ N(0,1) * w_std;  k=2 outlier rows of W (a seeded
  permutation, the first floor(frac*V) rows are scaled);  k=3 labels;  k=4 ignored rows
  (a seeded permutation, the first round(frac*N) rows get ignore_index).
Zipf(s) labels: rank k in 1..V drawn with P(k) proportional to k^-s by inverse-CDF sampling
of a uniform draw, then mapped through a seeded permutation of the vocabulary.
H and W are drawn in fp32 and rounded once to the compute dtype; the oracle receives exactly
those rounded values, upcast to float64.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    d: int
    V: int
    strip_V: int
    dtype: str                 # "bf16" or "f32": the dtype of H and W
    h_scale: float = 1.0       # H ~ N(0,1) * h_scale
    w_std: Optional[float] = None   # None -> 1/sqrt(d), i.e. W ~ N(0, 1/d)
    labels: str = "uniform"    # "uniform" or "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    outlier_frac: float = 0.0  # fraction of W rows scaled by outlier_scale
    outlier_scale: float = 8.0
    reduction: str = "mean"
    strip_sweep: tuple = ()

    def with_sizes(self, N=None, d=None, V=None, strip_V=None, **kw) -> "Workload":
        """Same distributions at other sizes (used for reduced-size parity cases)."""
        return dataclasses.replace(
            self,
            N=self.N if N is None else N,
            d=self.d if d is None else d,
            V=self.V if V is None else V,
            strip_V=self.strip_V if strip_V is None else strip_V,
            **kw,
        )

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs of one forward+backward: 8*N*d*V (logits, recomputed logits,
        dH and dW contractions, 2*N*d*V each)."""
        return 8 * self.N * self.d * self.V


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-fp32", N=256, d=256, V=4096, strip_V=512, dtype="f32"),
        Workload("n4096-d2048-v151936", N=4096, d=2048, V=151936, strip_V=8192,
                 dtype="bf16", labels="zipf"),
        Workload("n16384-d4096-v131072-ignore10", N=16384, d=4096, V=131072, strip_V=16384,
                 dtype="bf16", w_std=0.02, ignore_frac=0.10),
        Workload("n65536-d2048-v151936", N=65536, d=2048, V=151936, strip_V=8192,
                 dtype="bf16", labels="zipf", strip_sweep=(4096, 8192, 16384, 32768)),
        Workload("n32768-d6144-v151552-outliers", N=32768, d=6144, V=151552, strip_V=16384,
                 dtype="bf16", h_scale=0.5, labels="zipf", outlier_frac=0.01,
                 reduction="sum"),
        # The shape the Ring-DTP benchmark times in FP32 ("Flattening Every Memory Peak",
        # appendix C: N = 16,384, H = 7,168, V = 200,000); the pages give no distributions, so
        # the plain ones: H ~ N(0,1), W ~ N(0,1/d), uniform labels, mean reduction.
        Workload("n16384-d7168-v200000-fp32", N=16384, d=7168, V=200000, strip_V=16384,
                 dtype="f32"),
    ]
}

# The largest workload by FLOPs; the throughput figure is quoted on it.
HEADLINE = "n32768-d6144-v151552-outliers"


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def zipf_ranks(n: int, V: int, s: float, g: torch.Generator, device) -> torch.Tensor:
    """n draws of a rank in [0, V) with P(rank k-1) proportional to k^-s (inverse CDF)."""
    k = torch.arange(1, V + 1, dtype=torch.float64, device=device)
    cdf = torch.cumsum(k.pow(-s), 0)
    cdf = cdf / cdf[-1]
    u = torch.rand(n, generator=g, device=device, dtype=torch.float64)
    r = torch.searchsorted(cdf, u)
    return r.clamp_(max=V - 1)


def make_inputs(w: Workload, device="cpu", seed: int = 0):
    """Draw (H, W, labels) for workload ``w`` on ``device`` following the module recipe.

    Returns H [N, d] and W [V, d] in the workload dtype, labels [N] int64.
    """
    device = torch.device(device)
    N, d, V = w.N, w.d, w.V
    dt = torch_dtype(w.dtype)
    w_std = (1.0 / math.sqrt(d)) if w.w_std is None else w.w_std

    H = torch.randn(N, d, generator=_gen(device, seed + 0), device=device, dtype=torch.float32)
    if w.h_scale != 1.0:
        H.mul_(w.h_scale)
    H = H.to(dt)

    W = torch.randn(V, d, generator=_gen(device, seed + 1), device=device, dtype=torch.float32)
    W.mul_(w_std)
    n_out = int(math.floor(w.outlier_frac * V))
    if n_out > 0:
        rows = torch.randperm(V, generator=_gen(device, seed + 2), device=device)[:n_out]
        W[rows] *= w.outlier_scale
    W = W.to(dt)

    g3 = _gen(device, seed + 3)
    if w.labels == "uniform":
        labels = torch.randint(0, V, (N,), generator=g3, device=device, dtype=torch.int64)
    elif w.labels == "zipf":
        perm = torch.randperm(V, generator=g3, device=device)
        labels = perm[zipf_ranks(N, V, w.zipf_s, g3, device)]
    else:
        raise ValueError(f"unknown label distribution {w.labels!r}")

    n_ign = int(round(w.ignore_frac * N))
    if n_ign > 0:
        rows = torch.randperm(N, generator=_gen(device, seed + 4), device=device)[:n_ign]
        labels[rows] = IGNORE_INDEX
    return H.contiguous(), W.contiguous(), labels.contiguous()


def to_float64_numpy(t: torch.Tensor):
    """Exact upcast of a (possibly bf16) tensor to a float64 numpy array on the host."""
    return t.detach().to("cpu").to(torch.float64).numpy()
