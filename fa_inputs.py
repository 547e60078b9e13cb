"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and describes workload shapes; it holds
none of attention's arithmetic, so both the CUDA path and the float64 oracle can
take their inputs from it without sharing any of the method.

Workloads (shapes follow the pages' examples: the 1 x 32 x 8192 x 128 bf16
example of the 1point3acres FlashAttention write-up, and CS349E lecture 11's
N = 48, d = 16 gradient check):

=====  =======================================  ======  ======  =====================
name   shape B x H x N x d                       mask    dtype   distribution
=====  =======================================  ======  ======  =====================
tiny   1 x 1 x 48 x 16, scale 1/4                none    fp32    N(0,1), numpy seed 0
mha    1 x 32 x 2048 x 64                        none    bf16    N(0,1), torch seed 1
causal 1 x 32 x 8192 x 128                       causal  bf16    N(0,1), torch seed 2
ragged 4 x 16 x 4000 x 128                       causal  bf16    N(0,1), torch seed 3
long   1 x 8 x 32768 x 128                       causal  bf16    Q ~ N(0,16), rest N(0,1), seed 4
hd256  1 x 16 x 8192 x 256                       causal  bf16    N(0,1), torch seed 5
=====  =======================================  ======  ======  =====================

``hd256`` is the largest head dim the write-ups' d sweeps reach, at the
headline sequence length with half the heads (the same bytes per tensor).

The tiny workload mirrors CS349E lecture 11 demo 1: ``numpy.random.default_rng(0)``
and ``standard_normal((N, d))`` drawn in the order Q, K, V, G (G plays dO).  The
bf16 workloads draw float32 ``torch.randn`` in the order Q, K, V, dO from a CPU
generator seeded with the workload index and round to bf16 (round to nearest
even); the oracle upcasts exactly those rounded values.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "to_f64"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dtype: str  # "fp32" or "bf16"
    seed: int
    q_std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def counted_flops(self) -> float:
        """Five backward GEMMs: 10 B H N^2 d, halved under the causal mask."""
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 48, 16, False, "fp32", 0),
    "mha": Workload("mha", 1, 32, 2048, 64, False, "bf16", 1),
    "causal": Workload("causal", 1, 32, 8192, 128, True, "bf16", 2),
    "ragged": Workload("ragged", 4, 16, 4000, 128, True, "bf16", 3),
    "long": Workload("long", 1, 8, 32768, 128, True, "bf16", 4, q_std=4.0),
    "hd256": Workload("hd256", 1, 16, 8192, 256, True, "bf16", 5),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.with_(**overrides) if overrides else w


def make_inputs(w: Workload):
    """Return (Q, K, V, dO) as CPU torch tensors of the workload's dtype,
    shaped [B, H, N, d]."""
    if w.dtype == "fp32" and w.name == "tiny":
        rng = np.random.default_rng(w.seed)
        shape = (w.N, w.d)
        q, k, v, g = (rng.standard_normal(shape) for _ in range(4))
        out = []
        for x in (q * w.q_std, k, v, g):
            t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
            out.append(t.reshape(1, 1, w.N, w.d).expand(w.B, w.H, w.N, w.d).contiguous())
        return tuple(out)
    gen = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = []
    for i in range(4):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        if i == 0 and w.q_std != 1.0:
            x = x * w.q_std
        out.append(x.to(tdt).contiguous())
    return tuple(out)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a (CPU or CUDA) tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float32).to(torch.float64).numpy()
