"""Helpers shared by the GPU parity tests (imported only by tests)."""

from __future__ import annotations

import numpy as np
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64
from oracle import attention_backward


def ratio(x: np.ndarray, ref: np.ndarray) -> float:
    """max|x - ref| / max|ref| over the whole tensor (the parity metric)."""
    return float(np.abs(x - ref).max() / max(float(np.abs(ref).max()), 1e-30))


def run_gpu(w, dev="cuda:0", inputs=None):
    """Forward then backward through the C ABI; returns CPU tensors."""
    q, k, v, g = inputs if inputs is not None else make_inputs(w)
    q, k, v, g = (t.to(dev) for t in (q, k, v, g))
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal)
    torch.cuda.synchronize()
    status = fa.get_device_status()
    out = {n: t.cpu() for n, t in dict(q=q, k=k, v=v, g=g, o=o, L=L, dq=dq, dk=dk, dv=dv).items()}
    out["status"] = status
    return out


def oracle_head(out, w, b, h):
    """float64 oracle for one (b, h) from the same (rounded) inputs."""
    q, k, v, g = (to_f64(out[n][b, h]) for n in ("q", "k", "v", "g"))
    return attention_backward(q, k, v, g, w.scale, w.causal)


def compare_head(out, w, b, h, tol, L_tol=1e-3):
    ref = oracle_head(out, w, b, h)
    # Where the exact gradient is identically zero (N = 1: a single key makes
    # dS = 0, so dQ = dK = 0) the ratio is undefined; the bound is then
    # absolute, tol times the size of one term scale * dS_ij * K_j.
    q, k, v, g = (np.abs(to_f64(out[n][b, h])).max() for n in ("q", "k", "v", "g"))
    term = w.scale * g * v * max(q, k)
    errs = {}
    for name, key in (("dQ", "dq"), ("dK", "dk"), ("dV", "dv"), ("O", "o")):
        x = to_f64(out[key][b, h])
        assert np.all(np.isfinite(x)), f"non-finite {name}"
        r = getattr(ref, name)[0, 0]
        errs[name] = ratio(x, r) if np.abs(r).max() > 0 else float(np.abs(x).max() / term)
    Lx = to_f64(out["L"][b, h])
    errs["L"] = ratio(Lx, ref.L[0, 0])
    bad = {n: e for n, e in errs.items() if e > (L_tol if n == "L" else tol)}
    assert not bad, f"(b={b}, h={h}) errors {errs}"
    return errs
