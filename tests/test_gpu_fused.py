"""fa_backward_fused: preprocess, backward and convert in one launch.

It must give the results of the three separate launches: bitwise in
deterministic mode (same per-key-block slices, same summation order), and
within the usual bf16 tolerance of the float64 oracle by default.  Shapes
cover head counts that do not fill the last group of four heads, more than
three groups (the ticket decoder's uniform middle), N_q != N_k with rows
that see no key, every tensor-core head dim and the full-size workloads."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import compare_head, ratio
from oracle import attention_backward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


def _inputs(B, H, Nq, Nk, d, seed):
    gen = torch.Generator().manual_seed(seed)
    shapes = ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d))
    return [torch.randn(*s, generator=gen).to(torch.bfloat16).to(DEV) for s in shapes]


def _both(q, k, v, g, scale, causal, deterministic):
    o, L = fa.attention_forward(q, k, v, scale, causal)
    sep = fa.attention_backward(q, k, v, o, g, L, scale, causal, deterministic=deterministic)
    fus = fa.attention_backward(q, k, v, o, g, L, scale, causal, deterministic=deterministic, fused=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    return o, L, sep, fus


CASES = [
    # B, H, N_q, N_k, d, causal
    (1, 2, 300, 300, 128, True),
    (1, 5, 257, 257, 64, False),
    (2, 7, 200, 200, 128, True),    # 14 heads: four groups, the last partial
    (1, 13, 129, 129, 96, True),    # 13 heads: the uniform middle of the ticket order
    (1, 3, 100, 300, 128, True),
    (1, 4, 300, 100, 64, True),     # rows without keys
    (1, 6, 640, 384, 32, False),
    (1, 1, 1, 1, 128, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
def test_fused_deterministic_equals_separate_bitwise(B, H, Nq, Nk, d, causal):
    q, k, v, g = _inputs(B, H, Nq, Nk, d, seed=B * 100 + H * 10 + Nq + Nk + d)
    _, _, sep, fus = _both(q, k, v, g, 1.0 / np.sqrt(d), causal, True)
    for a, b in zip(sep, fus):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
def test_fused_matches_the_oracle(B, H, Nq, Nk, d, causal):
    scale = 1.0 / np.sqrt(d)
    q, k, v, g = _inputs(B, H, Nq, Nk, d, seed=7 + Nq + Nk + d)
    _, _, _, (dq, dk, dv) = _both(q, k, v, g, scale, causal, False)
    term = None
    for b in range(B):
        for h in range(H):
            x = [to_f64(t[b, h].cpu()) for t in (q, k, v, g)]
            ref = attention_backward(*x, scale, causal)
            term = scale * np.abs(x[3]).max() * np.abs(x[2]).max() * max(np.abs(x[0]).max(), np.abs(x[1]).max())
            for name, t in (("dQ", dq), ("dK", dk), ("dV", dv)):
                got = to_f64(t[b, h].cpu())
                r = getattr(ref, name)[0, 0]
                assert np.all(np.isfinite(got))
                err = ratio(got, r) if np.abs(r).max() > 0 else float(np.abs(got).max() / term)
                assert err <= 2e-2, (b, h, name, err)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha", "causal", "ragged"])
def test_fused_full_size_workloads(name):
    """The benchmark's workloads: fused == separate bitwise (deterministic),
    and the default fused result matches the oracle on sampled heads."""
    w = workload(name)
    q, k, v, g = (t.to(DEV) for t in make_inputs(w))
    o, L, sep, fus = _both(q, k, v, g, w.scale, w.causal, True)
    for a, b in zip(sep, fus):
        assert torch.equal(a, b)
    del sep, fus
    dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal, fused=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    out = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), g=g.cpu(), o=o.cpu(), L=L.cpu(), dq=dq.cpu(), dk=dk.cpu(),
               dv=dv.cpu())
    for bb, hh in ((0, 0), (w.B - 1, w.H - 1)):
        compare_head(out, w, bb, hh, 2e-2)
