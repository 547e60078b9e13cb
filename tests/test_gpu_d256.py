"""bf16 head dim 256 on the tensor cores: GPU parity against the float64 oracle.

The d = 256 backward runs two CTAs per 128-row key block, each accumulating
dK and dV for one half of the columns and recomputing the full S^T and dP^T;
query blocks are 64 rows and dQ is produced per 128-row tile.  The cases
cover one and several key blocks, ragged tails on both sides of a 64-row
block, N = 1, the causal diagonal, N_q != N_k (bottom-right causal), the
[B, N, H, d] layout through strides, a peaky softmax, deterministic mode and
one large case.  Tolerances as everywhere: max|dX - ref| / max|ref| <= 2e-2,
L <= 1e-3."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import compare_head, ratio, run_gpu
from oracle import attention_backward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 2, 64, True),     # one 64-row block: the tile's second block is past N
    (1, 2, 128, False),
    (1, 1, 1, True),
    (1, 1, 1, False),
    (2, 1, 190, True),    # tail inside the second block of a tile
    (1, 3, 300, False),
    (1, 2, 513, True),    # five key blocks, one-row tail
    (2, 2, 1000, True),
])
def test_d256_parity(B, H, N, causal):
    w = workload("causal", B=B, H=H, N=N, d=256, causal=causal, seed=500 + N)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    for b in range(B):
        for h in range(H):
            compare_head(out, w, b, h, TOL)


def test_d256_large_logits():
    """Queries with std 4: a peaky softmax."""
    w = workload("long", N=700, H=2, d=256, seed=29)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    for h in range(2):
        compare_head(out, w, 0, h, TOL)


@pytest.mark.parametrize("Nq,Nk,causal", [(300, 700, True), (700, 300, True), (129, 1000, True),
                                          (200, 77, False), (1, 300, True)])
def test_d256_cross_lengths(Nq, Nk, causal):
    d, scale = 256, 1.0 / 16.0
    gen = torch.Generator().manual_seed(Nq * 3 + Nk)
    q = torch.randn(1, 2, Nq, d, generator=gen).to(torch.bfloat16).to(DEV)
    k = torch.randn(1, 2, Nk, d, generator=gen).to(torch.bfloat16).to(DEV)
    v = torch.randn(1, 2, Nk, d, generator=gen).to(torch.bfloat16).to(DEV)
    g = torch.randn(1, 2, Nq, d, generator=gen).to(torch.bfloat16).to(DEV)
    o, L = fa.attention_forward(q, k, v, scale, causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, scale, causal)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    for h in range(2):
        ref = attention_backward(*(to_f64(t[0, h]) for t in (q, k, v, g)), scale, causal)
        for name, x in (("dQ", dq), ("dK", dk), ("dV", dv)):
            xr = to_f64(x[0, h])
            r = getattr(ref, name)[0, 0]
            assert np.all(np.isfinite(xr)), name
            if np.abs(r).max() > 0:
                assert ratio(xr, r) <= TOL, (name, h, ratio(xr, r))
            else:  # rows that see no key: exact zeros
                assert np.abs(xr).max() == 0.0, (name, h)


def test_d256_strided_layout():
    """[B, N, H, d] storage passed through strides."""
    B, H, N, d = 2, 3, 200, 256
    w = workload("causal", B=B, H=H, N=N, d=d, causal=True, seed=33)
    gen = torch.Generator().manual_seed(33)
    base = [torch.randn(B, N, H, d, generator=gen).to(torch.bfloat16) for _ in range(4)]
    q, k, v, g = (t.permute(0, 2, 1, 3).to(DEV) for t in base)
    assert q.stride(2) == H * d
    o, L = fa.attention_forward(q, k, v, w.scale, True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, w.scale, True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    out = {n: t.cpu() for n, t in dict(q=q, k=k, v=v, g=g, o=o, L=L, dq=dq, dk=dk, dv=dv).items()}
    for b in range(B):
        for h in range(H):
            compare_head(out, w, b, h, TOL)


def test_d256_deterministic():
    w = workload("causal", B=1, H=2, N=1000, d=256, causal=True, seed=77)
    q, k, v, g = (t.to(DEV) for t in make_inputs(w))
    o, L = fa.attention_forward(q, k, v, w.scale, True)
    runs = []
    for _ in range(2):
        runs.append(fa.attention_backward(q, k, v, o, g, L, w.scale, True, deterministic=True))
        torch.cuda.synchronize()
        assert fa.get_device_status() == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    # the same sums as the atomic mode, up to summation order
    at = fa.attention_backward(q, k, v, o, g, L, w.scale, True)
    torch.cuda.synchronize()
    for a, b in zip(runs[0], at):
        assert ratio(to_f64(a), to_f64(b)) <= 1e-2
    out = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), g=g.cpu(), o=o.cpu(), L=L.cpu(),
               dq=runs[0][0].cpu(), dk=runs[0][1].cpu(), dv=runs[0][2].cpu())
    for h in range(2):
        compare_head(out, w, 0, h, TOL)


def test_d256_large_sampled_head():
    """B=1, H=8, N=4096, causal: one head against the oracle, every head finite."""
    w = workload("causal", B=1, H=8, N=4096, d=256, causal=True, seed=81)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    for key in ("dq", "dk", "dv"):
        assert torch.isfinite(out[key].float()).all()
    compare_head(out, w, 0, 5, TOL)
