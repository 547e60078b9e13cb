"""N_q != N_k (bottom-right causal alignment): GPU parity against the float64
oracle, through the C ABI.

Covers more keys than queries and more queries than keys (rows that see no
key: O = 0, L = +inf, zero gradients), one query or one key, ragged tails,
the tensor-core kernels (bf16, d = 256 included), the CUDA-core kernels
(fp32), deterministic mode and the host-tensor pipeline.
Tolerances: max|dX - ref| / max|ref| <= 2e-2 for bf16 (L <= 1e-3), 1e-5 for
fp32 (L <= 1e-6); L = +inf exactly where the oracle has it."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import to_f64
from gpu_common import ratio
from oracle import attention_backward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


def _inputs(B, H, Nq, Nk, d, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Nq, d, generator=gen).to(dtype)
    k = torch.randn(B, H, Nk, d, generator=gen).to(dtype)
    v = torch.randn(B, H, Nk, d, generator=gen).to(dtype)
    g = torch.randn(B, H, Nq, d, generator=gen).to(dtype)
    return q, k, v, g


def _check(host, scale, causal, b, h, tol, L_tol):
    q, k, v, g = (to_f64(host[n][b, h]) for n in ("q", "k", "v", "g"))
    ref = attention_backward(q, k, v, g, scale, causal)
    term = scale * np.abs(g).max() * np.abs(v).max() * max(np.abs(q).max(), np.abs(k).max())
    for name, key in (("O", "o"), ("dQ", "dq"), ("dK", "dk"), ("dV", "dv")):
        x = to_f64(host[key][b, h])
        r = getattr(ref, name)[0, 0]
        assert np.all(np.isfinite(x)), f"non-finite {name}"
        err = ratio(x, r) if np.abs(r).max() > 0 else float(np.abs(x).max() / term)
        assert err <= tol, f"(b={b}, h={h}) {name} error {err}"
    Lx, Lr = to_f64(host["L"][b, h]), ref.L[0, 0]
    assert np.array_equal(np.isposinf(Lx), np.isposinf(Lr)), "rows without keys must have L = +inf"
    fin = np.isfinite(Lr)
    if fin.any():
        assert ratio(Lx[fin], Lr[fin]) <= L_tol


def _run(q, k, v, g, scale, causal, deterministic=False):
    q, k, v, g = (t.to(DEV) for t in (q, k, v, g))
    o, L = fa.attention_forward(q, k, v, scale, causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, scale, causal, deterministic=deterministic)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    return {n: t.cpu() for n, t in dict(q=q, k=k, v=v, g=g, o=o, L=L, dq=dq, dk=dk, dv=dv).items()}


BF16 = [
    # B, H, N_q, N_k, d, causal
    (1, 2, 100, 300, 64, True),
    (1, 2, 300, 100, 64, True),
    (2, 1, 257, 129, 128, True),
    (1, 2, 129, 1000, 128, True),
    (1, 2, 200, 77, 96, False),
    (1, 1, 1, 500, 128, True),
    (1, 1, 500, 1, 64, True),
    (1, 2, 640, 384, 32, True),
    (1, 2, 384, 640, 128, False),
    (1, 1, 100, 60, 256, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", BF16)
def test_bf16_cross_lengths(B, H, Nq, Nk, d, causal):
    scale = 1.0 / np.sqrt(d)
    host = _run(*_inputs(B, H, Nq, Nk, d, torch.bfloat16, seed=Nq * 7 + Nk + d), scale, causal)
    for b in range(B):
        for h in range(H):
            _check(host, scale, causal, b, h, 2e-2, 1e-3)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [(2, 1, 70, 130, 64, True), (1, 2, 130, 70, 96, True),
                                                (1, 1, 50, 90, 256, False), (1, 2, 33, 200, 16, True)])
def test_fp32_cross_lengths(B, H, Nq, Nk, d, causal):
    scale = 1.0 / np.sqrt(d)
    host = _run(*_inputs(B, H, Nq, Nk, d, torch.float32, seed=Nq + Nk * 3), scale, causal)
    for b in range(B):
        for h in range(H):
            _check(host, scale, causal, b, h, 1e-5, 1e-6)


@pytest.mark.parametrize("dtype,Nq,Nk,d", [(torch.bfloat16, 300, 100, 128), (torch.bfloat16, 100, 300, 64),
                                           (torch.float32, 90, 150, 32), (torch.bfloat16, 70, 40, 256)])
def test_deterministic_cross_lengths(dtype, Nq, Nk, d):
    scale = 1.0 / np.sqrt(d)
    inputs = _inputs(1, 2, Nq, Nk, d, dtype, seed=9 + Nq)
    a = _run(*inputs, scale, True, deterministic=True)
    b = _run(*inputs, scale, True, deterministic=True)
    for n in ("dq", "dk", "dv"):
        assert torch.equal(a[n], b[n])
    tol, L_tol = (2e-2, 1e-3) if dtype == torch.bfloat16 else (1e-5, 1e-6)
    for h in range(2):
        _check(a, scale, True, 0, h, tol, L_tol)


def test_host_pipeline_cross_lengths():
    B, H, Nq, Nk, d = 2, 3, 200, 450, 64
    scale = 0.125
    q, k, v, g = _inputs(B, H, Nq, Nk, d, torch.bfloat16, seed=44)
    dev = _run(q, k, v, g, scale, True, deterministic=True)
    pin = [t.pin_memory() for t in (q, k, v, g, dev["o"], dev["L"])]
    dq, dk, dv = fa.attention_backward_host(pin[0], pin[1], pin[2], pin[4], pin[3], pin[5], scale, True,
                                            heads_per_group=2, deterministic=True)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    assert torch.equal(dq, dev["dq"]) and torch.equal(dk, dev["dk"]) and torch.equal(dv, dev["dv"])
