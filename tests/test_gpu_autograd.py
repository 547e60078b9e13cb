"""flash_attn_func under autograd: the gradients it returns are the ones the
C ABI's fa_backward gives for dO = the incoming gradient (bitwise: the same
kernels run), and they match the float64 oracle.  Covers causal and not,
N_q != N_k, head dims 64 and 256, and [B, N, H, d] views."""

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


def _leaf(t):
    return t.detach().clone().requires_grad_(True)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,bnhd", [
    (2, 3, 300, 300, 64, True, False),
    (1, 2, 200, 330, 128, True, False),
    (1, 2, 257, 257, 256, False, False),
    (2, 2, 190, 190, 64, True, True),
])
def test_autograd_gradients(B, H, Nq, Nk, d, causal, bnhd):
    gen = torch.Generator().manual_seed(B * 1000 + Nq + d)
    shape_q, shape_k = ((B, Nq, H, d), (B, Nk, H, d)) if bnhd else ((B, H, Nq, d), (B, H, Nk, d))
    q, g = (torch.randn(shape_q, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    k, v = (torch.randn(shape_k, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    if bnhd:  # [B, N, H, d] storage seen as [B, H, N, d] views
        q, k, v, g = (t.permute(0, 2, 1, 3) for t in (q, k, v, g))
    ql, kl, vl = _leaf(q), _leaf(k), _leaf(v)
    o = fa.flash_attn_func(ql, kl, vl, causal=causal)
    (o.float() * g.float()).sum().backward()
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    scale = d ** -0.5
    o2, L = fa.attention_forward(q, k, v, scale, causal)
    ref = fa.attention_backward(q, k, v, o2, g, L, scale, causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    for got, want in zip((ql.grad, kl.grad, vl.grad), ref):
        assert got.shape == want.shape
        assert ratio(to_f64(got), to_f64(want)) <= 1e-2  # same kernels; reduction order may differ
    for b in range(B):
        for h in range(H):
            r = attention_backward(*(to_f64(t[b, h]) for t in (q, k, v, g)), scale, causal)
            for name, got in (("dQ", ql.grad), ("dK", kl.grad), ("dV", vl.grad)):
                x, rr = to_f64(got[b, h]), getattr(r, name)[0, 0]
                assert np.all(np.isfinite(x))
                assert ratio(x, rr) <= 2e-2, (name, b, h, ratio(x, rr))


def test_autograd_deterministic_is_bitwise_repeatable():
    gen = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(1, 2, 500, 128, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(3))
    grads = []
    for _ in range(2):
        ql, kl, vl = _leaf(q), _leaf(k), _leaf(v)
        fa.flash_attn_func(ql, kl, vl, causal=True, deterministic=True).float().square().sum().backward()
        grads.append((ql.grad, kl.grad, vl.grad))
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    for a, b in zip(*grads):
        assert torch.equal(a, b)


def test_check_status_raises_on_a_recorded_device_error():
    """A device-side error only reaches the status word; with check_status the
    Python layer reads it after the step and raises.  The error is planted by
    the library's bounded-wait self test (a barrier nothing arrives at), so no
    kernel of the backward itself has to fail."""
    gen = torch.Generator().manual_seed(9)
    q, k, v = (torch.randn(1, 2, 256, 64, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(3))
    ql, kl, vl = _leaf(q), _leaf(k), _leaf(v)
    o = fa.flash_attn_func(ql, kl, vl, causal=True, check_status=True)  # clean: no raise
    fa.selftest_wait_timeout(5_000_000)  # records FA_ERR_TIMEOUT after 5 ms
    with pytest.raises(fa.FaError) as err:
        o.float().sum().backward()
    assert err.value.code == fa.FA_ERR_TIMEOUT
    assert fa.get_device_status() == 0  # the read cleared the word
    o2, L = fa.attention_forward(q, k, v, 0.125, True)
    fa.selftest_wait_timeout(5_000_000)
    with pytest.raises(fa.FaError):
        fa.attention_backward(q, k, v, o2, o2, L, 0.125, True, check_status=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o2, o2, L, 0.125, True, check_status=True)
    assert torch.isfinite(dq.float()).all()
