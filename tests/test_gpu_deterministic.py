"""FA_FLAG_DETERMINISTIC: dQ from per-key-block slices summed in a fixed
order ("CUDA 算子工程" ch.16 §16.3, deterministic option) must be bitwise
reproducible and still match the float64 oracle."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, workload
from gpu_common import compare_head

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


def _run(w, inputs, deterministic):
    q, k, v, g = (t.to(DEV) for t in inputs)
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    outs = []
    for _ in range(2):
        dq, dk, dv = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal, deterministic=deterministic)
        torch.cuda.synchronize()
        assert fa.get_device_status() == 0
        outs.append((dq.cpu(), dk.cpu(), dv.cpu()))
    host = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), g=g.cpu(), o=o.cpu(), L=L.cpu())
    return host, outs


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 3, 1000, 128, True), (2, 2, 300, 64, False),
                                            (1, 2, 129, 128, False), (1, 4, 640, 64, True)])
def test_bf16_deterministic_is_bitwise_repeatable_and_correct(B, H, N, d, causal):
    w = workload("causal", B=B, H=H, N=N, d=d, causal=causal, seed=60 + N)
    host, outs = _run(w, make_inputs(w), True)
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    out = dict(host, dq=outs[0][0], dk=outs[0][1], dv=outs[0][2])
    for bb in range(B):
        for hh in range(H):
            compare_head(out, w, bb, hh, 2e-2)


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_deterministic(causal):
    w = workload("tiny", B=2, H=2, N=200, d=32, causal=causal)
    gen = torch.Generator().manual_seed(61)
    inputs = tuple(torch.randn(w.B, w.H, w.N, w.d, generator=gen) for _ in range(4))
    host, outs = _run(w, inputs, True)
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    out = dict(host, dq=outs[0][0], dk=outs[0][1], dv=outs[0][2])
    for bb in range(w.B):
        for hh in range(w.H):
            compare_head(out, w, bb, hh, 1e-5, L_tol=1e-6)


def test_host_pipeline_deterministic_equals_device_path():
    w = workload("causal", B=1, H=5, N=500, d=128, seed=62)
    host, outs = _run(w, make_inputs(w), True)
    pin = lambda t: t.contiguous().pin_memory()
    args = [pin(host[n]) for n in ("q", "k", "v", "o", "g", "L")]
    got = fa.attention_backward_host(*args, w.scale, w.causal, heads_per_group=2, deterministic=True)
    torch.cuda.synchronize()
    for a, b in zip(got, outs[0]):
        assert torch.equal(a, b)
