"""Repetition stress: a race in a kernel's barrier protocol (a missing or
mis-phased wait) tends to show up only now and then.  Each case runs the
forward once and the backward many times on the same inputs: with
FA_FLAG_DETERMINISTIC every run must be bitwise equal to the first; with
the default fire-and-forget reductions every run must agree with the first
to two bf16 units in the last place of the largest element (only the
summation order differs; a race would give errors of the order of the
values), and
the first must match the float64 oracle on a sampled head."""

import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import compare_head, ratio

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RUNS = 24


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


@pytest.mark.parametrize("H,N,d,causal", [(8, 2048, 128, True), (8, 2048, 64, False), (4, 2048, 256, True),
                                          (4, 1000, 256, False)])
@pytest.mark.parametrize("det", [False, True])
def test_repeated_backward_agrees(H, N, d, causal, det):
    w = workload("causal", B=1, H=H, N=N, d=d, causal=causal, seed=900 + d + N)
    q, k, v, g = (t.to(DEV) for t in make_inputs(w))
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    first = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal, deterministic=det)
    for _ in range(RUNS - 1):
        again = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal, deterministic=det)
        for a, b in zip(first, again):
            if det:
                assert torch.equal(a, b)
            else:
                # fp32 partial sums added in another order can round a bf16
                # output to the neighbouring value: one unit in the last
                # place is 2^-8 of the element; allow two at the maximum
                assert ratio(to_f64(b), to_f64(a)) <= 8e-3
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    out = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), g=g.cpu(), o=o.cpu(), L=L.cpu(),
               dq=first[0].cpu(), dk=first[1].cpu(), dv=first[2].cpu())
    compare_head(out, w, 0, H - 1, 2e-2)
