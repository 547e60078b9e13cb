"""fa_backward_host: backward from host-resident tensors, streamed through a
device workspace in groups of heads with overlapped copies.  Its results must
match the oracle (small case) and the device-resident path (groups that do
not divide the head count, one group, one head per group)."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import compare_head, ratio

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()


def _forward(w):
    q, k, v, g = make_inputs(w)
    o, L = fa.attention_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.scale, w.causal)
    pin = lambda t: t.contiguous().pin_memory()
    return [pin(t) for t in (q, k, v, o.cpu(), g, L.cpu())]


@pytest.mark.parametrize("d,heads_per_group", [(128, 0), (128, 1), (128, 3), (128, 64), (256, 2)])
def test_host_pipeline_matches_device_path(d, heads_per_group):
    w = workload("causal", B=2, H=5, N=700, d=d, seed=51)
    q, k, v, o, g, L = _forward(w)
    dq, dk, dv = fa.attention_backward_host(q, k, v, o, g, L, w.scale, w.causal, heads_per_group)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    ref = fa.attention_backward(q.to(DEV), k.to(DEV), v.to(DEV), o.to(DEV), g.to(DEV), L.to(DEV), w.scale, w.causal)
    torch.cuda.synchronize()
    for x, y in zip((dq, dk, dv), ref):
        assert not x.is_cuda
        assert ratio(to_f64(x), to_f64(y)) <= 1e-2


def test_host_pipeline_against_oracle_fp32():
    w = workload("tiny", B=2, H=3, N=130, d=32, causal=True)
    gen = torch.Generator().manual_seed(52)
    inputs = [torch.randn(w.B, w.H, w.N, w.d, generator=gen) for _ in range(4)]
    q, k, v, g = inputs
    o, L = fa.attention_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.scale, w.causal)
    pin = lambda t: t.contiguous().pin_memory()
    args = [pin(t) for t in (q, k, v, o.cpu(), g, L.cpu())]
    dq, dk, dv = fa.attention_backward_host(*args, w.scale, w.causal, heads_per_group=2)
    torch.cuda.synchronize()
    out = dict(q=q, k=k, v=v, g=g, o=o.cpu(), L=L.cpu(), dq=dq, dk=dk, dv=dv)
    for b in range(w.B):
        for h in range(w.H):
            compare_head(out, w, b, h, tol=1e-5, L_tol=1e-6)


def test_host_pipeline_rejects_strided_host_tensors():
    w = workload("causal", B=1, H=2, N=64, d=64, seed=53)
    q = torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16).permute(0, 2, 1, 3)
    p = fa.problem_for(q, w.scale, True)
    lib = fa.load_library()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    import ctypes
    r = lib.fa_backward_host(ctypes.byref(p), *([q.data_ptr()] * 6), *([q.data_ptr()] * 3), ws.data_ptr(),
                             ws.numel(), 0, None)
    assert r == fa.FA_ERR_INVALID_ARG


def test_host_pipeline_concurrent_threads():
    """Two host threads call fa_backward_host on one device at once, each on
    its own stream with its own inputs.  The library's streams and events are
    shared per device, so the calls must enqueue one after the other; each
    result must equal (bitwise, deterministic mode) the same call made alone."""
    import threading

    cases = []
    for seed in (61, 62):
        w = workload("causal", B=2, H=5, N=700, d=128, seed=seed)
        q, k, v, o, g, L = _forward(w)
        p = fa.problem_for(q, w.scale, True, True)
        ws = torch.empty(fa.fa_backward_host_workspace_bytes(p, 2), dtype=torch.uint8, device=DEV)
        out = tuple(torch.empty_like(t).pin_memory() for t in (q, k, v))
        cases.append(dict(w=w, args=(q, k, v, o, g, L), ws=ws, out=out, stream=torch.cuda.Stream()))
    alone = []
    for c in cases:
        res = fa.attention_backward_host(*c["args"], c["w"].scale, True, 2, workspace=c["ws"], out=c["out"],
                                         stream=c["stream"], deterministic=True)
        c["stream"].synchronize()
        alone.append(tuple(t.clone() for t in res))
    assert fa.get_device_status() == 0
    errors = []

    def worker(i):
        c = cases[i]
        try:
            torch.cuda.set_device(0)
            for _ in range(6):
                for t in c["out"]:
                    t.fill_(float("nan"))
                res = fa.attention_backward_host(*c["args"], c["w"].scale, True, 2, workspace=c["ws"], out=c["out"],
                                                 stream=c["stream"], deterministic=True)
                c["stream"].synchronize()
                for x, y in zip(res, alone[i]):
                    if not torch.equal(x, y):
                        errors.append(f"thread {i}: result differs from the call made alone")
                        return
        except Exception as e:  # reported below, in the test's own thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert fa.get_device_status() == 0
