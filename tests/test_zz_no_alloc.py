"""fa_backward_static_workspace: the backward entry point for callers that
cannot allocate device memory (a host framework or plugin that owns all device
memory, a process with a fixed device-memory budget, a loop that cannot pay for
cudaMalloc's synchronisation).  It keeps D and the dQ accumulator in fixed
arrays inside the library instead of taking them from the caller.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test.  The checks: two calls in a row
through the C ABI give the same dQ, dK, dV as fa_backward with caller-owned
scratch, within the tolerance of the other parity tests; in deterministic mode
(where the preprocess zeroes nothing and every accumulator element that the
convert reads is overwritten by the main kernel) the results are bitwise equal
to fa_backward's with NaN-filled caller scratch, also when the fixed arrays
still hold a larger, differently shaped problem's leftovers."""

import ctypes

import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import ratio

pytestmark = pytest.mark.gpu


def _entry():
    lib = fa.load_library()
    f = lib.fa_backward_static_workspace
    f.argtypes = [ctypes.POINTER(fa.FaProblem)] + [ctypes.c_void_p] * 10
    f.restype = ctypes.c_int
    return f


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name,overrides,tol", [("causal", dict(B=2, H=3, N=1000, seed=41), 2e-2),
                                                ("mha", dict(H=4, N=700, seed=42), 2e-2),
                                                ("tiny", {}, 1e-5)])
def test_static_workspace_matches_fa_backward(name, overrides, tol):
    f = _entry()
    w = workload(name, **overrides)
    q, k, v, g = (t.cuda() for t in make_inputs(w))
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    ref = fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal)  # caller-owned scratch
    torch.cuda.synchronize()
    p = fa.problem_for(q, w.scale, w.causal)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the second call must not see the first call's leftovers
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        r = f(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), g.data_ptr(),
              L.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), stream)
        assert r == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.get_device_status() == 0
        for x, y in zip((dq, dk, dv), ref):
            assert torch.isfinite(x.float()).all()
            assert ratio(to_f64(x), to_f64(y)) <= tol


def _static_call(f, p, q, k, v, o, g, L):
    dq = torch.full_like(q, float("nan"))
    dk, dv = torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
    r = f(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), g.data_ptr(), L.data_ptr(),
          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert r == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    return dq, dk, dv


def _cross_inputs(B, H, N, Nk, d, seed):
    gen = torch.Generator().manual_seed(seed)
    q, g = (torch.randn(B, H, N, d, generator=gen).to(torch.bfloat16).cuda() for _ in range(2))
    k, v = (torch.randn(B, H, Nk, d, generator=gen).to(torch.bfloat16).cuda() for _ in range(2))
    return q, k, v, g


def test_static_workspace_deterministic_bitwise_after_other_problem():
    f = _entry()
    # a larger causal problem first: its slices stay in the fixed arrays
    q, k, v, g = _cross_inputs(1, 4, 2048, 2048, 128, 51)
    o, L = fa.attention_forward(q, k, v, 128 ** -0.5, True)
    _static_call(f, fa.problem_for(q, 128 ** -0.5, True, True), q, k, v, o, g, L)
    # then a smaller ragged one with N_k != N, twice
    for d in (128, 64):
        q, k, v, g = _cross_inputs(2, 3, 1000, 777, d, 52 + d)
        scale = d ** -0.5
        o, L = fa.attention_forward(q, k, v, scale, True)
        p = fa.problem_for(q, scale, True, True, k=k)
        D = torch.full((2, 3, 1000), float("nan"), device="cuda")
        acc = torch.full((fa.fa_dq_accum_elems(p),), float("nan"), device="cuda")
        ref = fa.attention_backward(q, k, v, o, g, L, scale, True, workspace=(D, acc), deterministic=True)
        torch.cuda.synchronize()
        assert fa.get_device_status() == 0
        for _ in range(2):
            got = _static_call(f, p, q, k, v, o, g, L)
            for x, y in zip(got, ref):
                assert torch.isfinite(x.float()).all()
                assert torch.equal(x, y)


def test_static_workspace_rejects_problems_beyond_its_arrays():
    f = _entry()
    fake = 0x1000  # never dereferenced: the size check comes first
    q = torch.empty(1, 32, 8192, 128, dtype=torch.bfloat16, device="meta")  # 128 MiB of accumulator
    p = fa.FaProblem(1, 32, 8192, 128, 0.088, 1, fa.FA_BF16, 0, q.stride(0), q.stride(1), q.stride(2))
    r = f(ctypes.byref(p), *([fake] * 9), torch.cuda.current_stream().cuda_stream)
    assert r == fa.FA_ERR_UNSUPPORTED
