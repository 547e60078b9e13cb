"""Head dims beyond 64 and 128: GPU parity against the float64 oracle.

bf16 d = 32 and 96 run on the tensor-core kernels (tiles 64 and 128 columns
wide, the columns past d zero-filled by the TMA); bf16 d = 256 runs on the
tensor cores too (the forward with 64-row key blocks, the backward with two
CTAs per key block, one per half of the columns); fp32 d = 96, 256 run on the
CUDA-core kernels (fp32 arithmetic; 32-row key blocks at d = 256).  The
oracle is the same plain definition at every d.  Tolerances as everywhere:
max|dX - ref| / max|ref| <= 2e-2 for bf16 (L <= 1e-3), 1e-5 for fp32
(L <= 1e-6)."""

import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, workload
from gpu_common import compare_head, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


BF16 = [
    # B, H, N, d, causal
    (1, 2, 128, 32, False),
    (1, 2, 300, 32, True),
    (1, 1, 1, 32, True),
    (2, 1, 640, 32, False),
    (1, 2, 128, 96, True),
    (2, 2, 129, 96, False),
    (1, 1, 1, 96, False),
    (1, 2, 1000, 96, True),
    (1, 2, 100, 256, True),
    (1, 1, 257, 256, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", BF16)
def test_bf16_head_dims(B, H, N, d, causal):
    w = workload("causal", B=B, H=H, N=N, d=d, causal=causal, seed=200 + N + d)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    for b in range(B):
        for h in range(H):
            compare_head(out, w, b, h, 2e-2)


@pytest.mark.parametrize("d", [32, 96])
def test_bf16_head_dims_large_logits(d):
    """Peaky softmax (queries with std 4) through the lazy-rescale forward."""
    w = workload("long", N=700, H=2, d=d, seed=23)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    for h in range(2):
        compare_head(out, w, 0, h, 2e-2)


@pytest.mark.parametrize("N,d,causal", [(129, 96, True), (300, 96, False), (100, 256, True), (33, 256, False)])
def test_fp32_head_dims(N, d, causal):
    w = workload("tiny", N=N, d=d, causal=causal, B=2, H=2, seed=4).with_(name="fp32_case")
    gen = torch.Generator().manual_seed(N + d)
    inputs = tuple(torch.randn(w.B, w.H, N, d, generator=gen) for _ in range(4))
    out = run_gpu(w, DEV, inputs)
    assert out["status"] == 0
    for b in range(w.B):
        for h in range(w.H):
            compare_head(out, w, b, h, tol=1e-5, L_tol=1e-6)


@pytest.mark.parametrize("dtype,N,d,causal", [(torch.bfloat16, 300, 96, True), (torch.bfloat16, 200, 32, False),
                                              (torch.bfloat16, 100, 256, True), (torch.float32, 70, 256, False)])
def test_deterministic_head_dims(dtype, N, d, causal):
    if dtype == torch.bfloat16:
        w = workload("causal", B=1, H=2, N=N, d=d, causal=causal, seed=70 + d)
        inputs = make_inputs(w)
        tol, L_tol = 2e-2, 1e-3
    else:
        w = workload("tiny", B=1, H=2, N=N, d=d, causal=causal, seed=71).with_(name="fp32_case")
        gen = torch.Generator().manual_seed(72)
        inputs = tuple(torch.randn(w.B, w.H, N, d, generator=gen) for _ in range(4))
        tol, L_tol = 1e-5, 1e-6
    q, k, v, g = (t.to(DEV) for t in inputs)
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    runs = []
    for _ in range(2):
        runs.append(fa.attention_backward(q, k, v, o, g, L, w.scale, w.causal, deterministic=True))
        torch.cuda.synchronize()
        assert fa.get_device_status() == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    out = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), g=g.cpu(), o=o.cpu(), L=L.cpu(),
               dq=runs[0][0].cpu(), dk=runs[0][1].cpu(), dv=runs[0][2].cpu())
    for h in range(2):
        compare_head(out, w, 0, h, tol, L_tol=L_tol)
