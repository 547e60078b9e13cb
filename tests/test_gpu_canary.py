"""Out-of-bounds writes, checked without a sanitizer: every output of the
C ABI is placed in a larger buffer filled with a canary bit pattern: guard
bands before and after, and padding columns between rows (row stride d + pad).
After fa_fwd and fa_backward every canary byte must be unchanged, and the
gradients must still match the float64 oracle.  Covers the tensor-core
kernels (bf16, d = 64, 128, 256; causal and not; ragged N; N_q != N_k) and
the CUDA-core kernels (fp32), deterministic mode included."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import to_f64
from gpu_common import ratio
from oracle import attention_backward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096  # bytes of canary before and after every buffer
CANARY = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


class Guarded:
    """A [B, H, rows, d] view (row stride d + pad) inside a canary-filled
    byte buffer, or a flat view of `numel` elements."""

    def __init__(self, dtype, shape=None, pad=0, numel=None):
        es = torch.empty((), dtype=dtype).element_size()
        if shape is not None:
            B, H, rows, d = shape
            self.strides = (H * rows * (d + pad), rows * (d + pad), d + pad, 1)
            n = B * H * rows * (d + pad)
        else:
            n = numel
        self.raw = torch.full((GUARD + n * es + GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        flat = self.raw[GUARD:GUARD + n * es].view(dtype)
        self.t = flat.as_strided(shape, self.strides) if shape is not None else flat
        # the bytes a correct kernel may write
        self.mask = torch.zeros_like(self.raw, dtype=torch.bool)
        written = torch.zeros(n, dtype=torch.bool, device=DEV)
        if shape is not None:
            written.as_strided(shape, self.strides).fill_(True)
        else:
            written.fill_(True)
        self.mask[GUARD:GUARD + n * es] = written.repeat_interleave(es)

    def check(self, name):
        bad = (self.raw != CANARY) & ~self.mask
        assert not bool(bad.any()), f"{name}: {int(bad.sum())} canary bytes overwritten"


CASES = [
    # dtype, B, H, Nq, Nk, d, causal, deterministic
    (torch.bfloat16, 1, 2, 200, 200, 64, True, False),
    (torch.bfloat16, 2, 1, 129, 129, 128, False, False),
    (torch.bfloat16, 1, 2, 300, 170, 128, True, False),
    (torch.bfloat16, 1, 2, 190, 190, 256, True, False),
    (torch.bfloat16, 1, 1, 77, 300, 256, False, True),
    (torch.bfloat16, 1, 2, 257, 257, 128, True, True),
    (torch.float32, 1, 2, 70, 70, 32, True, False),
    (torch.float32, 1, 1, 40, 90, 256, False, True),
]


@pytest.mark.parametrize("dtype,B,H,Nq,Nk,d,causal,det", CASES)
def test_outputs_stay_inside_their_buffers(dtype, B, H, Nq, Nk, d, causal, det):
    pad = 16 // torch.empty((), dtype=dtype).element_size()  # keeps rows 16-byte aligned
    gen = torch.Generator().manual_seed(Nq * 31 + Nk + d)
    qs, ks = (B, H, Nq, d), (B, H, Nk, d)
    q, g, o, dq = (Guarded(dtype, qs, pad) for _ in range(4))
    k, v, dk, dv = (Guarded(dtype, ks, pad) for _ in range(4))
    for buf, shape in ((q, qs), (g, qs), (k, ks), (v, ks)):  # inputs: their padding must stay untouched too
        buf.t.copy_(torch.randn(shape, generator=gen).to(dtype))
    scale = d ** -0.5
    p = fa.problem_for(q.t, scale, causal, det, k=k.t)
    L = Guarded(torch.float32, numel=B * H * Nq)
    D = Guarded(torch.float32, numel=B * H * Nq)
    acc = Guarded(torch.float32, numel=fa.fa_dq_accum_elems(p))
    fa.fa_fwd(p, q.t, k.t, v.t, o.t, L.t)
    fa.fa_backward(p, q.t, k.t, v.t, o.t, g.t, L.t, D.t, acc.t, dq.t, dk.t, dv.t)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    for name, buf in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv), ("L", L), ("D", D), ("dQ_accum", acc),
                      ("Q", q), ("K", k), ("V", v), ("dO", g)):
        buf.check(name)
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-5
    for b in range(B):
        for h in range(H):
            ref = attention_backward(*(to_f64(t.t[b, h]) for t in (q, k, v, g)), scale, causal)
            for name, x in (("dQ", dq), ("dK", dk), ("dV", dv)):
                xr, rr = to_f64(x.t[b, h]), getattr(ref, name)[0, 0]
                assert np.all(np.isfinite(xr)), name
                if np.abs(rr).max() > 0:
                    assert ratio(xr, rr) <= tol, (name, b, h, ratio(xr, rr))
