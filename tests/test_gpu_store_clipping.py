"""The tensor-core kernels write O, dK and dV with TMA tensor stores of
128-row, 64-column boxes, which the tensor maps clip to the tensors' own rows
(N, N_k) and columns (d).  These tests check that nothing lands outside an
output tensor: with heads interleaved in memory ([B, N, H, d] storage, where
the columns past d of a row are the next head's) and with outputs that are
views into larger buffers whose remainder holds a sentinel.
"""
import pytest
import torch

import flashattention_backward_gb300 as fa

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SENTINEL = -12345.0  # exactly representable in bf16


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


def _run(q, k, v, g, scale, causal, outs):
    """Forward then deterministic backward; outs = (o, dq, dk, dv) views to fill."""
    o, dq, dk, dv = outs
    B, H, N, _ = q.shape
    L = torch.empty(B, H, N, device=DEV)
    p = fa.problem_for(q, scale, causal, True, k=k)
    fa.fa_fwd(p, q, k, v, o, L)
    D = torch.empty(B, H, N, device=DEV)
    acc = torch.empty(fa.fa_dq_accum_elems(p), device=DEV)
    fa.fa_backward(p, q, k, v, o, g, L, D, acc, dq, dk, dv)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    return L


@pytest.mark.parametrize("d", [32, 64, 96, 128])
def test_interleaved_heads_match_contiguous(d):
    """[B, N, H, d] storage: every output equals the contiguous run bitwise."""
    B, H, N, Nk = 2, 3, 333, 205
    gen = torch.Generator().manual_seed(7 + d)
    qs, gs = (torch.randn(B, N, H, d, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    ks, vs = (torch.randn(B, Nk, H, d, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    q, g = qs.permute(0, 2, 1, 3), gs.permute(0, 2, 1, 3)
    k, v = ks.permute(0, 2, 1, 3), vs.permute(0, 2, 1, 3)
    assert q.stride(2) == H * d
    scale = d ** -0.5
    # interleaved outputs, pre-filled with the sentinel
    o_s = torch.full((B, N, H, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    dq_s = torch.full((B, N, H, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    dk_s = torch.full((B, Nk, H, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    dv_s = torch.full((B, Nk, H, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    outs = tuple(t.permute(0, 2, 1, 3) for t in (o_s, dq_s, dk_s, dv_s))
    L1 = _run(q, k, v, g, scale, True, outs)
    cq, ck, cv, cg = (t.contiguous() for t in (q, k, v, g))
    ref = tuple(torch.empty_like(t) for t in (cq, cq, ck, cv))
    L2 = _run(cq, ck, cv, cg, scale, True, ref)
    assert torch.equal(L1, L2)
    for got, want in zip(outs, ref):
        assert not (got == SENTINEL).any()  # every element written
        assert torch.equal(got, want)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
def test_outputs_stay_inside_their_tensors(d):
    """Outputs as views at the start of larger buffers: the rest keeps the sentinel."""
    B, H, N, Nk = 1, 2, 333, 205
    gen = torch.Generator().manual_seed(11 + d)
    q, g = (torch.randn(B, H, N, d, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    k, v = (torch.randn(B, H, Nk, d, generator=gen).to(torch.bfloat16).to(DEV) for _ in range(2))
    guard = 128 * d  # one more 128-row box of the tensor's width
    bufs, outs = [], []
    for shape in ((B, H, N, d), (B, H, N, d), (B, H, Nk, d), (B, H, Nk, d)):
        n = B * H * shape[2] * d
        buf = torch.full((n + guard,), SENTINEL, dtype=torch.bfloat16, device=DEV)
        bufs.append((buf, n))
        outs.append(buf[:n].view(shape))
    _run(q, k, v, g, d ** -0.5, True, tuple(outs))
    for (buf, n), out in zip(bufs, outs):
        assert not (out == SENTINEL).any()
        assert bool((buf[n:] == SENTINEL).all())
