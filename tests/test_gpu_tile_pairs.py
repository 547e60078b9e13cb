"""Causal tile skip, counted on the device.

CS349E lecture 11 demo 4: over T x T square blocks a causal backward needs
only the T(T+1)/2 (key block, query block) pairs that hold a visible entry
("CUDA 算子工程" ch.16 §16.8 item 2: skip fully masked tiles).  Parity cannot
see extra fully masked pairs (they add zeros), so fa_bwd_tile_pair_count has
the kernels count the pairs they execute and those among them with no visible
entry.  The expected counts come from the oracle's block count
(causal_executed_tile_pairs, pinned against T(T+1)/2 and an entry-level brute
force), times B*H; the masked count must be 0.  The counting run's dK and dV
must equal plain fa_bwd's bit for bit (they are written once per key block)."""

import pytest
import torch

import flashattention_backward_gb300 as fa
from oracle import causal_executed_tile_pairs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


CASES = [
    # B, H, N, N_k, d, causal, dtype, deterministic
    (1, 32, 8192, 8192, 128, True, torch.bfloat16, False),    # 2080 pairs per head
    (4, 16, 4000, 4000, 128, True, torch.bfloat16, False),    # 528 pairs per head, ragged tail
    (1, 32, 2048, 2048, 64, False, torch.bfloat16, False),    # 16 x 16 per head
    (1, 8, 32768, 32768, 128, True, torch.bfloat16, False),   # 32896 pairs per head
    (1, 16, 8192, 8192, 256, True, torch.bfloat16, False),    # 128 x 64 blocks
    (2, 3, 1000, 777, 128, True, torch.bfloat16, False),
    (1, 2, 200, 330, 64, True, torch.bfloat16, True),
    (1, 2, 1000, 600, 256, True, torch.bfloat16, False),
    (1, 2, 330, 200, 96, True, torch.bfloat16, False),
    (1, 3, 300, 200, 64, True, torch.float32, False),
    (1, 2, 300, 300, 256, True, torch.float32, False),
]


@pytest.mark.parametrize("B,H,N,Nk,d,causal,dtype,det", CASES)
def test_executed_tile_pairs(B, H, N, Nk, d, causal, dtype, det):
    gen = torch.Generator(device=DEV).manual_seed(N + Nk + d)
    q, g = (torch.randn(B, H, N, d, device=DEV, generator=gen).to(dtype) for _ in range(2))
    k, v = (torch.randn(B, H, Nk, d, device=DEV, generator=gen).to(dtype) for _ in range(2))
    scale = d ** -0.5
    o, L = fa.attention_forward(q, k, v, scale, causal)
    p = fa.problem_for(q, scale, causal, det, k=k)
    D = torch.empty(B, H, N, device=DEV)
    acc = torch.empty(fa.fa_dq_accum_elems(p), device=DEV)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_preprocess(p, o, g, D, acc)
    counts = torch.zeros(2, dtype=torch.int64, device=DEV)
    kr, qr = fa.fa_bwd_tile_pair_count(p, q, k, v, g, L, D, acc, dk, dv, counts)
    dk2, dv2 = torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_preprocess(p, o, g, D, acc)
    fa.fa_bwd(p, q, k, v, g, L, D, acc, dk2, dv2)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    expect = B * H * causal_executed_tile_pairs(N, qr, kr, N_k=Nk, causal=causal)
    executed, masked = (int(x) for x in counts.cpu())
    assert (executed, masked) == (expect, 0)
    if causal and N == Nk and kr == qr and N % kr == 0:
        T = N // kr
        assert executed == B * H * T * (T + 1) // 2
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_tile_pair_count_rejects_bad_counts_pointer():
    import ctypes

    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=DEV)
    p = fa.problem_for(q, 0.125, True)
    lib = fa.load_library()
    kr, qr = ctypes.c_int32(0), ctypes.c_int32(0)
    ptr = q.data_ptr()
    r = lib.fa_bwd_tile_pair_count(ctypes.byref(p), *([ptr] * 9), None, ctypes.byref(kr), ctypes.byref(qr), None)
    assert r == fa.FA_ERR_INVALID_ARG
