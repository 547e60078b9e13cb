"""GPU parity of the bandwidth kernels, the forward and the fp32 backward
against the float64 oracle, plus the device status / bounded-wait checks."""

import numpy as np
import pytest
import torch

import flashattention_backward_gb300 as fa
from fa_inputs import make_inputs, to_f64, workload
from gpu_common import compare_head, ratio, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.load_library()
    assert fa.get_device_status() == 0


def _accum_index(B, H, N, d):
    """Float index of element (b, h, n, c) in the unit-blocked accumulator
    layout that include/fa.h documents."""
    T = -(-N // 128)
    b, h, n, c = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), np.arange(d), indexing="ij")
    unit = (((b * H + h) * T + n // 128) * 4 + (n % 128) // 32) * (d // 16) + c // 16
    return unit * 512 + ((c % 16) // 4) * 128 + (n % 32) * 4 + c % 4


@pytest.mark.parametrize("dtype,d,N", [(torch.bfloat16, 64, 300), (torch.bfloat16, 128, 129),
                                       (torch.float32, 16, 48), (torch.float32, 128, 1),
                                       (torch.bfloat16, 96, 200), (torch.bfloat16, 32, 130),
                                       (torch.bfloat16, 256, 129), (torch.float32, 96, 77),
                                       (torch.float32, 256, 300)])
def test_preprocess_computes_D_and_zeroes_accumulator(dtype, d, N):
    B, H = 2, 3
    gen = torch.Generator().manual_seed(5)
    o = torch.randn(B, H, N, d, generator=gen).to(dtype)
    do = torch.randn(B, H, N, d, generator=gen).to(dtype)
    p = fa.problem_for(o, 0.1, False)
    D = torch.full((B, H, N), float("nan"), device=DEV)
    acc = torch.full((fa.fa_dq_accum_elems(p),), float("nan"), device=DEV)
    fa.fa_bwd_preprocess(p, o.to(DEV), do.to(DEV), D, acc)
    torch.cuda.synchronize()
    ref = np.sum(to_f64(o) * to_f64(do), axis=-1)
    np.testing.assert_allclose(to_f64(D), ref, rtol=1e-5, atol=1e-5)
    assert torch.count_nonzero(acc).item() == 0


@pytest.mark.parametrize("dtype,d,N", [(torch.bfloat16, 128, 300), (torch.bfloat16, 64, 128),
                                       (torch.float32, 16, 48), (torch.float32, 32, 257),
                                       (torch.bfloat16, 96, 129), (torch.bfloat16, 256, 200),
                                       (torch.float32, 96, 130), (torch.float32, 256, 1)])
def test_convert_undoes_the_documented_layout(dtype, d, N):
    B, H = 2, 2
    q = torch.empty(B, H, N, d, dtype=dtype)
    p = fa.problem_for(q, 0.37, False)
    gen = torch.Generator().manual_seed(6)
    acc = torch.randn(fa.fa_dq_accum_elems(p), generator=gen)
    dq = torch.empty(B, H, N, d, dtype=dtype, device=DEV)
    fa.fa_convert_dq(p, acc.to(DEV), dq)
    torch.cuda.synchronize()
    idx = _accum_index(B, H, N, d)
    expect = (torch.from_numpy(acc.numpy()[idx]) * torch.tensor(0.37, dtype=torch.float32)).to(dtype)
    assert torch.equal(dq.cpu(), expect)  # bitwise: same fp32 product, same RNE cast


@pytest.mark.parametrize("dtype,d,N", [(torch.bfloat16, 128, 300), (torch.bfloat16, 64, 129),
                                       (torch.bfloat16, 32, 77), (torch.float32, 16, 48),
                                       (torch.float32, 128, 130)])
def test_convert_to_an_output_off_the_32_byte_grid(dtype, d, N):
    """dQ starting 16 bytes past a 32-byte boundary takes the 128-bit store
    path; the result is the same, and the guard elements on both sides stay."""
    B, H = 2, 2
    q = torch.empty(B, H, N, d, dtype=dtype)
    p = fa.problem_for(q, 0.37, False)
    gen = torch.Generator().manual_seed(16)
    acc = torch.randn(fa.fa_dq_accum_elems(p), generator=gen)
    shift = 16 // q.element_size()
    n = B * H * N * d
    buf = torch.full((n + 2 * shift,), -7.0, dtype=dtype, device=DEV)
    dq = buf[shift:shift + n].view(B, H, N, d)
    assert dq.data_ptr() % 32 == 16
    fa.fa_convert_dq(p, acc.to(DEV), dq)
    torch.cuda.synchronize()
    idx = _accum_index(B, H, N, d)
    expect = (torch.from_numpy(acc.numpy()[idx]) * torch.tensor(0.37, dtype=torch.float32)).to(dtype)
    assert torch.equal(dq.cpu(), expect)
    assert bool((buf[:shift] == -7.0).all()) and bool((buf[shift + n:] == -7.0).all())


def test_forward_four_numbers_across_a_tile_boundary():
    """The write-up's four-number example spread over two 64-key tiles:
    scores 0 then 10, values 0 then 1 -> 0.9999546 (not the 0.5 of a naive
    per-block average); the second tile brings the new row maximum."""
    N, d = 128, 16
    q = torch.zeros(1, 1, N, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, N, d)
    k[0, 0, 64:, 0] = 10.0
    v = torch.zeros(1, 1, N, d)
    v[0, 0, 64:, :] = 1.0
    o, L = fa.attention_forward(q.to(DEV), k.to(DEV), v.to(DEV), 1.0, False)
    torch.cuda.synchronize()
    assert abs(o[0, 0, 0, 0].item() - 0.9999546) < 5e-7
    assert abs(L[0, 0, 0].item() - (10 + np.log(64 + 64 * np.exp(-10.0)))) < 1e-5


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_forward_four_numbers_new_max_in_later_block(d):
    """Same example on the tensor-core forward: 128 keys of score 0, then
    128 keys of score 10.  The second key block raises the row maximum by
    14.4 in exp2 units, so the running base moves and O is rescaled."""
    N = 256
    q = torch.zeros(1, 1, N, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, N, d)
    k[0, 0, 128:, 0] = 10.0
    v = torch.zeros(1, 1, N, d)
    v[0, 0, 128:, :] = 1.0
    to = lambda t: t.to(torch.bfloat16).to(DEV)
    o, L = fa.attention_forward(to(q), to(k), to(v), 1.0, False)
    torch.cuda.synchronize()
    assert fa.get_device_status() == 0
    assert abs(o[0, 0, 0, 0].float().item() - 0.9999546) < 4e-3  # bf16 output, not the naive 0.5
    assert abs(L[0, 0, 0].item() - (10 + np.log(128 + 128 * np.exp(-10.0)))) < 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_tiny_workload(causal):
    w = workload("tiny", causal=causal)
    out = run_gpu(w, DEV)
    assert out["status"] == 0
    compare_head(out, w, 0, 0, tol=1e-5, L_tol=1e-6)


@pytest.mark.parametrize("N,d,causal", [(1, 16, True), (200, 32, True), (129, 64, False), (300, 128, True)])
def test_fp32_backward_shapes(N, d, causal):
    w = workload("tiny", N=N, d=d, causal=causal, B=2, H=2, seed=3).with_(name="fp32_case")
    gen = torch.Generator().manual_seed(N + d)
    inputs = tuple(torch.randn(w.B, w.H, N, d, generator=gen) for _ in range(4))
    out = run_gpu(w, DEV, inputs)
    assert out["status"] == 0
    for b in range(w.B):
        for h in range(w.H):
            compare_head(out, w, b, h, tol=1e-5, L_tol=1e-6)


@pytest.mark.parametrize("N,d,causal", [(1, 64, False), (77, 64, True), (256, 128, False), (1000, 128, True)])
def test_bf16_forward(N, d, causal):
    w = workload("causal", B=1, H=2, N=N, d=d, causal=causal, seed=11)
    q, k, v, _ = (t.to(DEV) for t in make_inputs(w))
    o, L = fa.attention_forward(q, k, v, w.scale, w.causal)
    torch.cuda.synchronize()
    from oracle import attention_forward

    for h in range(2):
        Or, Lr = attention_forward(to_f64(q[0, h]), to_f64(k[0, h]), to_f64(v[0, h]), w.scale, causal)
        assert ratio(to_f64(o[0, h]), Or[0, 0]) <= 2e-2
        assert ratio(to_f64(L[0, h]), Lr[0, 0]) <= 1e-3


def test_device_status_stays_clean_and_selftest_times_out():
    assert fa.get_device_status() == 0
    fa.selftest_wait_timeout(5_000_000)  # 5 ms; nothing ever arrives
    assert fa.get_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.get_device_status() == 0  # reading clears the word
    # the context is still usable afterwards
    x = torch.ones(4, device=DEV)
    assert x.sum().item() == 4.0
