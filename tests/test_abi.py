"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/fa.h declares, and rejects bad arguments before it
touches CUDA."""

import ctypes
import os
import re

import pytest
import torch

import flashattention_backward_gb300 as fa
from flashattention_backward_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "fa_bwd" in names and "fa_fwd" in names and "fa_convert_dq" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strings(lib):
    assert lib.fa_version() >= 100
    assert fa.status_string(fa.FA_ERR_TIMEOUT) == "device wait timed out"


def _prob(**kw):
    base = dict(B=1, H=2, N=100, d=64, scale=0.125, causal=1, dtype=fa.FA_BF16, flags=0,
                stride_b=2 * 100 * 64, stride_h=100 * 64, stride_n=64)
    base.update(kw)
    return fa.FaProblem(**base)


def test_dq_accum_size(lib):
    p = _prob(N=4000, d=128, H=16, B=4, stride_b=16 * 4000 * 128, stride_h=4000 * 128, stride_n=128)
    assert fa.fa_dq_accum_elems(p) == 4 * 16 * 32 * 128 * 128
    p = _prob(N=48, d=16, H=1, dtype=fa.FA_FP32, stride_b=48 * 16, stride_h=48 * 16, stride_n=16)
    assert fa.fa_dq_accum_elems(p) == 128 * 16
    assert fa.fa_dq_accum_elems(_prob(d=96, stride_n=96)) == 1 * 2 * 128 * 96
    assert fa.fa_dq_accum_elems(_prob(d=48, stride_n=48)) == 0  # unsupported head dim
    # deterministic: one slice per key block (128 keys on the tensor-core
    # kernels, bf16 d = 256 included; 64 on the CUDA-core kernels, 32 on
    # those at d = 256)
    p = _prob(N=4000, d=128, H=16, B=4, stride_b=16 * 4000 * 128, stride_h=4000 * 128, stride_n=128,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 32 * 4 * 16 * 32 * 128 * 128
    p = _prob(N=48, d=16, H=1, dtype=fa.FA_FP32, stride_b=48 * 16, stride_h=48 * 16, stride_n=16,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 1 * 128 * 16
    p = _prob(N=100, d=256, H=1, stride_b=100 * 256, stride_h=100 * 256, stride_n=256,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 1 * 128 * 256
    p = _prob(N=100, d=256, H=1, dtype=fa.FA_FP32, stride_b=100 * 256, stride_h=100 * 256, stride_n=256,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 4 * 128 * 256
    p = _prob(N=100, d=96, H=1, stride_b=100 * 96, stride_h=100 * 96, stride_n=96, flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 1 * 128 * 96
    # N_k != N: one accumulator tile per 128 query rows, one slice per key block
    p = _prob(N=100, N_k=300, kstride_b=2 * 300 * 64, kstride_h=300 * 64, kstride_n=64)
    assert fa.fa_dq_accum_elems(p) == 2 * 128 * 64
    p = _prob(N=100, N_k=300, kstride_b=2 * 300 * 64, kstride_h=300 * 64, kstride_n=64,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 3 * 2 * 128 * 64
    p = _prob(N=100, N_k=300, kstride_b=2 * 300 * 64, kstride_h=300 * 64, kstride_n=64, dtype=fa.FA_FP32,
              flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_dq_accum_elems(p) == 5 * 2 * 128 * 64


BAD = 0x1000  # a 16-byte aligned dummy address; validation fails before any use


@pytest.mark.parametrize(
    "kw,code",
    [
        (dict(N=0), fa.FA_ERR_INVALID_ARG),
        (dict(B=0), fa.FA_ERR_INVALID_ARG),
        (dict(d=48, stride_n=48), fa.FA_ERR_UNSUPPORTED),  # d in {32, 64, 96, 128, 256} for bf16
        (dict(d=16, stride_n=16), fa.FA_ERR_UNSUPPORTED),
        (dict(d=512, stride_n=512), fa.FA_ERR_UNSUPPORTED),
        (dict(d=80, stride_n=80, dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),
        (dict(N_k=-1), fa.FA_ERR_INVALID_ARG),
        (dict(reserved=1), fa.FA_ERR_INVALID_ARG),
        (dict(N_k=50), fa.FA_ERR_INVALID_ARG),  # K strides left at 0
        (dict(N_k=50, kstride_b=2 * 50 * 64, kstride_h=50 * 64, kstride_n=60), fa.FA_ERR_INVALID_ARG),
        (dict(N_k=50, kstride_b=2 * 50 * 64, kstride_h=50 * 64, kstride_n=68), fa.FA_ERR_INVALID_ARG),
        (dict(N_k=(1 << 24) + 1, kstride_b=64, kstride_h=64, kstride_n=64), fa.FA_ERR_UNSUPPORTED),
        # a 1-D grid of B*H*ceil(rows/32)*2 CTAs would pass 2^31 - 1
        (dict(B=1 << 10, H=1 << 14, N=1 << 12, stride_b=(1 << 14) * (1 << 12) * 64,
              stride_h=(1 << 12) * 64, stride_n=64), fa.FA_ERR_UNSUPPORTED),
        (dict(causal=2), fa.FA_ERR_INVALID_ARG),
        (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
        (dict(flags=2), fa.FA_ERR_INVALID_ARG),
        (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
        (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
        (dict(stride_n=60), fa.FA_ERR_INVALID_ARG),
        (dict(stride_n=68), fa.FA_ERR_INVALID_ARG),  # 136 bytes: not a multiple of 16
    ],
)
def test_validation_rejects(lib, kw, code):
    p = _prob(**kw)
    r = lib.fa_bwd(ctypes.byref(p), BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, None)
    assert r == code
    r = lib.fa_fwd(ctypes.byref(p), BAD, BAD, BAD, BAD, BAD, None)
    assert r == code


def test_fused_backward_host_checks(lib):
    p = _prob(B=2, H=3)
    assert lib.fa_backward_fused_sync_elems(ctypes.byref(p)) == 1 + 2 * 6
    p32 = _prob(dtype=fa.FA_FP32, stride_b=2 * 100 * 64, stride_h=100 * 64, stride_n=64)
    assert lib.fa_backward_fused_sync_elems(ctypes.byref(p32)) == 0  # CUDA-core problems: separate launches only
    args = [BAD] * 13
    assert lib.fa_backward_fused(ctypes.byref(p32), *args, None) == fa.FA_ERR_UNSUPPORTED
    p256 = _prob(d=256, stride_b=2 * 100 * 256, stride_h=100 * 256, stride_n=256)
    assert lib.fa_backward_fused(ctypes.byref(p256), *args, None) == fa.FA_ERR_UNSUPPORTED
    bad_sync = list(args)
    bad_sync[9] = BAD + 2  # sync must be 4-byte aligned
    assert lib.fa_backward_fused(ctypes.byref(p), *bad_sync, None) == fa.FA_ERR_INVALID_ARG
    bad_sync[9] = 0
    assert lib.fa_backward_fused(ctypes.byref(p), *bad_sync, None) == fa.FA_ERR_INVALID_ARG


def test_null_and_misaligned_pointers(lib):
    p = _prob()
    assert lib.fa_bwd(None, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd(ctypes.byref(p), 0, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd(ctypes.byref(p), BAD + 8, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_preprocess(ctypes.byref(p), BAD, BAD, BAD, BAD + 4, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_convert_dq(ctypes.byref(p), BAD, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_get_device_status(None, None) == fa.FA_ERR_INVALID_ARG


def test_binding_rejects_mismatched_tensors():
    q = torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16)
    p = fa.problem_for(q, 0.125, True)
    assert (p.B, p.H, p.N, p.d, p.stride_n) == (1, 2, 16, 64, 64)
    with pytest.raises(ValueError):
        fa.problem_for(q[..., ::2], 0.125, True)
    with pytest.raises(TypeError):
        fa.problem_for(q.half(), 0.125, True)
    with pytest.raises(ValueError):  # CPU tensors are refused: no CPU path exists
        fa._same_layout(p, q)


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(fa, "_LIB", None)
    monkeypatch.setenv("FA_LIBRARY", "/nonexistent/libfa.so")
    with pytest.raises(RuntimeError):
        fa.load_library()
