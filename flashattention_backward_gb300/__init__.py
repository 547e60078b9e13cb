"""GB300 (sm_103a) FlashAttention-2 backward: Python binding of libfa.

The binding only marshals arguments (shapes, strides, raw device pointers,
the current CUDA stream) into the C ABI of ``include/fa.h``; every step of
the computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.  There is no fallback: if ``libfa.so`` is missing or a
call fails, an exception is raised.

Entry points mirror the C names: :func:`fa_fwd`, :func:`fa_bwd_preprocess`,
:func:`fa_bwd`, :func:`fa_convert_dq`, :func:`fa_backward`, plus
:func:`attention_forward` / :func:`attention_backward`, which allocate their
outputs with torch and call those.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "FaError",
    "FaProblem",
    "FA_FLAG_DETERMINISTIC",
    "problem_for",
    "fa_dq_accum_elems",
    "fa_fwd",
    "fa_bwd_preprocess",
    "fa_bwd",
    "fa_bwd_tile_pair_count",
    "fa_convert_dq",
    "fa_backward",
    "fa_backward_host",
    "fa_backward_host_workspace_bytes",
    "attention_forward",
    "attention_backward_host",
    "attention_backward",
    "FlashAttnFunction",
    "flash_attn_func",
    "get_device_status",
    "set_wait_limit_ns",
    "selftest_wait_timeout",
    "library_path",
    "load_library",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_DEVICE = range(6)
FA_BF16, FA_FP32 = 0, 1
FA_FLAG_DETERMINISTIC = 1
TILE_ROWS = 128


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class FaProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("N", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("stride_b", ctypes.c_int64),
        ("stride_h", ctypes.c_int64),
        ("stride_n", ctypes.c_int64),
        ("N_k", ctypes.c_int32),  # 0: N_k = N, K-shaped strides = Q strides
        ("reserved", ctypes.c_int32),
        ("kstride_b", ctypes.c_int64),
        ("kstride_h", ctypes.c_int64),
        ("kstride_n", ctypes.c_int64),
    ]


_LIB: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return os.environ.get("FA_LIBRARY", _build.LIB)


def load_library() -> ctypes.CDLL:
    """Load libfa.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libfa.so not found at {path}: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FaProblem)
    vp, fp, st = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
    lib.fa_dq_accum_elems.argtypes = [P]
    lib.fa_dq_accum_elems.restype = ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, vp, vp, vp, vp, fp, vp]
    lib.fa_bwd_preprocess.argtypes = [P, vp, vp, fp, fp, vp]
    lib.fa_bwd.argtypes = [P, vp, vp, vp, vp, fp, fp, fp, vp, vp, vp]
    lib.fa_convert_dq.argtypes = [P, fp, vp, vp]
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.fa_bwd_tile_pair_count.argtypes = [P, vp, vp, vp, vp, fp, fp, fp, vp, vp, vp, i32p, i32p, vp]
    lib.fa_bwd_tile_pair_count.restype = st
    lib.fa_backward.argtypes = [P, vp, vp, vp, vp, vp, fp, fp, fp, vp, vp, vp, vp]
    for name in ("fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_convert_dq", "fa_backward"):
        getattr(lib, name).restype = st
    lib.fa_backward_fused_sync_elems.argtypes = [P]
    lib.fa_backward_fused_sync_elems.restype = ctypes.c_size_t
    lib.fa_backward_fused.argtypes = [P] + [vp] * 13
    lib.fa_backward_fused.restype = st
    lib.fa_backward_host_workspace_bytes.argtypes = [P, ctypes.c_int32]
    lib.fa_backward_host_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_backward_host.argtypes = [P] + [vp] * 9 + [vp, ctypes.c_size_t, ctypes.c_int32, vp]
    lib.fa_backward_host.restype = st
    lib.fa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.fa_get_device_status.restype = st
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.fa_set_wait_limit_ns.restype = None
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.fa_selftest_wait_timeout.restype = st
    lib.fa_status_string.argtypes = [st]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_int32
    _LIB = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load_library().fa_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - only for messages
        return "status"


def _check(code: int, what: str) -> None:
    if code != FA_OK:
        raise FaError(code, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def problem_for(q: torch.Tensor, scale: float, causal: bool, deterministic: bool = False,
                k: Optional[torch.Tensor] = None) -> FaProblem:
    """Problem descriptor for Q-shaped [B, H, N, d] tensors laid out like ``q``
    and, if ``k`` is given, K-shaped [B, H, N_k, d] tensors laid out like ``k``
    (otherwise N_k = N with q's strides).  Causal masks are aligned
    bottom-right: key j is visible to query i iff j <= i + N_k - N."""
    if q.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    if q.stride(3) != 1:
        raise ValueError("the last dimension must be contiguous")
    B, H, N, d = q.shape
    flags = FA_FLAG_DETERMINISTIC if deterministic else 0
    p = FaProblem(B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), flags,
                  q.stride(0), q.stride(1), q.stride(2))
    if k is not None:
        if k.dim() != 4 or k.shape[0] != B or k.shape[1] != H or k.shape[3] != d or k.stride(3) != 1:
            raise ValueError("k must be a [B, H, N_k, d] tensor with a contiguous last dimension")
        p.N_k = k.shape[2]
        p.kstride_b, p.kstride_h, p.kstride_n = k.stride(0), k.stride(1), k.stride(2)
    return p


def _k_rows(p: FaProblem):
    """Rows and strides of the K-shaped tensors of p."""
    if p.N_k == 0:
        return p.N, (p.stride_b, p.stride_h, p.stride_n, 1)
    return p.N_k, (p.kstride_b, p.kstride_h, p.kstride_n, 1)


def _check_tensors(p: FaProblem, shape, strides, ts) -> None:
    for t in ts:
        if tuple(t.shape) != shape or t.stride() != strides:
            raise ValueError(f"tensor of shape {tuple(t.shape)} strides {t.stride()}: expected {shape} {strides}")
        if _dtype_code(t) != p.dtype:
            raise ValueError("all [B, H, rows, d] tensors must share the dtype")
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")


def _same_layout(p: FaProblem, *ts: torch.Tensor) -> None:
    """Q-shaped tensors: [B, H, N, d] with the Q strides."""
    _check_tensors(p, (p.B, p.H, p.N, p.d), (p.stride_b, p.stride_h, p.stride_n, 1), ts)


def _k_layout(p: FaProblem, *ts: torch.Tensor) -> None:
    """K-shaped tensors: [B, H, N_k, d] with the K strides."""
    rows, strides = _k_rows(p)
    _check_tensors(p, (p.B, p.H, rows, p.d), strides, ts)


def _rows(p: FaProblem, *ts: torch.Tensor) -> None:
    for t in ts:
        if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != p.B * p.H * p.N or not t.is_cuda:
            raise ValueError("L and D must be contiguous float32 CUDA tensors of B*H*N elements")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def fa_dq_accum_elems(p: FaProblem) -> int:
    return int(load_library().fa_dq_accum_elems(ctypes.byref(p)))


def fa_fwd(p: FaProblem, q, k, v, o, L, stream=None) -> None:
    _same_layout(p, q, o)
    _k_layout(p, k, v)
    _rows(p, L)
    _check(load_library().fa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), _stream(stream)),
           "fa_fwd")


def fa_bwd_preprocess(p: FaProblem, o, do, D, dq_accum, stream=None) -> None:
    _same_layout(p, o, do)
    _rows(p, D)
    _accum(p, dq_accum)
    _check(load_library().fa_bwd_preprocess(ctypes.byref(p), _ptr(o), _ptr(do), _ptr(D), _ptr(dq_accum),
                                            _stream(stream)), "fa_bwd_preprocess")


def _accum(p: FaProblem, acc: torch.Tensor) -> None:
    if acc.dtype != torch.float32 or not acc.is_contiguous() or acc.numel() < fa_dq_accum_elems(p):
        raise ValueError("dq_accum must be a contiguous float32 tensor of fa_dq_accum_elems() elements")


def fa_bwd(p: FaProblem, q, k, v, do, L, D, dq_accum, dk, dv, stream=None) -> None:
    _same_layout(p, q, do)
    _k_layout(p, k, v, dk, dv)
    _rows(p, L, D)
    _accum(p, dq_accum)
    _check(load_library().fa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(L), _ptr(D),
                                 _ptr(dq_accum), _ptr(dk), _ptr(dv), _stream(stream)), "fa_bwd")


def fa_bwd_tile_pair_count(p: FaProblem, q, k, v, do, L, D, dq_accum, dk, dv, counts, stream=None):
    """fa_bwd that also adds the executed (key block, query block) pairs to
    ``counts[0]`` and those with no visible entry to ``counts[1]`` (``counts``:
    a zeroed int64 CUDA tensor of 2 elements).  Returns the kernel's block
    heights (key_rows, query_rows)."""
    _same_layout(p, q, do)
    _k_layout(p, k, v, dk, dv)
    _rows(p, L, D)
    _accum(p, dq_accum)
    if counts.dtype != torch.int64 or not counts.is_cuda or counts.numel() < 2:
        raise ValueError("counts must be an int64 CUDA tensor of 2 elements")
    kr, qr = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().fa_bwd_tile_pair_count(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(L),
                                                 _ptr(D), _ptr(dq_accum), _ptr(dk), _ptr(dv), _ptr(counts),
                                                 ctypes.byref(kr), ctypes.byref(qr), _stream(stream)),
           "fa_bwd_tile_pair_count")
    return int(kr.value), int(qr.value)


def fa_convert_dq(p: FaProblem, dq_accum, dq, stream=None) -> None:
    _same_layout(p, dq)
    _accum(p, dq_accum)
    _check(load_library().fa_convert_dq(ctypes.byref(p), _ptr(dq_accum), _ptr(dq), _stream(stream)),
           "fa_convert_dq")


def fa_backward(p: FaProblem, q, k, v, o, do, L, D, dq_accum, dq, dk, dv, stream=None) -> None:
    _same_layout(p, q, o, do, dq)
    _k_layout(p, k, v, dk, dv)
    _rows(p, L, D)
    _accum(p, dq_accum)
    _check(load_library().fa_backward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                      _ptr(D), _ptr(dq_accum), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)),
           "fa_backward")


def fa_backward_fused_sync_elems(p: FaProblem) -> int:
    return int(load_library().fa_backward_fused_sync_elems(ctypes.byref(p)))


def fa_backward_fused(p: FaProblem, q, k, v, o, do, L, D, dq_accum, sync, dq, dk, dv, stream=None) -> None:
    """fa_backward in a single kernel launch (tensor-core problems only)."""
    _same_layout(p, q, o, do, dq)
    _k_layout(p, k, v, dk, dv)
    _rows(p, L, D)
    _accum(p, dq_accum)
    if sync.dtype != torch.int32 or not sync.is_cuda or sync.numel() < fa_backward_fused_sync_elems(p):
        raise ValueError("sync must be an int32 CUDA tensor of fa_backward_fused_sync_elems() elements")
    _check(load_library().fa_backward_fused(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                            _ptr(D), _ptr(dq_accum), _ptr(sync), _ptr(dq), _ptr(dk), _ptr(dv),
                                            _stream(stream)), "fa_backward_fused")


def attention_forward(q, k, v, scale: float, causal: bool = False, stream=None):
    """O, L for [B, H, N, d] queries and [B, H, N_k, d] keys/values (CUDA, bf16
    or fp32; last dimension contiguous)."""
    p = problem_for(q, scale, causal, k=k)
    o = torch.empty_like(q)
    L = torch.empty((p.B, p.H, p.N), dtype=torch.float32, device=q.device)
    fa_fwd(p, q, k, v, o, L, stream)
    return o, L


def _raise_on_device_error(stream, what: str) -> None:
    code = get_device_status(stream)
    if code != FA_OK:
        raise FaError(code, what)


def attention_backward(q, k, v, o, do, L, scale: float, causal: bool = False, stream=None, workspace=None,
                       deterministic: bool = False, fused: bool = False, check_status: bool = False):
    """dQ, dK, dV.  ``workspace`` may pass preallocated (D, dq_accum) or, with
    ``fused`` (one kernel launch, tensor-core problems), (D, dq_accum, sync).

    The kernels report device-side errors (a bounded wait that ran out) only
    through the device status word, and leave their outputs partial in that
    case.  With ``check_status`` the call synchronises the stream, reads the
    word and raises :class:`FaError` if it holds an error; otherwise the
    caller should call :func:`get_device_status` after the step."""
    p = problem_for(q, scale, causal, deterministic, k=k)
    if workspace is None:
        D = torch.empty((p.B, p.H, p.N), dtype=torch.float32, device=q.device)
        acc = torch.empty(fa_dq_accum_elems(p), dtype=torch.float32, device=q.device)
        sync = torch.empty(fa_backward_fused_sync_elems(p) if fused else 0, dtype=torch.int32, device=q.device)
    else:
        D, acc = workspace[0], workspace[1]
        sync = workspace[2] if fused else None
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if fused:
        fa_backward_fused(p, q, k, v, o, do, L, D, acc, sync, dq, dk, dv, stream)
    else:
        fa_backward(p, q, k, v, o, do, L, D, acc, dq, dk, dv, stream)
    if check_status:
        _raise_on_device_error(stream, "fa_backward (device)")
    return dq, dk, dv


class FlashAttnFunction(torch.autograd.Function):
    """Autograd node over the library: forward = fa_fwd (O and the row
    logsumexp L are saved), backward = fa_backward (preprocess, main kernel,
    convert).  Tensors are [B, H, N, d] (K, V: [B, H, N_k, d]) on a CUDA
    device, bf16 or fp32, last dimension contiguous; tensors of one shape
    whose strides differ are passed to the library as dense copies.  With
    ``check_status`` both passes read the device status word and raise
    :class:`FaError` on a device-side error (see :func:`attention_backward`)."""

    @staticmethod
    def forward(ctx, q, k, v, causal: bool, scale: float, deterministic: bool, check_status: bool = False):
        if q.stride(-1) != 1:
            q = q.contiguous()
        if k.stride(-1) != 1 or v.stride() != k.stride():
            k, v = k.contiguous(), v.contiguous()
        o, L = attention_forward(q, k, v, scale, causal)
        if check_status:
            _raise_on_device_error(None, "fa_fwd (device)")
        ctx.save_for_backward(q, k, v, o, L)
        ctx.causal, ctx.scale, ctx.deterministic, ctx.check_status = causal, scale, deterministic, check_status
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, L = ctx.saved_tensors
        if do.stride() != o.stride():
            if q.is_contiguous():
                do = do.contiguous()
            else:  # the library takes dO with the strides of O
                do = torch.empty_like(o).copy_(do)
        dq, dk, dv = attention_backward(q, k, v, o, do, L, ctx.scale, ctx.causal,
                                        deterministic=ctx.deterministic, check_status=ctx.check_status)
        return dq, dk, dv, None, None, None, None


def flash_attn_func(q, k, v, causal: bool = False, softmax_scale: Optional[float] = None,
                    deterministic: bool = False, check_status: bool = False):
    """O = softmax(softmax_scale Q K^T) V (default scale 1/sqrt(d)), with the
    FlashAttention-2 backward of this library under autograd.

    A device-side error (a bounded wait that ran out inside a kernel) is only
    recorded in the device status word and leaves the outputs partial: pass
    ``check_status=True`` to have both passes check the word and raise
    :class:`FaError`, or call :func:`get_device_status` after the step."""
    scale = float(softmax_scale) if softmax_scale is not None else q.shape[-1] ** -0.5
    return FlashAttnFunction.apply(q, k, v, bool(causal), scale, bool(deterministic), bool(check_status))


def fa_backward_host_workspace_bytes(p: FaProblem, heads_per_group: int = 0) -> int:
    return int(load_library().fa_backward_host_workspace_bytes(ctypes.byref(p), int(heads_per_group)))


def fa_backward_host(p: FaProblem, q, k, v, o, do, L, dq, dk, dv, workspace, heads_per_group: int = 0,
                     stream=None) -> None:
    """Backward from host tensors (dense, ideally pinned) through a device
    workspace; see include/fa.h."""
    rows_k, _ = _k_rows(p)
    for t, rows in ((q, p.N), (o, p.N), (do, p.N), (dq, p.N), (k, rows_k), (v, rows_k), (dk, rows_k), (dv, rows_k)):
        if t.is_cuda or not t.is_contiguous() or t.shape != (p.B, p.H, rows, p.d) or _dtype_code(t) != p.dtype:
            raise ValueError("host tensors must be dense [B, H, rows, d] CPU tensors of the problem dtype")
    if L.is_cuda or not L.is_contiguous() or L.numel() != p.B * p.H * p.N or L.dtype != torch.float32:
        raise ValueError("L must be a dense float32 CPU tensor of B*H*N elements")
    if not workspace.is_cuda:
        raise ValueError("workspace must be device memory")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load_library().fa_backward_host(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                           _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), nbytes,
                                           int(heads_per_group), _stream(stream)), "fa_backward_host")


def attention_backward_host(q, k, v, o, do, L, scale: float, causal: bool = False, heads_per_group: int = 0,
                            workspace=None, out=None, stream=None, deterministic: bool = False):
    """dQ, dK, dV (pinned host tensors) for host-resident inputs."""
    p = problem_for(q, scale, causal, deterministic, k=k)
    if workspace is None:
        workspace = torch.empty(fa_backward_host_workspace_bytes(p, heads_per_group), dtype=torch.uint8,
                                device="cuda")
    if out is None:
        out = (torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory(), torch.empty_like(v).pin_memory())
    fa_backward_host(p, q, k, v, o, do, L, *out, workspace, heads_per_group, stream)
    return out


def get_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    code = ctypes.c_int32(0)
    _check(load_library().fa_get_device_status(_stream(stream), ctypes.byref(code)), "fa_get_device_status")
    return int(code.value)


def set_wait_limit_ns(ns: int) -> None:
    load_library().fa_set_wait_limit_ns(int(ns))


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load_library().fa_selftest_wait_timeout(int(limit_ns), _stream(stream)), "fa_selftest_wait_timeout")
