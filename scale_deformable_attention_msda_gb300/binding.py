"""Thin Python binding of libmsda's C ABI (include/msda.h), same names.

Argument marshalling only: every step of the operator runs in libmsda's CUDA
kernels. Tensors must be CUDA, contiguous and of one float dtype; the calls are
enqueued on the current torch CUDA stream and return without synchronising.
There is no CPU path: if libmsda.so is missing or the tensors are not on a GPU,
the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MSDA_F32, MSDA_BF16, MSDA_F16, MSDA_F64 = 0, 1, 2, 3
MSDA_ACC_NATIVE, MSDA_ACC_FP32_BUFFER, MSDA_ACC_AUTO, MSDA_ACC_FP16_BUFFER = 0, 1, 2, 3
_DTYPES = {torch.float32: MSDA_F32, torch.bfloat16: MSDA_BF16, torch.float16: MSDA_F16,
           torch.float64: MSDA_F64}
STATUS = {0: "MSDA_OK", 1: "MSDA_ERR_NULL", 2: "MSDA_ERR_SHAPE", 3: "MSDA_ERR_DTYPE",
          4: "MSDA_ERR_ALIGN", 5: "MSDA_ERR_WORKSPACE", 6: "MSDA_ERR_CUDA",
          7: "MSDA_ERR_DEVICE_BOUNDS"}
MSDA_ERR_DEVICE_BOUNDS = 7
EXPORTED = ("msda_forward", "msda_backward_workspace_bytes", "msda_backward",
            "msda_backward_zero", "msda_backward_accumulate", "msda_backward_finish",
            "msda_backward_static_workspace", "msda_forward_softmax", "msda_backward_softmax",
            "msda_debug_corners", "msda_checked_build", "msda_device_check",
            "msda_debug_bounds_self_test", "msda_set_sample_split", "msda_status_string",
            "msda_version")


class msda_dims_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "S", "Q", "M", "D", "L", "K")]


class MSDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({lib().msda_status_string(status).decode()})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBRARY


def load(path: str | None = None):
    """Open libmsda.so and declare its entry points (no CUDA call is made)."""
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libmsda.so not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    so = ctypes.CDLL(path)
    vp, i32p = ctypes.c_void_p, ctypes.c_void_p
    dims = ctypes.POINTER(msda_dims_t)
    so.msda_forward.argtypes = [vp, vp, vp, vp, vp, i32p, vp, dims, ctypes.c_int, vp]
    so.msda_forward.restype = ctypes.c_int
    so.msda_backward_workspace_bytes.argtypes = [dims, ctypes.c_int, ctypes.c_int]
    so.msda_backward_workspace_bytes.restype = ctypes.c_size_t
    so.msda_backward.argtypes = [vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                 ctypes.c_int, dims, ctypes.c_int, vp]
    so.msda_backward.restype = ctypes.c_int
    so.msda_forward_softmax.argtypes = so.msda_forward.argtypes
    so.msda_forward_softmax.restype = ctypes.c_int
    so.msda_backward_softmax.argtypes = so.msda_backward.argtypes
    so.msda_backward_softmax.restype = ctypes.c_int
    so.msda_backward_accumulate.argtypes = so.msda_backward.argtypes
    so.msda_backward_accumulate.restype = ctypes.c_int
    so.msda_backward_zero.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int, dims, ctypes.c_int, vp]
    so.msda_backward_zero.restype = ctypes.c_int
    so.msda_backward_finish.argtypes = [vp, ctypes.c_size_t, vp, ctypes.c_int, dims, ctypes.c_int,
                                        vp]
    so.msda_backward_finish.restype = ctypes.c_int
    so.msda_backward_static_workspace.argtypes = [vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, dims,
                                                  ctypes.c_int, vp]
    so.msda_backward_static_workspace.restype = ctypes.c_int
    so.msda_debug_corners.argtypes = [vp, vp, vp, vp, dims, ctypes.c_int, vp]
    so.msda_debug_corners.restype = ctypes.c_int
    so.msda_checked_build.argtypes = []
    so.msda_checked_build.restype = ctypes.c_int
    so.msda_device_check.argtypes = [vp]
    so.msda_device_check.restype = ctypes.c_int
    so.msda_debug_bounds_self_test.argtypes = [vp]
    so.msda_debug_bounds_self_test.restype = ctypes.c_int
    so.msda_set_sample_split.argtypes = [ctypes.c_int]
    so.msda_set_sample_split.restype = ctypes.c_int
    so.msda_status_string.argtypes = [ctypes.c_int]
    so.msda_status_string.restype = ctypes.c_char_p
    so.msda_version.argtypes = []
    so.msda_version.restype = ctypes.c_int
    return so


def use_library(path: str | None = None):
    """Make every call of this module go to the library at `path` (default:
    libmsda.so), e.g. the range-checked build at build.CHECKED_LIBRARY;
    returns its handle."""
    global _lib
    with _lock:
        _lib = load(path)
    return _lib


def lib():
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                _lib = load()
    return _lib


# ------------------------------------------------------------- marshalling

def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(*tensors):
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libmsda runs on CUDA tensors only (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("libmsda needs contiguous tensors")


def dims_of(value, spatial_shapes, sampling_locations) -> msda_dims_t:
    B, S, M, D = value.shape
    _, Q, M2, L, K, two = sampling_locations.shape
    if M2 != M or two != 2 or tuple(spatial_shapes.shape) != (L, 2):
        raise ValueError("inconsistent operand shapes")
    return msda_dims_t(B, S, Q, M, D, L, K)


def _dtype(t) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _call(name, status):
    if status != 0:
        raise MSDAError(status, name)


def msda_forward(value, spatial_shapes, level_start_index, sampling_locations,
                 attention_weights, query_order=None, out=None, stream=None, softmax=False):
    """out (B, Q, M*D) of value's dtype; see msda_forward in include/msda.h.
    softmax=True: attention_weights are logits (msda_forward_softmax)."""
    d = dims_of(value, spatial_shapes, sampling_locations)
    if out is None:
        out = torch.empty((d.B, d.Q, d.M * d.D), dtype=value.dtype, device=value.device)
    _check_cuda(value, spatial_shapes, level_start_index, sampling_locations,
                attention_weights, query_order, out)
    name = "msda_forward_softmax" if softmax else "msda_forward"
    _call(name, getattr(lib(), name)(
        _ptr(value), _ptr(spatial_shapes), _ptr(level_start_index), _ptr(sampling_locations),
        _ptr(attention_weights), _ptr(query_order), _ptr(out), ctypes.byref(d), _dtype(value),
        _stream(stream)))
    return out


def msda_backward_workspace_bytes(dims: msda_dims_t, dtype, accum: int) -> int:
    dt = dtype if isinstance(dtype, int) else _DTYPES[dtype]
    return int(lib().msda_backward_workspace_bytes(ctypes.byref(dims), dt, accum))


def msda_backward(value, spatial_shapes, level_start_index, sampling_locations,
                  attention_weights, grad_out, accum: int = MSDA_ACC_FP32_BUFFER,
                  query_order=None, grad_value=None, grad_sampling_locations=None,
                  grad_attention_weights=None, workspace=None, stream=None, softmax=False):
    """(grad_value, grad_sampling_locations, grad_attention_weights); with
    softmax=True the weights are logits and the third output is their
    gradient (msda_backward_softmax)."""
    d = dims_of(value, spatial_shapes, sampling_locations)
    dev, dt = value.device, value.dtype
    if grad_value is None:
        grad_value = torch.empty_like(value)
    if grad_sampling_locations is None:
        grad_sampling_locations = torch.empty_like(sampling_locations)
    if grad_attention_weights is None:
        grad_attention_weights = torch.empty_like(attention_weights)
    need = msda_backward_workspace_bytes(d, dt, accum)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check_cuda(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                grad_out, query_order, grad_value, grad_sampling_locations,
                grad_attention_weights, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    name = "msda_backward_softmax" if softmax else "msda_backward"
    _call(name, getattr(lib(), name)(
        _ptr(value), _ptr(spatial_shapes), _ptr(level_start_index), _ptr(sampling_locations),
        _ptr(attention_weights), _ptr(query_order), _ptr(grad_out), _ptr(grad_value),
        _ptr(grad_sampling_locations), _ptr(grad_attention_weights), _ptr(workspace),
        ctypes.c_size_t(ws_bytes), accum, ctypes.byref(d), _dtype(value), _stream(stream)))
    return grad_value, grad_sampling_locations, grad_attention_weights


class BackwardBuffers:
    """Outputs and workspace of one backward shape, allocated once and reused
    (the benchmark and the split-step API use this to avoid per-call allocation)."""

    def __init__(self, value, sampling_locations, attention_weights, accum=MSDA_ACC_FP32_BUFFER):
        self.dims = msda_dims_t(*[int(v) for v in value.shape[:2]], int(sampling_locations.shape[1]),
                                *[int(v) for v in value.shape[2:]],
                                *[int(v) for v in sampling_locations.shape[3:5]])
        self.accum = accum
        self.grad_value = torch.empty_like(value)
        self.grad_sampling_locations = torch.empty_like(sampling_locations)
        self.grad_attention_weights = torch.empty_like(attention_weights)
        need = msda_backward_workspace_bytes(self.dims, value.dtype, accum)
        self.workspace = (torch.empty(need, dtype=torch.uint8, device=value.device)
                          if need > 0 else None)
        self.workspace_bytes = need


def msda_backward_zero(buf: BackwardBuffers, dtype, stream=None):
    _call("msda_backward_zero", lib().msda_backward_zero(
        _ptr(buf.grad_value), _ptr(buf.workspace), ctypes.c_size_t(buf.workspace_bytes),
        buf.accum, ctypes.byref(buf.dims), _DTYPES[dtype], _stream(stream)))


def msda_backward_accumulate(value, spatial_shapes, level_start_index, sampling_locations,
                             attention_weights, grad_out, buf: BackwardBuffers,
                             query_order=None, stream=None):
    _check_cuda(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                grad_out, query_order)
    _call("msda_backward_accumulate", lib().msda_backward_accumulate(
        _ptr(value), _ptr(spatial_shapes), _ptr(level_start_index), _ptr(sampling_locations),
        _ptr(attention_weights), _ptr(query_order), _ptr(grad_out), _ptr(buf.grad_value),
        _ptr(buf.grad_sampling_locations), _ptr(buf.grad_attention_weights),
        _ptr(buf.workspace), ctypes.c_size_t(buf.workspace_bytes), buf.accum,
        ctypes.byref(buf.dims), _dtype(value), _stream(stream)))


def msda_backward_finish(buf: BackwardBuffers, dtype, stream=None):
    _call("msda_backward_finish", lib().msda_backward_finish(
        _ptr(buf.workspace), ctypes.c_size_t(buf.workspace_bytes), _ptr(buf.grad_value),
        buf.accum, ctypes.byref(buf.dims), _DTYPES[dtype], _stream(stream)))


def msda_device_check(stream=None) -> int:
    """Synchronize `stream`, then read and clear the range-fault word of the
    checked build: returns MSDA_OK (0) or MSDA_ERR_DEVICE_BOUNDS (7); always
    0 with the normal library. Raises on a CUDA failure."""
    st = int(lib().msda_device_check(_stream(stream)))
    if st not in (0, MSDA_ERR_DEVICE_BOUNDS):
        raise MSDAError(st, "msda_device_check")
    return st


def msda_set_sample_split(log2_groups: int = -1):
    """Process-wide sample split of the 16-bit and fp32 kernels: -1 (the
    default) chooses it per launch from the problem size, 0..3 force 2^s lane
    groups per query-head (clamped per launch). For tests and tuning."""
    _call("msda_set_sample_split", lib().msda_set_sample_split(int(log2_groups)))


def msda_debug_bounds_self_test(stream=None):
    """Enqueue one range check that must fail (no memory access): the next
    msda_device_check of the checked build returns MSDA_ERR_DEVICE_BOUNDS."""
    _call("msda_debug_bounds_self_test", lib().msda_debug_bounds_self_test(_stream(stream)))


def msda_debug_corners(spatial_shapes, level_start_index, sampling_locations, S: int,
                       stream=None):
    """int32 (B,Q,M,L,K,4) corner rows, -1 outside the map."""
    B, Q, M, L, K, _ = sampling_locations.shape
    d = msda_dims_t(B, S, Q, M, 8, L, K)
    rows = torch.empty((B, Q, M, L, K, 4), dtype=torch.int32, device=sampling_locations.device)
    _check_cuda(spatial_shapes, level_start_index, sampling_locations, rows)
    _call("msda_debug_corners", lib().msda_debug_corners(
        _ptr(spatial_shapes), _ptr(level_start_index), _ptr(sampling_locations), _ptr(rows),
        ctypes.byref(d), _dtype(sampling_locations), _stream(stream)))
    return rows


class MSDAFunction(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run libmsda kernels.
    With softmax=True the weights are logits (the fused-softmax variant)."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, sampling_locations,
                attention_weights, accum=MSDA_ACC_FP32_BUFFER, softmax=False):
        ctx.save_for_backward(value, spatial_shapes, level_start_index, sampling_locations,
                              attention_weights)
        ctx.accum = accum
        ctx.softmax = softmax
        return msda_forward(value, spatial_shapes, level_start_index, sampling_locations,
                            attention_weights, softmax=softmax)

    @staticmethod
    def backward(ctx, grad_out):
        value, shapes, starts, loc, attn = ctx.saved_tensors
        gv, gl, ga = msda_backward(value, shapes, starts, loc, attn, grad_out.contiguous(),
                                   accum=ctx.accum, softmax=ctx.softmax)
        return gv, None, None, gl, ga, None, None


def multi_scale_deformable_attention(value, spatial_shapes, level_start_index,
                                     sampling_locations, attention_weights,
                                     accum=MSDA_ACC_FP32_BUFFER, softmax=False):
    """Differentiable MSDA: value (B,S,M,D), locations (B,Q,M,L,K,2), weights
    (B,Q,M,L,K) or (B,Q,M,L*K) -> (B,Q,M*D). softmax=True: the weights are
    logits normalised over L*K inside the kernels."""
    B, Q, M, L, K, _ = sampling_locations.shape
    attn = attention_weights.reshape(B, Q, M, L, K).contiguous()
    return MSDAFunction.apply(value.contiguous(), spatial_shapes, level_start_index,
                              sampling_locations.contiguous(), attn, accum, softmax)
