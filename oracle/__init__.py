"""fp64 CPU oracle for multi-scale deformable attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The CUDA
library never calls it and shares no code with it; it is the independent
definition the CUDA path is checked against.

The arithmetic lives in ``msda_oracle.c`` (plain C, fp64, OpenMP over
independent output rows); this module compiles it with the host C compiler and
marshals numpy arrays to it. Every input is upcast to float64 exactly, so a
bf16 or fp32 run of the CUDA path is checked against the oracle on the very
values the kernel saw.

Sources: msda-triton course, ch. 1 "Deformable attention, from scratch"
(sections "The equation, term by term", "Bilinear interpolation", "The simplest
possible implementation") for the forward and the integer parts; the course
index, chapter 5 "The backward kernel", names the three gradients, which the C
file derives by the chain rule.

Parity status: forward, backward and corner indices are all pinned by
``tests/test_oracle_pins.py`` (page facts, grid_sample and scipy
cross-checks, finite differences, mutation checks); nothing here is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "msda_oracle.c")
LIBRARY = os.path.join(_HERE, "libmsda_oracle.so")

# Plain IEEE arithmetic: no fused multiply-add contraction and no fast-math, so
# every product and sum is the one written in the C source, on x86 and Arm.
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def compile_library(source: str = SOURCE, output: str = LIBRARY,
                    extra_flags=()) -> str:
    """Compile an oracle source file into a shared library; returns its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def build(force: bool = False) -> str:
    """Compile ``msda_oracle.c`` if the library is missing or older than it."""
    with _lock:
        if (force or not os.path.exists(LIBRARY)
                or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
            compile_library()
    return LIBRARY


def _declare(lib):
    i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.msda_oracle_forward.argtypes = [dp] * 6 + [i64] * 7 + [ip]
    lib.msda_oracle_forward.restype = ctypes.c_int
    lib.msda_oracle_backward.argtypes = [dp] * 9 + [i64] * 7 + [ip]
    lib.msda_oracle_backward.restype = ctypes.c_int
    lib.msda_oracle_corners.argtypes = [dp] * 3 + [i64] * 3 + [dp]
    lib.msda_oracle_corners.restype = ctypes.c_int
    return lib


def load_library(path: str):
    """Load an oracle shared library (the built one, or a test's variant)."""
    return _declare(ctypes.CDLL(path))


def _library():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dims(value, shapes, loc):
    B, S, M, D = value.shape
    _, Q, M2, L, K, two = loc.shape
    if M2 != M or two != 2 or shapes.shape != (L, 2):
        raise ValueError("inconsistent operand shapes")
    return B, S, Q, M, D, L, K


def forward(value, spatial_shapes, level_start_index, sampling_locations,
            attention_weights, nthreads: int = 0, lib=None):
    """out (B, Q, M*D) float64. Argument layouts as in the C file."""
    lib = lib or _library()
    value, loc, attn = _f64(value), _f64(sampling_locations), _f64(attention_weights)
    shapes, starts = _i64(spatial_shapes), _i64(level_start_index)
    B, S, Q, M, D, L, K = _dims(value, shapes, loc)
    attn = attn.reshape(B, Q, M, L, K)
    out = np.empty((B, Q, M * D), dtype=np.float64)
    rc = lib.msda_oracle_forward(_ptr(value), _ptr(shapes), _ptr(starts), _ptr(loc),
                                 _ptr(attn), _ptr(out), B, S, Q, M, D, L, K, nthreads)
    if rc != 0:
        raise ValueError("oracle forward rejected its arguments")
    return out


def backward(value, spatial_shapes, level_start_index, sampling_locations,
             attention_weights, grad_out, nthreads: int = 0, lib=None):
    """(grad_value (B,S,M,D), grad_loc (B,Q,M,L,K,2), grad_attn (B,Q,M,L,K)), float64."""
    lib = lib or _library()
    value, loc, attn = _f64(value), _f64(sampling_locations), _f64(attention_weights)
    shapes, starts = _i64(spatial_shapes), _i64(level_start_index)
    B, S, Q, M, D, L, K = _dims(value, shapes, loc)
    attn = attn.reshape(B, Q, M, L, K)
    g = _f64(grad_out).reshape(B, Q, M * D)
    gv = np.empty_like(value)
    gl = np.empty_like(loc)
    ga = np.empty_like(attn)
    rc = lib.msda_oracle_backward(_ptr(value), _ptr(shapes), _ptr(starts), _ptr(loc),
                                  _ptr(attn), _ptr(g), _ptr(gv), _ptr(gl), _ptr(ga),
                                  B, S, Q, M, D, L, K, nthreads)
    if rc != 0:
        raise ValueError("oracle backward rejected its arguments")
    return gv, gl, ga


def corners(spatial_shapes, level_start_index, sampling_locations, lib=None):
    """int32 (B,Q,M,L,K,4): value row of each corner inside the map, -1 outside."""
    lib = lib or _library()
    loc = _f64(sampling_locations)
    shapes, starts = _i64(spatial_shapes), _i64(level_start_index)
    *lead, L, K, two = loc.shape
    BQM = int(np.prod(lead)) if lead else 1
    idx = np.empty(tuple(lead) + (L, K, 4), dtype=np.int32)
    rc = lib.msda_oracle_corners(_ptr(shapes), _ptr(starts), _ptr(loc), BQM, L, K, _ptr(idx))
    if rc != 0:
        raise ValueError("oracle corners rejected its arguments")
    return idx


# --------------------------------------------------------------------------
# The softmax variant (deformops README, "Multi-scale deformable attention":
# with the softmax method the kernel normalises raw logits jointly over the
# levels and points of each (b, q, m)). Composition of a softmax over the L*K
# logits with the operator above; the backward is the chain rule through the
# softmax: d loss / d z_i = a_i (g_i - sum_j a_j g_j) with g = d loss / d a.

def softmax_weights(logits):
    """a (B,Q,M,L,K) = softmax of the logits over their last two axes jointly."""
    z = _f64(logits)
    lead = z.shape[:-2]
    flat = z.reshape(lead + (-1,))
    e = np.exp(flat - flat.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).reshape(z.shape)


def forward_softmax(value, spatial_shapes, level_start_index, sampling_locations,
                    attention_logits, nthreads: int = 0, lib=None):
    return forward(value, spatial_shapes, level_start_index, sampling_locations,
                   softmax_weights(attention_logits), nthreads=nthreads, lib=lib)


def backward_softmax(value, spatial_shapes, level_start_index, sampling_locations,
                     attention_logits, grad_out, nthreads: int = 0, lib=None):
    """(grad_value, grad_loc, grad_logits), float64."""
    a = softmax_weights(attention_logits)
    gv, gl, ga = backward(value, spatial_shapes, level_start_index, sampling_locations, a,
                          grad_out, nthreads=nthreads, lib=lib)
    lead = a.shape[:-2]
    af, gf = a.reshape(lead + (-1,)), ga.reshape(lead + (-1,))
    gz = af * (gf - np.sum(af * gf, axis=-1, keepdims=True))
    return gv, gl, gz.reshape(a.shape)
