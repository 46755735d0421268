"""msda_backward_static_workspace: the backward for callers that cannot
allocate device memory at call time (an engine plugin with no scratch from its
host, or an application that allows no allocation after start-up). It must
give what msda_backward gives with a caller-allocated fp32 workspace.

This file is named to be collected last, so a failure here leaves every other
test already run. It passes alone in a fresh process and after the others:
the library's array keeps the previous call's contents, and each call must
clear what it uses."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from scale_deformable_attention_msda_gb300 import binding, workloads as wl  # noqa: E402

TD = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
MSDA_ERR_WORKSPACE = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _up(a, dt):
    return torch.tensor(a, dtype=torch.float64).to(TD[dt]).cuda()


def _static_call(t, dims, dt):
    gv = torch.full_like(t["value"], float("nan"))        # proves every element is written
    gl = torch.full_like(t["loc"], float("nan"))
    ga = torch.full_like(t["attn"], float("nan"))
    p = lambda x: ctypes.c_void_p(x.data_ptr())            # noqa: E731
    st = binding.lib().msda_backward_static_workspace(
        p(t["value"]), p(t["shapes"]), p(t["starts"]), p(t["loc"]), p(t["attn"]),
        ctypes.c_void_p(0), p(t["grad_out"]), p(gv), p(gl), p(ga), ctypes.byref(dims),
        binding._DTYPES[t["value"].dtype], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.STATUS.get(st, st)
    return gv, gl, ga


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("w,tol", [(wl.encoder("bf16"), 2e-2), (wl.decoder("bf16"), 2e-2),
                                   (wl.decoder("f16"), 2e-2), (wl.decoder("f32"), 1e-4)],
                         ids=lambda x: getattr(x, "name", "") + "-" + getattr(x, "dtype", ""))
def test_matches_msda_backward_on_two_calls_in_a_row(w, tol):
    p = wl.make_inputs(w)
    t = {k: _up(p[k], w.dtype) for k in ("value", "loc", "attn", "grad_out")}
    t["shapes"] = torch.tensor(p["shapes"]).cuda()
    t["starts"] = torch.tensor(p["starts"]).cuda()
    dims = binding.dims_of(t["value"], t["shapes"], t["loc"])
    ref = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"],
                                t["grad_out"], accum=binding.MSDA_ACC_FP32_BUFFER)
    for _ in range(2):                                     # the second call sees stale contents
        got = _static_call(t, dims, w.dtype)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.isfinite(g).all()
            assert _rel(g, r) <= tol


@pytest.mark.parametrize("dtype,tol", [("bf16", 2e-2), ("f32", 1e-4)])
def test_matches_the_fp64_oracle_on_the_decoder(dtype, tol):
    """The allocation-free backward against the fp64 CPU oracle itself (not
    only against msda_backward), on the decoder shape, two calls in a row."""
    import oracle
    oracle.build()
    w = wl.decoder(dtype)
    p = wl.make_inputs(w)
    t = {k: _up(p[k], w.dtype) for k in ("value", "loc", "attn", "grad_out")}
    t["shapes"] = torch.tensor(p["shapes"]).cuda()
    t["starts"] = torch.tensor(p["starts"]).cuda()
    dims = binding.dims_of(t["value"], t["shapes"], t["loc"])
    ref = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                          p["grad_out"])
    for _ in range(2):
        got = _static_call(t, dims, w.dtype)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            g = g.double().cpu().numpy()
            assert np.isfinite(g).all()
            assert np.linalg.norm(g - r) / np.linalg.norm(r) <= tol


def test_rejects_a_problem_larger_than_the_static_array():
    # bf16, B*S*M*D*4 bytes = 128 MiB > 64 MiB: refused before any launch
    dims = binding.msda_dims_t(B=4, S=32768, Q=10, M=8, D=32, L=1, K=4)
    assert 4 * 4 * 32768 * 8 * 32 > 64 << 20
    z = ctypes.c_void_p(0x10000)
    st = binding.lib().msda_backward_static_workspace(z, z, z, z, z, ctypes.c_void_p(0), z, z, z, z,
                                                      ctypes.byref(dims), binding.MSDA_BF16,
                                                      ctypes.c_void_p(0))
    assert st == MSDA_ERR_WORKSPACE
