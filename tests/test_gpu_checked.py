"""The range-checked build (libmsda_checked.so) on the GPU.

Every global access of every kernel is checked against its tensor's extent
in that build (a skipped access sets a device word, nothing traps). These
tests run the parity workloads through it, at small and full sizes, and
require both oracle parity and a clean fault word; the self-test proves the
word and its readback work, with a check that fails on purpose without
touching memory.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_msda_gb300 import binding, build, workloads as wl
from test_gpu_parity import (FP32BUF, NATIVE, _small, check, gpu_run, np64, oracle_run, to_dev,
                             upload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()
    so = binding.use_library(build.CHECKED_LIBRARY)
    assert so.msda_checked_build() == 1
    yield so
    binding.use_library()          # back to libmsda.so for the other test files


def clean():
    return binding.msda_device_check() == 0


def test_self_test_sets_and_clears_the_fault_word():
    assert clean()
    binding.msda_debug_bounds_self_test()
    assert binding.msda_device_check() == binding.MSDA_ERR_DEVICE_BOUNDS
    assert clean()                 # read and cleared


@pytest.mark.parametrize("w,accum", [(wl.tiny(), FP32BUF), (wl.decoder("bf16"), FP32BUF),
                                     (wl.decoder("bf16"), NATIVE), (wl.decoder("f16"), FP32BUF),
                                     (wl.decoder("bf16"), binding.MSDA_ACC_AUTO),
                                     (wl.decoder("f64"), FP32BUF), (wl.sweep(5000, 4, 4), FP32BUF),
                                     (wl.encoder("bf16"), FP32BUF)],
                         ids=lambda x: getattr(x, "name", str(x)))
def test_workloads_stay_in_bounds(w, accum):
    p = wl.make_inputs(w)
    got = gpu_run(p, w.dtype, accum)
    assert clean()
    check(got, oracle_run(p), w.dtype, f"checked {w.name}")


@pytest.mark.parametrize("dtype,D", [("f32", 4), ("bf16", 8), ("bf16", 256), ("f64", 2),
                                     ("f16", 32)])
def test_edge_shapes_stay_in_bounds(dtype, D):
    w = _small(Q=37, M=3, D=D, dtype=dtype)
    p = wl.make_inputs(w)
    perm = np.random.default_rng(D).permutation(w.Q).astype(np.int32)
    got = gpu_run(p, w.dtype, FP32BUF, order=perm)
    assert clean()
    check(got, oracle_run(p), w.dtype, f"checked D={D}")


def test_softmax_and_corners_stay_in_bounds():
    w = wl.decoder("bf16")
    p = wl.make_inputs(w)
    t = upload(p, w.dtype)
    z = to_dev(p["logits"], w.dtype)
    out = binding.msda_forward(t["value"], t["shapes"], t["starts"], t["loc"], z, softmax=True)
    gv, gl, gz = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"], z,
                                       t["grad_out"], softmax=True)
    rows = binding.msda_debug_corners(t["shapes"], t["starts"], t["loc"], w.S)
    assert clean()
    ref = {"out": oracle.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                         p["logits"])}
    ref["gv"], ref["gl"], ref["ga"] = oracle.backward_softmax(
        p["value"], p["shapes"], p["starts"], p["loc"], p["logits"], p["grad_out"])
    got = {"out": np64(out), "gv": np64(gv), "gl": np64(gl), "ga": np64(gz)}
    check(got, ref, w.dtype, "checked softmax")
    assert np.array_equal(rows.cpu().numpy(), oracle.corners(p["shapes"], p["starts"], p["loc"]))
