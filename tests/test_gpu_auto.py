"""MSDA_ACC_AUTO (16-bit data) against the fp64 oracle.

AUTO is resolved on the host from the sizes: native accumulation when the
value rows receive on average at most 4 corner adds per head (4 Q K L <= 4 S),
the fp32 workspace otherwise. Bars: relative L2 <= 2e-2 for every gradient, as
for the other 16-bit modes. The decoder shape (0.9 adds per row), the tiny
case and the one-level sweep point resolve to native; the encoder, Mask2Former
and the other sweep points (contention included) to the fp32 workspace, whose
result AUTO must then reproduce.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_msda_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu
AUTO, FP32BUF = binding.MSDA_ACC_AUTO, binding.MSDA_ACC_FP32_BUFFER
TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()


def _up(a, dt):
    return torch.tensor(a, dtype=torch.float64).to(TD[dt]).cuda()


def _rel(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def _gpu(w, p, accum, softmax=False):
    t = {k: _up(p[k], w.dtype) for k in ("value", "loc", "attn", "logits", "grad_out")}
    shapes = torch.tensor(p["shapes"]).cuda()
    starts = torch.tensor(p["starts"]).cuda()
    a = t["logits"] if softmax else t["attn"]
    gv = torch.full_like(t["value"], float("nan"))      # every element must be written
    gl = torch.full_like(t["loc"], float("nan"))
    ga = torch.full_like(a, float("nan"))
    binding.msda_backward(t["value"], shapes, starts, t["loc"], a, t["grad_out"], accum=accum,
                          grad_value=gv, grad_sampling_locations=gl, grad_attention_weights=ga,
                          softmax=softmax)
    torch.cuda.synchronize()
    assert binding.msda_device_check() == 0
    got = [x.double().cpu().numpy() for x in (gv, gl, ga)]
    for g in got:
        assert np.isfinite(g).all()
    return got


def _run(w, softmax=False):
    p = wl.make_inputs(w)
    got = _gpu(w, p, AUTO, softmax)
    if softmax:
        ref = oracle.backward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                      p["logits"], p["grad_out"])
    else:
        ref = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                              p["grad_out"])
    errs = {k: _rel(g, r) for k, g, r in zip(("gv", "gl", "ga"), got, ref)}
    print(w.name, w.dtype, "auto", "softmax" if softmax else "",
          {k: f"{v:.2e}" for k, v in errs.items()})
    return p, got, errs


@pytest.mark.parametrize("w", [wl.tiny().with_dtype("bf16"), wl.decoder("bf16"), wl.decoder("f16"),
                               wl.encoder("bf16"), wl.mask2former("bf16"), wl.mask2former("f16"),
                               wl.sweep(5000, 2, 1), wl.sweep(10000, 8, 3), wl.sweep(22223, 4, 4),
                               wl.sweep(5000, 4, 4, contention=True)],
                         ids=lambda w: f"{w.name}-{w.dtype}")
def test_auto_matches_the_oracle(w):
    _, _, errs = _run(w)
    assert max(errs.values()) <= 2e-2, errs


@pytest.mark.parametrize("w", [wl.decoder("bf16"), wl.encoder("bf16")], ids=lambda w: w.name)
def test_auto_softmax_variant(w):
    _, _, errs = _run(w, softmax=True)
    assert max(errs.values()) <= 2e-2, errs


@pytest.mark.parametrize("split", [0, 1, 2, 3])
def test_auto_with_every_sample_split(split):
    binding.msda_set_sample_split(split)
    try:
        _, _, errs = _run(wl.decoder("bf16"))
    finally:
        binding.msda_set_sample_split(-1)
    assert max(errs.values()) <= 2e-2, errs


def test_auto_on_a_contended_shape_is_the_fp32_buffer():
    """The encoder has contended levels: AUTO accumulates in fp32, so its
    grad_value equals MSDA_ACC_FP32_BUFFER's up to the atomics' order (a few
    16-bit rounding flips), far closer than native accumulation would be."""
    w = wl.encoder("bf16")
    p, got, _ = _run(w)
    buf = _gpu(w, p, FP32BUF)
    assert _rel(got[0], buf[0]) <= 2e-3
    for a, b in zip(got[1:], buf[1:]):
        assert np.array_equal(a, b)            # grad_loc and grad_attn are deterministic


def test_auto_fp32_data_is_plain_accumulation():
    """For fp32 data the mode changes nothing: fp32 atomics into grad_value."""
    _, _, errs = _run(wl.decoder("f32"))
    assert max(errs.values()) <= 1e-4, errs
