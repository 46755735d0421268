"""Randomised parity of the CUDA path with the fp64 oracle.

Seeded draws over what the hand-written cases fix one at a time: batch,
query and head counts (ragged against the warp's groups), channel widths
(1 to 32 lanes per query-head), level sets of random sizes (1x1 to 40x40,
one to five levels), point counts, offset spreads from sub-pixel to far off
the map, dtypes, the accumulator, the fused softmax and the sample split.
Every case meets the tolerances of test_gpu_parity.py and records no range
fault. The draw depends only on the seed, so a failing case can be re-run
alone by its id.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_msda_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CHANNELS = {"f32": (4, 8, 16, 32, 64, 128), "bf16": (8, 16, 32, 64, 256), "f16": (8, 32, 64)}
N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()
    yield
    binding.msda_set_sample_split(-1)


def draw(seed):
    """One case: (workload, accumulator, softmax, split)."""
    rng = np.random.default_rng(1000 + seed)
    dtype = ("f32", "bf16", "f16")[rng.integers(3)]
    L = int(rng.integers(1, 6))
    levels = tuple((int(rng.integers(1, 41)), int(rng.integers(1, 41))) for _ in range(L))
    K = int(rng.integers(1, 10))
    w = wl.Workload(f"random{seed}", B=int(rng.integers(1, 4)), Q=int(rng.integers(1, 301)),
                    M=int(rng.integers(1, 10)), D=int(rng.choice(CHANNELS[dtype])), K=K,
                    levels=levels, dtype=dtype,
                    sigma_px=float(rng.choice([0.3, 1.0, 2.0, 6.0, 20.0])), seed=seed)
    # native 16-bit adds round at every add; the fp32 buffer is the mode at
    # parity, and the scaled fp16 buffer (native adds for fp16 data) is held to
    # the same tolerance. Drawn from a stream of its own, so that the shapes of
    # each seed stay as they were.
    accum = (binding.MSDA_ACC_FP32_BUFFER, binding.MSDA_ACC_FP16_BUFFER)[
        np.random.default_rng(5000 + seed).integers(2)]
    # the fused softmax keeps a query-head's L*K weights in 16 slots per 16-byte lane
    lanes16 = w.D * (4 if dtype == "f32" else 2) // 16
    softmax = bool(rng.integers(2)) and L * K <= 16 * lanes16
    split = int(rng.choice([-1, -1, 0, 1, 2, 3]))
    return w, accum, softmax, split


def rel_l2(got, ref):
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    run_case(seed)


@pytest.mark.parametrize("seed", range(0, N_CASES, 4))
def test_random_case_range_checked(seed):
    """Every fourth draw again through libmsda_checked.so, where any kernel
    access outside its tensor would set the fault word."""
    from scale_deformable_attention_msda_gb300 import build
    binding.use_library(build.CHECKED_LIBRARY)
    try:
        run_case(seed)
    finally:
        binding.use_library(build.LIBRARY)


def run_case(seed):
    w, accum, softmax, split = draw(seed)
    p = wl.make_inputs(w)
    dt, dev = TORCH_DTYPE[w.dtype], torch.device("cuda:0")
    up = lambda a: torch.tensor(a, dtype=torch.float64).to(dt).to(dev)
    v, loc, g = up(p["value"]), up(p["loc"]), up(p["grad_out"])
    a = up(p["logits"] if softmax else p["attn"])
    shapes = torch.tensor(p["shapes"], dtype=torch.int64, device=dev)
    starts = torch.tensor(p["starts"], dtype=torch.int64, device=dev)
    binding.msda_set_sample_split(split)
    try:
        out = binding.msda_forward(v, shapes, starts, loc, a, softmax=softmax)
        gv, gl, ga = binding.msda_backward(v, shapes, starts, loc, a, g, accum=accum,
                                           softmax=softmax)
        torch.cuda.synchronize()
    finally:
        binding.msda_set_sample_split(-1)
    assert binding.msda_device_check() == 0
    got = [t.double().cpu().numpy() for t in (out, gv, gl, ga)]
    if softmax:
        ref = [oracle.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"], p["logits"]),
               *oracle.backward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                        p["logits"], p["grad_out"])]
    else:
        ref = [oracle.forward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"]),
               *oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                                p["grad_out"])]
    label = (w.name, w.dtype, w.B, w.Q, w.M, w.D, w.K, w.levels, w.sigma_px, softmax, split, accum)
    if w.dtype == "f32":
        scale = max(float(np.max(np.abs(ref[0]))), 1e-300)
        assert np.max(np.abs(got[0] - ref[0])) / scale <= 1e-5, label
        for k in (1, 2, 3):
            assert rel_l2(got[k], ref[k]) <= 1e-4, (label, k)
    else:
        for k in range(4):
            assert rel_l2(got[k], ref[k]) <= 2e-2, (label, k)
