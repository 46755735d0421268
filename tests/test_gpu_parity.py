"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances:
  fp32 forward      max |gpu - oracle| <= 1e-5 * max |oracle|
  fp32 backward     relative L2 error <= 1e-4 for each gradient
  bf16 / fp16       relative L2 error <= 2e-2 (forward and backward)
  fp64              forward max error <= 1e-12 * max |oracle|, gradients
                    relative L2 <= 1e-12 (only the summation order differs)
  integer parts     bit-exact (corner rows and in-map masks)
The oracle receives exactly the values the GPU saw (16-bit inputs upcast).
Every workload runs at its full size; the oracle finishes each in seconds.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_msda_gb300 import binding, workloads as wl

pytestmark = pytest.mark.gpu

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16,
               "f64": torch.float64}
NATIVE, FP32BUF = binding.MSDA_ACC_NATIVE, binding.MSDA_ACC_FP32_BUFFER


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()


def dev():
    return torch.device("cuda:0")


def to_dev(a, dtype):
    return torch.tensor(a, dtype=torch.float64).to(TORCH_DTYPE[dtype]).to(dev())


def np64(t):
    return t.detach().double().cpu().numpy()


def rel_l2(got, ref):
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def upload(p, dtype):
    t = {k: to_dev(p[k], dtype) for k in ("value", "loc", "attn", "grad_out") if k in p}
    t["shapes"] = torch.tensor(p["shapes"], dtype=torch.int64, device=dev())
    t["starts"] = torch.tensor(p["starts"], dtype=torch.int64, device=dev())
    return t


def gpu_run(p, dtype, accum=FP32BUF, order=None, backward=True):
    t = upload(p, dtype)
    o = None if order is None else torch.tensor(order, dtype=torch.int32, device=dev())
    out = binding.msda_forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"],
                               query_order=o)
    res = {"out": out}
    if backward:
        gv, gl, ga = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"],
                                           t["attn"], t["grad_out"], accum=accum, query_order=o)
        res.update(gv=gv, gl=gl, ga=ga)
    torch.cuda.synchronize()
    return {k: np64(v) for k, v in res.items()}


def oracle_run(p, backward=True):
    r = {"out": oracle.forward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"])}
    if backward:
        r["gv"], r["gl"], r["ga"] = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"],
                                                    p["attn"], p["grad_out"])
    return r


def check(got, ref, dtype, label=""):
    errs = {}
    if dtype in ("f32", "f64"):
        tol_out, tol_grad = (1e-5, 1e-4) if dtype == "f32" else (1e-12, 1e-12)
        scale = max(np.max(np.abs(ref["out"])), 1e-300)
        errs["out"] = float(np.max(np.abs(got["out"] - ref["out"])) / scale)
        assert errs["out"] <= tol_out, (label, errs)
        for k in ("gv", "gl", "ga"):
            if k in got:
                errs[k] = rel_l2(got[k], ref[k])
                assert errs[k] <= tol_grad, (label, k, errs)
    else:
        for k in ("out", "gv", "gl", "ga"):
            if k in got:
                errs[k] = rel_l2(got[k], ref[k])
                assert errs[k] <= 2e-2, (label, k, errs)
    print(label, dtype, {k: f"{v:.2e}" for k, v in errs.items()})
    return errs


def run_and_check(w, accum=FP32BUF, order=None, label=None):
    p = wl.make_inputs(w)
    got = gpu_run(p, w.dtype, accum, order)
    assert binding.msda_device_check() == 0      # no fault recorded by any kernel
    ref = oracle_run(p)
    return check(got, ref, w.dtype, label or w.name)


# ------------------------------------------------------------ workloads

def test_tiny_f32():
    run_and_check(wl.tiny())


@pytest.mark.parametrize("dtype,accum", [("f32", FP32BUF), ("bf16", FP32BUF), ("bf16", NATIVE),
                                         ("f16", FP32BUF), ("f16", NATIVE)])
def test_decoder(dtype, accum):
    run_and_check(wl.decoder(dtype), accum)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_encoder(dtype):
    run_and_check(wl.encoder(dtype), FP32BUF)


@pytest.mark.parametrize("dtype,accum", [("bf16", FP32BUF), ("bf16", NATIVE), ("f32", FP32BUF)])
def test_mask2former(dtype, accum):
    run_and_check(wl.mask2former(dtype), accum)


# Native 16-bit accumulation rounds grad_value to bf16 at every atomic add, so
# its error grows with the number of contributions per element. It meets the
# 2e-2 bar on the decoder and Mask2Former workloads (checked above); on the
# encoder (about 1300 contributions per level-3 pixel and head) it sits at the
# bar (measured 1.9e-2, with atomics in nondeterministic order) and under the
# 4x4-patch contention workload it misses it (5.5e-2); the fp32 buffer is the
# mode that holds parity there. These measured bounds guard against regressions
# of the native path; every other output must still meet the bar.
NATIVE_GRAD_VALUE_BOUND = {"encoder": 3e-2, "sweep_Q5000_K4_L4_contention": 8e-2}


@pytest.mark.parametrize("w", [wl.encoder("bf16"), wl.sweep(5000, 4, 4, contention=True)],
                         ids=lambda w: w.name)
def test_native_bf16_accumulation_characterised(w):
    p = wl.make_inputs(w)
    got = gpu_run(p, w.dtype, NATIVE)
    ref = oracle_run(p)
    err = {k: rel_l2(got[k], ref[k]) for k in ("out", "gv", "gl", "ga")}
    print(w.name, "native", {k: f"{v:.2e}" for k, v in err.items()})
    assert max(err["out"], err["gl"], err["ga"]) <= 2e-2, err
    assert err["gv"] <= NATIVE_GRAD_VALUE_BOUND[w.name], err


@pytest.mark.parametrize("Q,K,L", [(5000, 2, 1), (10000, 8, 3), (22223, 4, 4), (5000, 8, 2)])
def test_sweep_points(Q, K, L):
    run_and_check(wl.sweep(Q, K, L), FP32BUF)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_shape_example_of_the_pages(dtype):
    """The operand shapes the deformops README prints for its backend example:
    value (1, 80, 4, 8) over levels (8, 8) and (4, 4), starts [0, 64]; here
    with 10 queries and 4 points. D = 8 gives one or two lanes per
    query-head. Plain and softmax variants; for 16-bit data both buffers."""
    w = wl.Workload("readme_example", B=1, Q=10, M=4, D=8, K=4, levels=((8, 8), (4, 4)),
                    dtype=dtype, sigma_px=1.5, ref="uniform", seed=4242)
    p = wl.make_inputs(w)
    assert list(p["starts"]) == [0, 64] and p["value"].shape == (1, 80, 4, 8)
    ref = oracle_run(p)
    accs = [FP32BUF] if dtype == "f32" else [FP32BUF, binding.MSDA_ACC_FP16_BUFFER]
    for accum in accs:
        check(gpu_run(p, dtype, accum), ref, dtype, f"example {dtype} accum {accum}")
    _softmax_check(w, FP32BUF, f"example softmax {dtype}")


@pytest.mark.parametrize("w", list(wl.sweep_grid()), ids=lambda w: w.name)
def test_whole_ablation_grid_both_buffers(w):
    """Every point of the ablation grid the sweep times (Q x K x L, bf16):
    forward and backward with the fp32 buffer and with the scaled fp16
    buffer, against one oracle run. K = 2 and 4 with L = 1, 2 or 3 take the
    forward's 4-sample gather steps."""
    p = wl.make_inputs(w)
    ref = oracle_run(p)
    for accum, name in ((FP32BUF, "fp32 buffer"), (binding.MSDA_ACC_FP16_BUFFER, "fp16 buffer")):
        got = gpu_run(p, w.dtype, accum)
        check(got, ref, w.dtype, f"{w.name} {name}")


@pytest.mark.parametrize("w", [wl.tiny().with_dtype("f64"), wl.decoder("f64"), wl.encoder("f64")],
                         ids=lambda w: w.name)
def test_f64(w):
    run_and_check(w)


def test_sweep_contention():
    run_and_check(wl.sweep(5000, 4, 4, contention=True), FP32BUF)


@pytest.mark.parametrize("kind", ["morton", "hilbert"])
def test_dispatch_order_changes_nothing(kind):
    """Forward, grad_loc and grad_attn are bit-identical under any dispatch
    order (each is computed by one group); grad_value agrees within tolerance."""
    w = wl.sweep(10000, 4, 4)
    p = wl.make_inputs(w)
    lin = gpu_run(p, w.dtype)
    perm = wl.query_order(w, kind)
    assert not np.array_equal(perm, np.arange(w.Q))
    got = gpu_run(p, w.dtype, order=perm)
    for k in ("out", "gl", "ga"):
        assert np.array_equal(got[k], lin[k]), k
    check(got, oracle_run(p), w.dtype, f"order {kind}")


# ------------------------------------------------ the softmax variant

@pytest.mark.parametrize("w", [wl.tiny(), wl.decoder("f32"), wl.decoder("bf16"),
                               wl.encoder("f32"), wl.encoder("bf16"),
                               wl.sweep(5000, 8, 4), wl.decoder("f64")],
                         ids=lambda w: f"{w.name}-{w.dtype}")
def test_softmax_variant(w):
    _softmax_check(w, FP32BUF, f"softmax {w.name}")


def _softmax_check(w, accum, label):
    """The fused-softmax entry points on w's logits against the oracle's."""
    p = wl.make_inputs(w)
    t = upload(p, w.dtype)
    z = to_dev(p["logits"], w.dtype)
    out = binding.msda_forward(t["value"], t["shapes"], t["starts"], t["loc"], z, softmax=True)
    gv, gl, gz = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"], z,
                                       t["grad_out"], softmax=True, accum=accum)
    torch.cuda.synchronize()
    assert binding.msda_device_check() == 0
    got = {"out": np64(out), "gv": np64(gv), "gl": np64(gl), "ga": np64(gz)}
    ref = {"out": oracle.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                         p["logits"])}
    ref["gv"], ref["gl"], ref["ga"] = oracle.backward_softmax(
        p["value"], p["shapes"], p["starts"], p["loc"], p["logits"], p["grad_out"])
    check(got, ref, w.dtype, label)


# ------------------------------------------------------- integer parity

def _corners_case(w, loc=None):
    p = wl.make_inputs(w, with_grad=False)
    if loc is not None:
        p["loc"] = loc
    t = upload(p, w.dtype)
    rows = binding.msda_debug_corners(t["shapes"], t["starts"], t["loc"], w.S)
    torch.cuda.synchronize()
    ref = oracle.corners(p["shapes"], p["starts"], p["loc"])
    assert np.array_equal(rows.cpu().numpy(), ref)


@pytest.mark.parametrize("w", [wl.tiny(), wl.decoder("f32"), wl.decoder("bf16"),
                               wl.encoder("bf16"), wl.mask2former("bf16"),
                               wl.sweep(5000, 4, 4, contention=True), wl.decoder("f64")],
                         ids=lambda w: f"{w.name}-{w.dtype}")
def test_corner_rows_bit_exact(w):
    _corners_case(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "f64"])
def test_corner_rows_at_cell_boundaries(dtype):
    """Locations whose pixel coordinate is an integer or one ulp either side:
    the floor must be the exact one on both sides."""
    levels = ((100, 167), (13, 21), (1, 1), (1, 5))
    w = wl.Workload("edges", B=1, Q=64, M=2, D=8, K=8, levels=levels, dtype=dtype, seed=9)
    rng = np.random.default_rng(1)
    np_t = {"f32": np.float32, "f16": np.float16, "bf16": np.float32, "f64": np.float64}[dtype]
    loc = np.empty((1, w.Q, w.M, w.L, w.K, 2))
    for l, (h, ww) in enumerate(levels):
        for axis, n in ((0, ww), (1, h)):
            j = rng.integers(-2, n + 2, size=(w.Q, w.M, w.K))
            base = ((j + 0.5) / n).astype(np_t)
            step = rng.integers(-1, 2, size=base.shape)
            v = np.where(step > 0, np.nextafter(base, np_t(np.inf)),
                         np.where(step < 0, np.nextafter(base, np_t(-np.inf)), base))
            loc[0, :, :, l, :, axis] = v.astype(np.float64)
    loc = wl.round_to(loc, dtype)
    _corners_case(w, loc)


# ----------------------------------------------------------- edge cases

def _small(B=2, Q=37, M=3, D=8, K=3, levels=((9, 11), (4, 7), (1, 3)), dtype="f32", sigma=3.0,
           seed=31):
    return wl.Workload("edge", B=B, Q=Q, M=M, D=D, K=K, levels=levels, dtype=dtype,
                       sigma_px=sigma, seed=seed)


@pytest.mark.parametrize("dtype,D", [("f32", 4), ("f32", 8), ("f32", 16), ("f32", 64),
                                     ("f32", 128), ("bf16", 8), ("bf16", 16), ("bf16", 64),
                                     ("bf16", 256), ("f16", 32), ("f64", 2), ("f64", 64)])
def test_channel_widths(dtype, D):
    run_and_check(_small(D=D, dtype=dtype, M=2), FP32BUF, label=f"D={D}")


@pytest.fixture
def sample_split(request):
    """Force the kernels' sample split (2^s lane groups per query-head) for
    one test, then restore the size-based choice."""
    binding.msda_set_sample_split(request.param)
    yield request.param
    binding.msda_set_sample_split(-1)


SPLITS = [-1, 0, 1, 3]      # automatic, off, two groups, eight groups (clamped)


@pytest.mark.parametrize("sample_split", SPLITS, indirect=True)
@pytest.mark.parametrize("Q", [1, 7, 31, 33, 129, 1001])
def test_ragged_query_counts(Q, sample_split):
    run_and_check(_small(Q=Q, B=3), label=f"Q={Q} split={sample_split}")


@pytest.mark.parametrize("sample_split", SPLITS, indirect=True)
@pytest.mark.parametrize("dtype,accum,D,K", [("f32", FP32BUF, 32, 4), ("bf16", FP32BUF, 32, 4),
                                             ("bf16", NATIVE, 32, 4), ("f16", FP32BUF, 64, 3),
                                             ("bf16", FP32BUF, 8, 5), ("f32", FP32BUF, 4, 2)])
def test_sample_split_modes(dtype, accum, D, K, sample_split):
    """Every split level on every lane mapping (16-byte and 8-byte lanes,
    native and fp32 accumulation, one to 16 lanes per query-head), with
    sample counts that do not divide the groups, plain and softmax."""
    w = _small(Q=45, M=3, D=D, K=K, dtype=dtype)
    run_and_check(w, accum, label=f"{dtype} D={D} K={K} split={sample_split}")
    p = wl.make_inputs(w)
    t = upload(p, w.dtype)
    z = to_dev(p["logits"], w.dtype)
    out = binding.msda_forward(t["value"], t["shapes"], t["starts"], t["loc"], z, softmax=True)
    gv, gl, gz = binding.msda_backward(t["value"], t["shapes"], t["starts"], t["loc"], z,
                                       t["grad_out"], softmax=True, accum=accum)
    torch.cuda.synchronize()
    got = {"out": np64(out), "gv": np64(gv), "gl": np64(gl), "ga": np64(gz)}
    ref = {"out": oracle.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                         p["logits"])}
    ref["gv"], ref["gl"], ref["ga"] = oracle.backward_softmax(
        p["value"], p["shapes"], p["starts"], p["loc"], p["logits"], p["grad_out"])
    check(got, ref, w.dtype, f"softmax {dtype} D={D} K={K} split={sample_split}")


@pytest.mark.parametrize("dtype,D,Q,M", [("f32", 32, 1, 3), ("f32", 32, 33, 5), ("bf16", 32, 7, 3),
                                         ("bf16", 32, 1001, 3), ("f16", 64, 5, 3),
                                         ("f32", 128, 9, 2), ("bf16", 128, 31, 2)])
def test_fp32_target_ragged_heads_and_orders(dtype, D, Q, M):
    """fp32 targets with 4 channels per lane (fp32 data; 16-bit data with the
    fp32 workspace on 8-byte lanes): ragged query counts, head counts that do
    not divide the warp's groups, tight offsets (many shared corners), and a
    permuted dispatch order."""
    w = _small(Q=Q, M=M, D=D, dtype=dtype, sigma=1.0)
    run_and_check(w, FP32BUF, label=f"D={D} Q={Q} M={M}")
    perm = np.random.default_rng(Q).permutation(Q).astype(np.int32)
    run_and_check(w, FP32BUF, order=perm, label=f"D={D} Q={Q} M={M} permuted")


@pytest.mark.parametrize("w", [wl.sweep(5000, 4, 4), wl.sweep(5000, 4, 4, contention=True),
                               wl.sweep(5000, 4, 4, dtype="f32")],
                         ids=lambda w: f"{w.name}-{w.dtype}")
def test_grad_value_elementwise_bound(w):
    """Every grad_value element within a bound of the sum of the magnitudes
    of its contributions, sum |a w_c g| (the oracle backward with |grad_out|):
    a dropped, duplicated or misrouted contribution breaks it in any row with
    few contributions, where a tensor-wide relative norm could miss it."""
    p = wl.make_inputs(w)
    got = gpu_run(p, w.dtype, FP32BUF)
    ref = oracle_run(p)
    mag, _, _ = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                                np.abs(p["grad_out"]))
    # fp32 sums of at most a few thousand terms, then (16-bit) one rounding
    rel = 1e-4 if w.dtype == "f32" else 2.0 ** -8 + 1e-4
    err = np.abs(got["gv"] - ref["gv"])
    bound = rel * mag + 1e-30
    worst = float(np.max(err / bound))
    assert worst <= 1.0, (w.name, w.dtype, worst)


@pytest.mark.parametrize("K,levels", [(1, ((5, 6),)), (1, ((1, 1),)), (16, ((3, 2), (1, 4))),
                                      (5, tuple((2 + l, 3 + l) for l in range(16)))])
def test_level_and_point_counts(K, levels):
    run_and_check(_small(K=K, levels=levels), label=f"K={K} L={len(levels)}")


@pytest.mark.parametrize("sample_split", [-1, 3], indirect=True)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_points_per_query_head(dtype, sample_split):
    """K = 200 over three levels: 600 samples per query-head, so every group
    walks many chunks of descriptors (and a split group takes every eighth
    sample of a long list)."""
    w = _small(B=2, Q=40, M=3, D=32, K=200, levels=((30, 40), (15, 20), (4, 5)), dtype=dtype,
               sigma=4.0)
    run_and_check(w, FP32BUF, label=f"K=200 {dtype} split={sample_split}")


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_softmax_at_slot_capacity(dtype, D):
    """The fused softmax keeps a warp's d loss / d weight in 512 shared
    slots: L*K = 16 x (16-byte lanes per query-head) fills every slot of a
    warp's query-heads (here 16 levels x 16 points)."""
    levels = tuple((2 + l % 5, 3 + l % 4) for l in range(16))
    w = _small(B=1, Q=20, M=3, D=D, K=16, levels=levels, dtype=dtype)
    assert w.L * w.K == 16 * (D * (4 if dtype == "f32" else 2) // 16)
    _softmax_check(w, FP32BUF, label=f"softmax at capacity {dtype} D={D}")


def test_empty_problems():
    w = _small(B=2, Q=0)
    p = wl.make_inputs(w)
    got = gpu_run(p, "f32")
    assert got["out"].size == 0 and got["gl"].size == 0
    assert np.array_equal(got["gv"], np.zeros_like(got["gv"]))      # zeroed, not left as is
    w = _small(B=0)
    p = wl.make_inputs(w)
    got = gpu_run(p, "f32")
    assert got["out"].size == 0 and got["gv"].size == 0


def test_off_map_and_non_finite_locations():
    w = _small(B=1, Q=40, sigma=40.0)                     # most samples far off the map
    p = wl.make_inputs(w)
    loc = p["loc"]
    loc[0, 0, 0, 0, 0] = (np.nan, 0.5)
    loc[0, 1, 1, 1, 1] = (0.5, np.inf)
    loc[0, 2, 2, 2, 2] = (-np.inf, np.nan)
    loc[0, 3, 0, 1, 0] = (3e38, -3e38)
    got = gpu_run(p, "f32")
    ref = oracle_run(p)
    assert np.all(np.isfinite(got["out"])) and np.all(np.isfinite(got["gl"]))
    check(got, ref, "f32", "off-map")
    assert np.all(got["gl"][0, 0, 0, 0, 0] == 0) and got["ga"][0, 0, 0, 0, 0] == 0


def test_invalid_level_table_is_empty():
    """A level whose (start, H, W) does not fit in [0, S) contributes nothing."""
    w = _small(levels=((9, 11), (4, 7), (2, 3)))
    p = wl.make_inputs(w)
    bad = dict(p)
    bad["starts"] = p["starts"].copy()
    bad["starts"][2] = w.S - 2                               # 2x3 level would overrun S
    got = gpu_run(bad, "f32")
    ref_in = dict(p)
    ref_in["attn"] = p["attn"].copy()
    ref_in["attn"][:, :, :, 2] = 0.0                          # same as dropping the level
    ref = oracle_run(ref_in)
    check({"out": got["out"]}, {"out": ref["out"]}, "f32", "bad level")


def test_autograd_function_bf16():
    w = _small(dtype="bf16", D=32, M=4, Q=64)
    p = wl.make_inputs(w)
    t = upload(p, "bf16")
    v = t["value"].clone().requires_grad_(True)
    loc = t["loc"].clone().requires_grad_(True)
    attn = t["attn"].clone().requires_grad_(True)
    out = binding.multi_scale_deformable_attention(v, t["shapes"], t["starts"], loc, attn)
    out.backward(t["grad_out"])
    got = {"out": np64(out), "gv": np64(v.grad), "gl": np64(loc.grad), "ga": np64(attn.grad)}
    check(got, oracle_run(p), "bf16", "autograd")


def test_misaligned_device_pointer_is_rejected():
    w = _small()
    p = wl.make_inputs(w)
    t = upload(p, "f32")
    flat = torch.empty(t["value"].numel() + 1, device=dev())
    shifted = flat[1:].view_as(t["value"])                    # 4 bytes off 16-byte alignment
    shifted.copy_(t["value"])
    with pytest.raises(binding.MSDAError, match="ALIGN"):
        binding.msda_forward(shifted, t["shapes"], t["starts"], t["loc"], t["attn"])


def test_largest_supported_value_tensor():
    """S*M*D just under 2^31 (an fp32 value tensor of 8.6 GB, rows up to the
    last one). The field is linear inside each 16x16-pixel tile and every
    sample keeps its four corners inside one tile, so bilinear sampling is
    exact there and the output and gradients have closed forms."""
    H = W = 2896                                   # S*M*D = 2,147,024,896 < 2^31
    P = 16                                         # tile period; W = 181 * P
    M, D, Q, K, B = 8, 32, 512, 4, 1
    S = H * W
    assert S * M * D < 2 ** 31 and W % P == 0
    c1, c2 = 1.0, 0.5
    rows = torch.arange(S, device=dev(), dtype=torch.int64)

    def make_value():
        f = ((rows % W) % P).float() * c1 + ((rows // W) % P).float() * c2     # exact in fp32
        return f.view(1, S, 1, 1).expand(B, S, M, D).contiguous()

    rng = np.random.default_rng(3)
    ntile = W // P

    def coords(n):
        tile = rng.integers(0, ntile, size=n)
        tile[:64] = ntile - 1                       # the last tile: the last rows and columns
        return tile, tile * P + rng.uniform(0.05, P - 1.05, size=n)

    tx, px = coords(B * Q * M * K)
    ty, py = coords(B * Q * M * K)
    shp = (B, Q, M, 1, K)
    loc = np.stack([((px + 0.5) / W).reshape(shp), ((py + 0.5) / H).reshape(shp)],
                   axis=-1).astype(np.float32)
    attn = rng.random(shp).astype(np.float32)
    g = rng.standard_normal((B, Q, M * D)).astype(np.float32)
    loc64, attn64, g64 = loc.astype(np.float64), attn.astype(np.float64), g.astype(np.float64)
    x = loc64[..., 0] * W - 0.5 - (tx * P).reshape(shp)
    y = loc64[..., 1] * H - 0.5 - (ty * P).reshape(shp)
    assert np.all((x >= 0) & (x < P - 1) & (y >= 0) & (y < P - 1))
    samp = c1 * x + c2 * y                                                  # (B,Q,M,1,K)
    expect = np.repeat(np.sum(attn64 * samp, axis=(3, 4))[..., None], D, axis=-1)
    shapes = torch.tensor([[H, W]], device=dev())
    starts = torch.zeros(1, dtype=torch.int64, device=dev())
    tl, ta, tg = (torch.tensor(a, device=dev()) for a in (loc, attn, g))
    value = make_value()
    out = binding.msda_forward(value, shapes, starts, tl, ta)
    gv, gl, ga = binding.msda_backward(value, shapes, starts, tl, ta, tg)
    torch.cuda.synchronize()
    got = np64(out).reshape(B, Q, M, D)
    assert np.max(np.abs(got - expect)) <= 1e-5 * np.max(np.abs(expect))
    gsum = g64.reshape(B, Q, M, D).sum(-1)[..., None, None]                 # sum_d g
    assert rel_l2(np64(ga), samp * gsum) <= 1e-4
    assert rel_l2(np64(gl)[..., 0], attn64 * W * c1 * gsum) <= 1e-4
    assert rel_l2(np64(gl)[..., 1], attn64 * H * c2 * gsum) <= 1e-4
    # every sample's four weights sum to 1, so grad_value sums to sum a*g per head
    exp_tot = np.einsum("bqmlk,bqmd->md", attn64, g64.reshape(B, Q, M, D))
    tot = gv.double().sum(dim=(0, 1)).cpu().numpy()
    assert rel_l2(tot, exp_tot) <= 1e-4
