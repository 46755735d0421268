"""Pins for the fp64 oracle: it is checked against things other than itself.

* facts the pages state (msda-triton course ch. 1, "Bilinear interpolation"):
  a point on a pixel centre gets that pixel with weight 1; a point in the
  middle of four pixels gives each a quarter; the four weights lie in [0,1] and
  sum to 1; normalised x = 0.5/W lands on the centre of the first pixel; a
  corner outside the map contributes zero and the sample fades to zero as it
  leaves the map; softmax-weighted samples of a constant map return it;
* the stated equivalence with torch's grid_sample(bilinear, zeros,
  align_corners=False), forward and (autograd) backward, run in float64;
* scipy's linear RegularGridInterpolator on a map padded with a ring of zeros;
* central finite differences of the forward for every gradient;
* the identities that hold because out is linear in value and in attn;
* mutation checks: plausible mistakes planted in a COPY of the oracle's C
  source, or of the Python source of its softmax variant (never in the
  oracle itself), must each fail one of these pins; an unmutated copy taken
  the same way passes them all (the control).
"""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from scale_deformable_attention_msda_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


# ---------------------------------------------------------------- helpers

def _problem(B=2, Q=5, M=3, D=4, K=3, levels=((5, 7), (3, 4), (2, 2)), sigma=2.0,
             seed=11, ref="uniform"):
    w = wl.Workload("pin", B=B, Q=Q, M=M, D=D, K=K, levels=levels, dtype="f32",
                    sigma_px=sigma, ref=ref, seed=seed)
    return wl.make_inputs(w)


def grid_sample_msda(value, shapes, starts, loc, attn):
    """The operator written with torch's grid_sample (float64, CPU)."""
    B, S, M, D = value.shape
    Q, L, K = loc.shape[1], loc.shape[3], loc.shape[4]
    out = torch.zeros(B, Q, M * D, dtype=torch.float64)
    for l in range(L):
        H, W = int(shapes[l][0]), int(shapes[l][1])
        s0 = int(starts[l])
        v = value[:, s0:s0 + H * W].reshape(B, H, W, M, D).permute(0, 3, 4, 1, 2)
        v = v.reshape(B * M, D, H, W)
        g = loc[:, :, :, l].permute(0, 2, 1, 3, 4).reshape(B * M, Q, K, 2) * 2 - 1
        smp = F.grid_sample(v, g, mode="bilinear", padding_mode="zeros",
                            align_corners=False)                       # (B*M, D, Q, K)
        a = attn[:, :, :, l].permute(0, 2, 1, 3).reshape(B * M, 1, Q, K)
        o = (smp * a).sum(-1).reshape(B, M, D, Q).permute(0, 3, 1, 2)
        out = out + o.reshape(B, Q, M * D)
    return out


def _torch_reference(p):
    t = {k: torch.tensor(p[k], dtype=torch.float64, requires_grad=True)
         for k in ("value", "loc", "attn")}
    out = grid_sample_msda(t["value"], p["shapes"], p["starts"], t["loc"], t["attn"])
    g = torch.tensor(p["grad_out"], dtype=torch.float64)
    out.backward(g)
    return (out.detach().numpy(), t["value"].grad.numpy(), t["loc"].grad.numpy(),
            t["attn"].grad.numpy())


def _away_from_kinks(p, margin):
    """True for samples whose pixel coordinates are not within margin of an integer."""
    H = p["shapes"][:, 0].astype(np.float64)[None, None, None, :, None]
    W = p["shapes"][:, 1].astype(np.float64)[None, None, None, :, None]
    x = p["loc"][..., 0] * W - 0.5
    y = p["loc"][..., 1] * H - 0.5
    fx = np.abs(x - np.round(x))
    fy = np.abs(y - np.round(y))
    return (fx > margin) & (fy > margin)


# ------------------------------------------------ pins as reusable checks
# Each check raises AssertionError on a mismatch; ``lib`` selects which oracle
# library is checked (the real one, or a mutant in the mutation test).

def check_pixel_centres(oracle, lib=None):
    """A point on a pixel centre returns that pixel exactly; x=0.5/W is pixel 0."""
    rng = np.random.default_rng(5)
    levels = ((5, 7), (3, 4), (2, 6))
    p = _problem(B=2, Q=6, M=3, D=5, K=2, levels=levels)
    B, Q, M, L, K = 2, 6, 3, len(levels), 2
    loc = np.empty((B, Q, M, L, K, 2))
    attn = np.zeros((B, Q, M, L, K))
    expect = np.empty((B, Q, M, p["value"].shape[3]))
    for b in range(B):
        for q in range(Q):
            for m in range(M):
                for l, (h, w) in enumerate(levels):
                    for k in range(K):
                        i, j = rng.integers(h), rng.integers(w)
                        if b == 0 and q == 0:
                            i, j = 0, 0            # x = 0.5/W, y = 0.5/H
                        loc[b, q, m, l, k] = ((j + 0.5) / w, (i + 0.5) / h)
                lsel, ksel = rng.integers(L), rng.integers(K)
                attn[b, q, m, lsel, ksel] = 1.0
                h, w = levels[lsel]
                j = loc[b, q, m, lsel, ksel, 0] * w - 0.5
                i = loc[b, q, m, lsel, ksel, 1] * h - 0.5
                row = p["starts"][lsel] + int(round(i)) * w + int(round(j))
                expect[b, q, m] = p["value"][b, row, m]
    out = oracle.forward(p["value"], p["shapes"], p["starts"], loc, attn, lib=lib)
    assert np.array_equal(out.reshape(expect.shape), expect)


def check_quarters_and_weights(oracle, lib=None):
    """One-hot maps read back the four corner weights: each in [0,1], summing
    to 1; weight 1 on a pixel centre; a quarter each at the middle of four."""
    h, w = 6, 9
    i0, j0 = 2, 4
    corners_ij = ((i0, j0), (i0, j0 + 1), (i0 + 1, j0), (i0 + 1, j0 + 1))
    value = np.zeros((1, h * w, 1, 4))
    for c, (i, j) in enumerate(corners_ij):
        value[0, i * w + j, 0, c] = 1.0
    fr = np.arange(8) / 8.0
    lx, ly = np.meshgrid(fr, fr, indexing="ij")
    lx, ly = lx.ravel(), ly.ravel()
    Q = lx.size
    loc = np.empty((1, Q, 1, 1, 1, 2))
    loc[0, :, 0, 0, 0, 0] = (j0 + lx + 0.5) / w
    loc[0, :, 0, 0, 0, 1] = (i0 + ly + 0.5) / h
    attn = np.ones((1, Q, 1, 1, 1))
    out = oracle.forward(value, np.array([[h, w]]), np.array([0]), loc, attn, lib=lib)
    wts = out.reshape(Q, 4)
    assert np.all(wts >= 0.0) and np.all(wts <= 1.0)
    assert np.allclose(wts.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    on_pixel = (lx == 0) & (ly == 0)
    assert np.array_equal(wts[on_pixel], [[1.0, 0.0, 0.0, 0.0]])
    middle = (lx == 0.5) & (ly == 0.5)
    assert np.array_equal(wts[middle], [[0.25, 0.25, 0.25, 0.25]])
    # moving right shifts weight from the left corners to the right corners
    right = wts[:, 1] + wts[:, 3]
    assert np.allclose(right, lx, rtol=0, atol=1e-15)
    below = wts[:, 2] + wts[:, 3]
    assert np.allclose(below, ly, rtol=0, atol=1e-15)


def check_constant_map(oracle, lib=None):
    """Softmax weights over interior samples of a constant map return the constant."""
    w = wl.Workload("const", B=2, Q=40, M=4, D=3, K=4, levels=((12, 17), (6, 9)),
                    sigma_px=0.7, ref="uniform", seed=3)
    p = wl.make_inputs(w)
    loc = p["loc"].copy()
    for l, (h, ww) in enumerate(w.levels):   # keep every sample at least 1 px inside
        loc[..., l, :, 0] = np.clip(loc[..., l, :, 0], 1.0 / ww, 1 - 1.0 / ww)
        loc[..., l, :, 1] = np.clip(loc[..., l, :, 1], 1.0 / h, 1 - 1.0 / h)
    attn = p["attn"] / p["attn"].sum(axis=(-1, -2), keepdims=True)
    value = np.full_like(p["value"], 2.75)
    out = oracle.forward(value, p["shapes"], p["starts"], loc, attn, lib=lib)
    assert np.allclose(out, 2.75, rtol=0, atol=1e-14)


def check_off_map(oracle, lib=None):
    """A sample with every corner off the map contributes nothing and gets zero gradients."""
    p = _problem(B=1, Q=4, M=2, D=3, K=2, levels=((4, 5), (2, 3)))
    loc = p["loc"].copy()
    far = np.array([[-0.5, 0.5], [1.5, 0.5], [0.5, -0.6], [0.5, 1.7]])
    loc[0, :, :, :, :, :] = far[:, None, None, None, :]
    loc[0, 0, 0, 0, 0] = (np.nan, 0.5)
    loc[0, 1, 1, 1, 1] = (0.3, np.inf)
    loc[0, 2, 0, 1, 0] = (-1e30, 1e30)
    out = oracle.forward(p["value"], p["shapes"], p["starts"], loc, p["attn"], lib=lib)
    assert np.array_equal(out, np.zeros_like(out))
    gv, gl, ga = oracle.backward(p["value"], p["shapes"], p["starts"], loc, p["attn"],
                                 p["grad_out"], lib=lib)
    assert not gv.any() and not gl.any() and not ga.any()


def check_fade_at_border(oracle, lib=None):
    """As a point leaves through the left edge the sample fades linearly to 0."""
    h, w = 3, 4
    value = np.random.default_rng(2).standard_normal((1, h * w, 1, 2))
    xs = np.linspace(0.5, -1.25, 71)                 # pixel coordinate of the point
    Q = xs.size
    loc = np.empty((1, Q, 1, 1, 1, 2))
    loc[0, :, 0, 0, 0, 0] = (xs + 0.5) / w
    loc[0, :, 0, 0, 0, 1] = (1 + 0.5) / h          # on the centre of row 1
    out = oracle.forward(value, np.array([[h, w]]), np.array([0]), loc,
                         np.ones((1, Q, 1, 1, 1)), lib=lib).reshape(Q, 2)
    v0 = value[0, 1 * w + 0, 0]
    expect = np.clip(xs + 1.0, 0.0, None)[:, None] * v0[None, :]
    expect[xs >= 0] = np.nan                         # checked only off the left column
    m = xs < 0
    assert np.allclose(out[m], expect[m], rtol=0, atol=1e-13)
    assert np.max(np.abs(np.diff(out, axis=0))) < 0.1  # continuous: small steps, small changes


def check_grid_sample(oracle, lib=None, seed=11):
    """Forward and all three gradients equal torch grid_sample + autograd in float64."""
    p = _problem(B=2, Q=7, M=3, D=4, K=3, levels=((5, 7), (3, 4), (2, 2)), sigma=2.5,
                 seed=seed)
    out_t, gv_t, gl_t, ga_t = _torch_reference(p)
    out = oracle.forward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"], lib=lib)
    assert np.allclose(out, out_t, rtol=1e-12, atol=1e-12)
    gv, gl, ga = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                                 p["grad_out"], lib=lib)
    assert np.allclose(gv, gv_t, rtol=1e-11, atol=1e-11)
    assert np.allclose(ga, ga_t, rtol=1e-11, atol=1e-11)
    ok = _away_from_kinks(p, 1e-6)[..., None]
    assert np.allclose(np.where(ok, gl, 0), np.where(ok, gl_t, 0), rtol=1e-10, atol=1e-10)


def check_finite_differences(oracle, lib=None):
    """Every gradient entry of the tiny workload against central differences."""
    p = wl.make_inputs(wl.tiny())
    g = p["grad_out"]

    def loss(value, loc, attn):
        o = oracle.forward(value, p["shapes"], p["starts"], loc, attn, lib=lib)
        return float(np.sum(o * g))

    gv, gl, ga = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                                 g, lib=lib)
    h = 1e-6
    for name, arr, grad in (("value", p["value"], gv), ("attn", p["attn"], ga),
                            ("loc", p["loc"], gl)):
        flat = arr.reshape(-1)
        fd = np.empty(flat.size)
        for i in range(flat.size):
            plus, minus = flat.copy(), flat.copy()
            plus[i] += h
            minus[i] -= h
            args = {"value": p["value"], "loc": p["loc"], "attn": p["attn"]}
            args[name] = plus.reshape(arr.shape)
            fp = loss(**args)
            args[name] = minus.reshape(arr.shape)
            fm = loss(**args)
            fd[i] = (fp - fm) / (2 * h)
        fd = fd.reshape(arr.shape)
        if name == "loc":
            # the one-sided derivative at a cell boundary is not a central difference
            keep = _away_from_kinks(p, 20 * h * 8)[..., None] & np.ones_like(arr, bool)
            fd, grad = fd[keep], grad[keep]
        err = np.linalg.norm(fd - grad) / max(np.linalg.norm(fd), 1e-300)
        assert err <= 1e-6, (name, err)


def check_linearity_identities(oracle, lib=None):
    """<g,out> = <grad_value,value> = <grad_attn,attn> (out is linear in each)."""
    p = _problem(B=2, Q=9, M=2, D=6, K=4, levels=((7, 5), (4, 3)), sigma=3.0, seed=21)
    out = oracle.forward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"], lib=lib)
    gv, gl, ga = oracle.backward(p["value"], p["shapes"], p["starts"], p["loc"], p["attn"],
                                 p["grad_out"], lib=lib)
    lhs = np.sum(p["grad_out"] * out)
    assert abs(lhs - np.sum(gv * p["value"])) <= 1e-12 * max(1.0, abs(lhs))
    assert abs(lhs - np.sum(ga * p["attn"])) <= 1e-12 * max(1.0, abs(lhs))


ALL_CHECKS = (check_pixel_centres, check_quarters_and_weights, check_constant_map,
              check_off_map, check_fade_at_border, check_grid_sample,
              check_finite_differences, check_linearity_identities)


# ------------------------------------------------------------------ tests

@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_grid_sample_more_seeds(oracle_mod, seed):
    check_grid_sample(oracle_mod, seed=seed)


def test_scipy_interpolator(oracle_mod):
    """Forward against scipy's linear interpolation on a zero-padded grid."""
    from scipy.interpolate import RegularGridInterpolator
    p = _problem(B=1, Q=11, M=2, D=3, K=4, levels=((6, 9), (3, 5)), sigma=3.0, seed=8)
    got = oracle_mod.forward(p["value"], p["shapes"], p["starts"], p["loc"],
                             p["attn"]).reshape(1, 11, 2, 3)
    expect = np.zeros_like(got)
    for l, (h, w) in enumerate(((6, 9), (3, 5))):
        s0 = p["starts"][l]
        for m in range(2):
            grid = np.zeros((h + 2, w + 2, 3))           # ring of zeros at -1 and H / W
            grid[1:-1, 1:-1] = p["value"][0, s0:s0 + h * w, m].reshape(h, w, 3)
            f = RegularGridInterpolator((np.arange(-1, h + 1), np.arange(-1, w + 1)), grid,
                                        method="linear", bounds_error=False, fill_value=0.0)
            x = p["loc"][0, :, m, l, :, 0] * w - 0.5
            y = p["loc"][0, :, m, l, :, 1] * h - 0.5
            smp = f(np.stack([y.ravel(), x.ravel()], axis=1)).reshape(11, 4, 3)
            expect[0, :, m] += np.einsum("qk,qkd->qd", p["attn"][0, :, m, l], smp)
    assert np.allclose(got, expect, rtol=1e-12, atol=1e-12)


def test_corner_rows_are_the_rows_that_receive_gradient(oracle_mod):
    """Single-sample problems: the corner rows with nonzero weight are exactly
    the value rows whose gradient is nonzero (the backward is pinned above)."""
    rng = np.random.default_rng(4)
    levels = ((5, 6), (3, 2))
    shapes = wl.spatial_shapes(levels)
    starts = wl.level_start_index(levels)
    for trial in range(200):
        l = int(rng.integers(2))
        loc = np.zeros((1, 1, 1, 2, 1, 2))
        loc[0, 0, 0, l, 0] = rng.uniform(-0.3, 1.3, 2)
        attn = np.zeros((1, 1, 1, 2, 1))
        attn[0, 0, 0, l, 0] = 1.0
        value = rng.standard_normal((1, 36, 1, 1))
        gv, _, _ = oracle_mod.backward(value, shapes, starts, loc, attn, np.ones((1, 1, 1)))
        rows = set(np.nonzero(gv.reshape(-1))[0].tolist())
        idx = oracle_mod.corners(shapes, starts, loc)[0, 0, 0, l, 0]
        h, w = levels[l]
        x = loc[0, 0, 0, l, 0, 0] * w - 0.5
        y = loc[0, 0, 0, l, 0, 1] * h - 0.5
        fx, fy = x - np.floor(x), y - np.floor(y)
        wts = ((1 - fx) * (1 - fy), fx * (1 - fy), (1 - fx) * fy, fx * fy)
        expect = {int(r) for r, wt in zip(idx, wts) if r >= 0 and wt > 0}
        assert rows == expect
        for r in idx:                                   # rows stay inside their level
            assert r == -1 or starts[l] <= r < starts[l] + h * w


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                lhs, rhs = line.split("->")
                rows.append((lhs.strip(), rhs.strip()))
    return rows


def test_golden_level_tables():
    rows = _read_golden("level_tables.txt")
    assert len(rows) == 2
    for lhs, rhs in rows:
        levels = tuple(tuple(int(v) for v in lv.split(",")) for lv in lhs.split(";"))
        expect = [int(v) for v in rhs.split(",")]
        assert wl.level_start_index(levels).tolist() == expect


def test_golden_counts(oracle_mod):
    """The pages' counts, reached through the oracle: on the decoder shape
    with every sample strictly inside its map, oracle.corners must give each
    query M*L*K samples of 4 in-map corners each, and those corners times D
    channels must land in the pages' "roughly twenty million" multiply-adds."""
    rows = dict(_read_golden("counts.txt"))
    reads = int(rows["reads_per_query M=8 L=4 K=4"])
    lo, hi = (int(v) for v in rows["multiply_adds B=4 Q=300 M=8 D=32 L=4 K=4"].split())
    B, Q, M, D, L, K = 4, 300, 8, 32, 4, 4
    shapes = wl.spatial_shapes(wl.LEVELS_DETR)
    starts = wl.level_start_index(wl.LEVELS_DETR)
    rng = np.random.Generator(np.random.PCG64(11))
    hw = shapes.astype(np.float64)                       # (L, 2) = (H, W)
    # pixel coordinates in [0.1, dim - 1.1]: all four corners inside the map
    px = 0.1 + rng.random((B, Q, M, L, K)) * (hw[:, 1][None, None, None, :, None] - 1.2)
    py = 0.1 + rng.random((B, Q, M, L, K)) * (hw[:, 0][None, None, None, :, None] - 1.2)
    loc = np.stack([(px + 0.5) / hw[:, 1][None, None, None, :, None],
                    (py + 0.5) / hw[:, 0][None, None, None, :, None]], axis=-1)
    c = oracle_mod.corners(shapes, starts, loc)          # (B, Q, M, L, K, 4) rows, -1 off the map
    assert c.shape == (B, Q, M, L, K, 4)
    in_map = c >= 0
    samples_per_query = np.count_nonzero(in_map.any(axis=-1).reshape(B, Q, -1), axis=-1)
    assert (samples_per_query == reads).all()
    assert lo <= int(np.count_nonzero(in_map)) * D <= hi


def test_workload_shapes_and_seeds():
    enc = wl.encoder()
    assert (enc.S, enc.Q, enc.samples) == (22223, 22223, 5689088)
    assert wl.level_start_index(wl.LEVELS_DETR).tolist() == [0, 16700, 20900, 21950]
    assert wl.mask2former().S == 21504 and wl.mask2former().samples == 8257536
    assert wl.decoder().samples == 76800
    a = wl.make_inputs(wl.tiny())
    b = wl.make_inputs(wl.tiny())
    assert all(np.array_equal(a[k], b[k]) for k in a)
    bf = wl.make_inputs(wl.decoder("bf16"))
    for k in ("value", "loc", "attn", "grad_out"):
        t = torch.tensor(bf[k]).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(t, bf[k]), k           # already on the bf16 grid


def test_query_orders_are_space_filling():
    n = 8
    x, y = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    x, y = x.ravel(), y.ravel()
    for key in (wl.hilbert_key(x, y, 3), wl.morton_key(x, y, 3)):
        assert sorted(key.tolist()) == list(range(n * n))
    o = np.argsort(wl.hilbert_key(x, y, 3))
    steps = np.abs(np.diff(x[o])) + np.abs(np.diff(y[o]))
    assert np.all(steps == 1)                          # Hilbert: every step to a neighbour
    w = wl.sweep(5000, 4, 4)
    for kind in ("linear", "morton", "hilbert"):
        perm = wl.query_order(w, kind)
        assert sorted(perm.tolist()) == list(range(5000))


# ------------------------------------------------------- mutation checks

MUTATIONS = {
    "swap_W_and_H": ("double x = loc_x * (double)W - 0.5;", "double x = loc_x * (double)H - 0.5;"),
    "drop_half_pixel": ("double y = loc_y * (double)H - 0.5;", "double y = loc_y * (double)H;"),
    "transposed_corner_weight": ("c->wgt[1] = lx * (1.0 - ly);", "c->wgt[1] = (1.0 - lx) * ly;"),
    "off_by_one_mask": ("c->xx[i] < W &&", "c->xx[i] <= W &&"),
    "row_stride_H": ("(b * S + starts[l] + c.yy[i] * W + c.xx[i]) * M + m) * D;",
                     "(b * S + starts[l] + c.yy[i] * H + c.xx[i]) * M + m) * D;"),
    "grad_loc_sign": ("(1.0 - c.ly) * (sc[1] - sc[0])", "(1.0 - c.ly) * (sc[0] - sc[1])"),
    "grad_loc_scale": ("a * (double)W * dlx", "a * (double)H * dlx"),
    "grad_value_drops_a": ("gv[d] += a * c.wgt[i] * g[d];", "gv[d] += c.wgt[i] * g[d];"),
    "grad_attn_extra_a": ("ga += c.wgt[i] * sc[i];", "ga += a * c.wgt[i] * sc[i];"),
    "grad_y_wrong_pair": ("c.lx * (sc[3] - sc[1])", "c.lx * (sc[3] - sc[2])"),
}


def _run_checks_in_child(lib_path):
    """Run every pin against a mutant library in a child process.

    Returns the names of the checks that failed; a mutant that crashes the
    child (an out-of-range read, for instance) counts as caught."""
    code = (
        "import sys; sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})\n"
        "import oracle, test_oracle_pins as t\n"
        "lib = oracle.load_library({lib!r})\n"
        "bad = []\n"
        "for c in t.ALL_CHECKS:\n"
        "    try:\n"
        "        c(oracle, lib=lib)\n"
        "    except AssertionError:\n"
        "        bad.append(c.__name__)\n"
        "print('FAILED:' + ','.join(bad))\n"
    ).format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib_path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    if r.returncode != 0:
        return ["crashed"]
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED:")][-1]
    return [x for x in line[len("FAILED:"):].split(",") if x]


def test_pins_pass_on_an_unmutated_copy(oracle_mod):
    """Control for the mutation checks: the oracle's C source compiled and
    checked through the same child-process path, unchanged, fails no pin and
    does not crash (so a caught mutant is caught by its mistake)."""
    with open(oracle_mod.SOURCE) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "copy.c")
        with open(path, "w") as f:
            f.write(src)
        lib = oracle_mod.compile_library(path, os.path.join(d, "c.so"))
        failed = _run_checks_in_child(lib)
    assert failed == [], failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(oracle_mod, name):
    old, new = MUTATIONS[name]
    with open(oracle_mod.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, name
    src = src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mutant.c")
        with open(path, "w") as f:
            f.write(src)
        lib = oracle_mod.compile_library(path, os.path.join(d, "m.so"))
        failed = _run_checks_in_child(lib)
    assert failed, f"no pin caught mutation {name}"


# ------------------------------------------------ the softmax variant

def test_softmax_variant_constant_map(oracle_mod):
    """Softmax weights sum to 1: interior samples of a constant map return it."""
    w = wl.Workload("c", B=1, Q=20, M=3, D=2, K=3, levels=((10, 12), (5, 6)), sigma_px=0.5,
                    seed=6)
    p = wl.make_inputs(w)
    loc = p["loc"].copy()
    for l, (h, ww) in enumerate(w.levels):
        loc[..., l, :, 0] = np.clip(loc[..., l, :, 0], 1.0 / ww, 1 - 1.0 / ww)
        loc[..., l, :, 1] = np.clip(loc[..., l, :, 1], 1.0 / h, 1 - 1.0 / h)
    logits = np.random.default_rng(1).standard_normal(p["attn"].shape) * 3
    out = oracle_mod.forward_softmax(np.full_like(p["value"], -1.5), p["shapes"], p["starts"],
                                     loc, logits)
    assert np.allclose(out, -1.5, rtol=0, atol=1e-14)


def test_softmax_variant_matches_torch_autograd(oracle_mod):
    p = _problem(B=2, Q=6, M=2, D=3, K=3, levels=((5, 7), (3, 4)), sigma=2.0, seed=17)
    logits = np.random.default_rng(2).standard_normal(p["attn"].shape) * 2
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in (("value", p["value"]), ("loc", p["loc"]), ("z", logits))}
    B, Q, M, L, K = logits.shape
    a = torch.softmax(t["z"].reshape(B, Q, M, L * K), dim=-1).reshape(B, Q, M, L, K)
    out = grid_sample_msda(t["value"], p["shapes"], p["starts"], t["loc"], a)
    out.backward(torch.tensor(p["grad_out"]))
    got = oracle_mod.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"], logits)
    assert np.allclose(got, out.detach().numpy(), rtol=1e-12, atol=1e-12)
    gv, gl, gz = oracle_mod.backward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                             logits, p["grad_out"])
    assert np.allclose(gv, t["value"].grad.numpy(), rtol=1e-11, atol=1e-11)
    assert np.allclose(gz, t["z"].grad.numpy(), rtol=1e-11, atol=1e-11)
    ok = _away_from_kinks(p, 1e-6)[..., None]
    assert np.allclose(np.where(ok, gl, 0), np.where(ok, t["loc"].grad.numpy(), 0),
                       rtol=1e-10, atol=1e-10)


def test_softmax_variant_finite_differences(oracle_mod):
    p = wl.make_inputs(wl.tiny())
    logits = np.random.default_rng(3).standard_normal(p["attn"].shape)
    g = p["grad_out"]
    _, _, gz = oracle_mod.backward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                           logits, g)
    h = 1e-6
    flat = logits.reshape(-1)
    fd = np.empty(flat.size)
    for i in range(flat.size):
        zp, zm = flat.copy(), flat.copy()
        zp[i] += h
        zm[i] -= h
        fp = np.sum(g * oracle_mod.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                                   zp.reshape(logits.shape)))
        fm = np.sum(g * oracle_mod.forward_softmax(p["value"], p["shapes"], p["starts"], p["loc"],
                                                   zm.reshape(logits.shape)))
        fd[i] = (fp - fm) / (2 * h)
    assert np.linalg.norm(fd - gz.reshape(-1)) <= 1e-6 * np.linalg.norm(fd)


SOFTMAX_MUTATIONS = {
    "softmax_over_points_only": ("    lead = z.shape[:-2]\n", "    lead = z.shape[:-1]\n"),
    "logit_grad_drops_the_mean": ("    gz = af * (gf - np.sum(af * gf, axis=-1, keepdims=True))",
                                  "    gz = af * gf"),
    "logit_grad_sign": ("    gz = af * (gf - np.sum(af * gf, axis=-1, keepdims=True))",
                        "    gz = af * (np.sum(af * gf, axis=-1, keepdims=True) - gf)"),
    "logit_grad_wrong_axis": ("    gz = af * (gf - np.sum(af * gf, axis=-1, keepdims=True))",
                              "    gz = af * (gf - np.sum(af * gf, axis=0, keepdims=True))"),
}
SOFTMAX_PINS = (test_softmax_variant_constant_map, test_softmax_variant_matches_torch_autograd,
                test_softmax_variant_finite_differences)


def _oracle_copy(old=None, new=None):
    """A separate module made from the oracle's Python source, with `old`
    replaced by `new` (no replacement: an exact copy), over the same
    compiled library."""
    import importlib.util
    path = os.path.join(ROOT, "oracle", "__init__.py")
    with open(path) as f:
        src = f.read()
    if old is not None:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    spec = importlib.util.spec_from_loader("oracle_softmax_copy", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__file__ = path                             # the compiled library is found from here
    exec(compile(src, path, "exec"), mod.__dict__)
    return mod


def test_softmax_pins_pass_on_an_unmutated_copy(oracle_mod):
    """Control for the mutation checks below: the copy mechanism itself
    leaves every softmax pin passing."""
    copy = _oracle_copy()
    for pin in SOFTMAX_PINS:
        pin(copy)


@pytest.mark.parametrize("name", sorted(SOFTMAX_MUTATIONS))
def test_softmax_pins_catch_planted_mistake(oracle_mod, name):
    """A plausible mistake planted in a COPY of the oracle's softmax variant
    (its Python source, loaded as a separate module over the same compiled
    library) must fail at least one of the softmax pins above."""
    mutant = _oracle_copy(*SOFTMAX_MUTATIONS[name])
    caught = []
    for pin in SOFTMAX_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no softmax pin caught mutation {name}"
