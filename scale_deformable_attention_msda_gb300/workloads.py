"""Seeded synthetic inputs for multi-scale deformable attention.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It only DRAWS operands; it holds none of the operator's arithmetic (no
coordinate mapping, no interpolation, no gradients). Everything is generated in
float64 with numpy's PCG64 and rounded once to the run dtype's grid, so a bf16
run and the fp64 oracle see exactly the same numbers.

Workloads (shapes of the pages' detector workloads; no dataset is used):
  tiny         B=1, Q=16, M=2, D=8, L=2 levels (8,8),(4,4) [S=80], K=2, fp32.
  decoder      Deformable-DETR decoder: B=2, Q=300, M=8, D=32, K=4, the four
               levels of an 800x1333 image at strides 8/16/32/64 [S=22223],
               reference points U[0,1]^2.
  encoder      Deformable-DETR encoder: as decoder but Q=S=22223, each query's
               reference point the pixel centre of its own token.
  mask2former  Mask2Former pixel-decoder encoder: B=4, levels (128,128),
               (64,64),(32,32) [S=Q=21504], M=8, D=32, K=4.
  sweep        B=1, M=8, D=32, the first L levels of the encoder set,
               Q in {5000,10000,22223}, K in {2,4,8}; query i takes token
               floor(i*S/Q); optional high-contention variant.

Value, logits and grad_out are N(0,1). Attention weights are the softmax of the
logits over the L*K samples of each (b,q,m) (the operator itself uses them as
given). Offsets are N(0, sigma px) per level, divided by W_l for x and H_l for
y and added to the reference point. Seeds are 1000*config_number + variant.

Level tables follow the deformops README ("Multi-scale deformable attention"
section): spatial_shapes rows are (H_l, W_l) and level_start_index is the
exclusive prefix sum of H_l*W_l.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

LEVELS_DETR = ((100, 167), (50, 84), (25, 42), (13, 21))   # strides 8..64 of 800x1333
LEVELS_M2F = ((128, 128), (64, 64), (32, 32))              # strides 8..32 of 1024^2
LEVELS_TINY = ((8, 8), (4, 4))

DTYPES = ("f32", "bf16", "f16", "f64")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Q: int
    M: int
    D: int
    K: int
    levels: tuple
    dtype: str = "f32"
    sigma_px: float = 2.0
    ref: str = "uniform"          # "uniform" | "token" | "stride"
    contention: bool = False      # every sample of level l inside a 4x4 patch at the level centre
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def L(self) -> int:
        return len(self.levels)

    @property
    def S(self) -> int:
        return int(sum(h * w for h, w in self.levels))

    @property
    def samples(self) -> int:
        return self.B * self.Q * self.M * self.L * self.K

    def with_dtype(self, dtype: str) -> "Workload":
        return replace(self, dtype=dtype)


def level_start_index(levels) -> np.ndarray:
    """Exclusive prefix sum of H_l*W_l (int64)."""
    sizes = np.array([h * w for h, w in levels], dtype=np.int64)
    return np.concatenate([np.zeros(1, np.int64), np.cumsum(sizes)[:-1]])


def spatial_shapes(levels) -> np.ndarray:
    return np.array(levels, dtype=np.int64).reshape(-1, 2)


# --------------------------------------------------------------------------
# rounding to a storage format (round-to-nearest-even, applied once to fp64)

def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # 8 significant bits; the normal range of bf16 is that of fp32. Values
        # below the smallest normal are flushed to zero (none occur here).
        m, e = np.frexp(x)                    # x = m * 2**e, 0.5 <= |m| < 1
        r = np.ldexp(np.round(m * 256.0) / 256.0, e)
        r[np.abs(x) < 2.0 ** -126] = 0.0
        return r
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# reference points

def _token_centres(levels) -> np.ndarray:
    """(S, 2) normalised pixel centre (x, y) of every token, in token order."""
    pts = []
    for h, w in levels:
        i, j = np.meshgrid(np.arange(h), np.arange(w), indexing="ij")
        pts.append(np.stack([(j.ravel() + 0.5) / w, (i.ravel() + 0.5) / h], axis=1))
    return np.concatenate(pts, axis=0)


def reference_points(wl: Workload, rng) -> np.ndarray:
    """(B, Q, 2) reference point per query, (x, y) normalised."""
    if wl.ref == "uniform":
        return rng.random((wl.B, wl.Q, 2))
    centres = _token_centres(wl.levels)
    S = centres.shape[0]
    if wl.ref == "token":
        if wl.Q != S:
            raise ValueError("token reference points need Q == S")
        tok = np.arange(S)
    elif wl.ref == "stride":
        tok = (np.arange(wl.Q, dtype=np.int64) * S) // wl.Q
    else:
        raise ValueError(wl.ref)
    return np.broadcast_to(centres[tok][None], (wl.B, wl.Q, 2)).copy()


# --------------------------------------------------------------------------
# operands

def make_inputs(wl: Workload, with_grad: bool = True) -> dict:
    """Draw every operand of one forward+backward call.

    Returns float64 arrays already on the dtype's grid: value (B,S,M,D),
    loc (B,Q,M,L,K,2), attn (B,Q,M,L,K) (softmax of logits), logits
    (B,Q,M,L,K), grad_out (B,Q,M*D); int64 shapes (L,2) and starts (L,).
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, Q, M, D, L, K, S = wl.B, wl.Q, wl.M, wl.D, wl.L, wl.K, wl.S
    hw = np.array(wl.levels, dtype=np.float64)          # (L, 2) = (H, W)
    value = rng.standard_normal((B, S, M, D))
    logits = rng.standard_normal((B, Q, M, L * K))
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))
    attn = (e / e.sum(axis=-1, keepdims=True)).reshape(B, Q, M, L, K)
    if wl.contention:
        # uniform inside the 4x4-pixel patch at each level's centre
        u = rng.random((B, Q, M, L, K, 2)) * 4.0
        loc = np.empty_like(u)
        loc[..., 0] = (hw[:, 1][None, None, None, :, None] / 2 - 2 + u[..., 0]) / hw[:, 1][None, None, None, :, None]
        loc[..., 1] = (hw[:, 0][None, None, None, :, None] / 2 - 2 + u[..., 1]) / hw[:, 0][None, None, None, :, None]
    else:
        ref = reference_points(wl, rng)                  # (B, Q, 2)
        off = rng.standard_normal((B, Q, M, L, K, 2)) * wl.sigma_px
        loc = np.empty_like(off)
        loc[..., 0] = ref[:, :, None, None, None, 0] + off[..., 0] / hw[:, 1][None, None, None, :, None]
        loc[..., 1] = ref[:, :, None, None, None, 1] + off[..., 1] / hw[:, 0][None, None, None, :, None]
    out = {
        "value": round_to(value, wl.dtype),
        "shapes": spatial_shapes(wl.levels),
        "starts": level_start_index(wl.levels),
        "loc": round_to(loc, wl.dtype),
        "attn": round_to(attn, wl.dtype),
        # the raw logits, for the variant that applies the softmax itself
        "logits": round_to(logits.reshape(B, Q, M, L, K), wl.dtype),
    }
    if with_grad:
        out["grad_out"] = round_to(rng.standard_normal((B, Q, M * D)), wl.dtype)
    return out


# --------------------------------------------------------------------------
# query dispatch orders (linear / Morton / Hilbert on the reference point)

def _quantise(ref: np.ndarray, bits: int = 16) -> tuple:
    n = 1 << bits
    q = np.clip(np.floor(ref * n), 0, n - 1).astype(np.int64)
    return q[..., 0], q[..., 1]


def morton_key(x: np.ndarray, y: np.ndarray, bits: int = 16) -> np.ndarray:
    key = np.zeros_like(x)
    for i in range(bits):
        key |= ((x >> i) & 1) << (2 * i)
        key |= ((y >> i) & 1) << (2 * i + 1)
    return key


def hilbert_key(x: np.ndarray, y: np.ndarray, bits: int = 16) -> np.ndarray:
    """Distance along the Hilbert curve of order ``bits`` (vectorised)."""
    x = x.astype(np.int64).copy()
    y = y.astype(np.int64).copy()
    d = np.zeros_like(x)
    s = 1 << (bits - 1)
    while s > 0:
        rx = ((x & s) > 0).astype(np.int64)
        ry = ((y & s) > 0).astype(np.int64)
        d += s * s * ((3 * rx) ^ ry)
        # keep the low bits and rotate that quadrant into the canonical
        # orientation of the sub-curve
        x &= s - 1
        y &= s - 1
        flip = (ry == 0) & (rx == 1)
        x = np.where(flip, s - 1 - x, x)
        y = np.where(flip, s - 1 - y, y)
        swap = ry == 0
        x, y = np.where(swap, y, x), np.where(swap, x, y)
        s >>= 1
    return d


def query_order(wl: Workload, kind: str) -> np.ndarray:
    """int32 (Q,) permutation: dispatch slot i processes query order[i].

    Keys come from each query's reference point quantised to a 2^16 x 2^16
    grid (batch 0's points; every batch shares the same points for the
    token/stride reference modes)."""
    if kind == "linear":
        return np.arange(wl.Q, dtype=np.int32)
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    ref = reference_points(wl, rng)[0]
    x, y = _quantise(ref)
    if kind == "morton":
        key = morton_key(x, y)
    elif kind == "hilbert":
        key = hilbert_key(x, y)
    else:
        raise ValueError(kind)
    return np.argsort(key, kind="stable").astype(np.int32)


# --------------------------------------------------------------------------
# the configurations

def tiny(variant: int = 0) -> Workload:
    return Workload("tiny", B=1, Q=16, M=2, D=8, K=2, levels=LEVELS_TINY,
                    dtype="f32", sigma_px=1.5, ref="uniform", seed=1000 + variant)


def decoder(dtype: str = "f32", variant: int = 0) -> Workload:
    return Workload("decoder", B=2, Q=300, M=8, D=32, K=4, levels=LEVELS_DETR,
                    dtype=dtype, sigma_px=2.0, ref="uniform", seed=2000 + variant)


def encoder(dtype: str = "f32", variant: int = 0, B: int = 2) -> Workload:
    S = sum(h * w for h, w in LEVELS_DETR)
    return Workload("encoder", B=B, Q=S, M=8, D=32, K=4, levels=LEVELS_DETR,
                    dtype=dtype, sigma_px=2.0, ref="token", seed=3000 + variant)


def mask2former(dtype: str = "bf16", variant: int = 0) -> Workload:
    S = sum(h * w for h, w in LEVELS_M2F)
    return Workload("mask2former", B=4, Q=S, M=8, D=32, K=4, levels=LEVELS_M2F,
                    dtype=dtype, sigma_px=2.0, ref="token", seed=4000 + variant)


def sweep(Q: int, K: int, L: int, contention: bool = False, dtype: str = "bf16",
          variant: int = 0) -> Workload:
    if not 1 <= L <= 4:
        raise ValueError("the sweep uses 1 to 4 levels of the encoder set")
    return Workload(f"sweep_Q{Q}_K{K}_L{L}" + ("_contention" if contention else ""),
                    B=1, Q=Q, M=8, D=32, K=K, levels=LEVELS_DETR[:L], dtype=dtype,
                    sigma_px=2.0, ref="stride", contention=contention,
                    seed=5000 + variant)


def sweep_grid():
    for Q in (5000, 10000, 22223):
        for K in (2, 4, 8):
            for L in (1, 2, 3, 4):
                yield sweep(Q, K, L)


# --------------------------------------------------------------------------
# counting (for the benchmark's roofline; no operator arithmetic)

ELEMENT_BYTES = {"f64": 8, "f32": 4, "bf16": 2, "f16": 2}


def compulsory_bytes(wl: Workload) -> dict:
    """Each operand counted once at its storage dtype.

    forward  = value + loc + attn + out
    backward = grad_out + value + loc + attn + grad_value + grad_loc + grad_attn
    """
    e = ELEMENT_BYTES[wl.dtype]
    n = wl.samples
    value = wl.B * wl.S * wl.M * wl.D * e
    out = wl.B * wl.Q * wl.M * wl.D * e
    loc = 2 * n * e
    attn = n * e
    fwd = value + loc + attn + out
    bwd = out + value + loc + attn + value + loc + attn
    return {"forward": fwd, "backward": bwd}


def multiply_adds(wl: Workload) -> int:
    """Forward multiply-adds: 4 corners x D channels per sample."""
    return wl.samples * 4 * wl.D
