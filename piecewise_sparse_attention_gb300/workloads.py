"""Seeded synthetic Q/K/V workloads shaped like the DiT attention layers that
PISA targets.

This module only draws numbers: it holds none of the attention arithmetic, so
both the CUDA path and the CPU reference (``oracle/``) can take their inputs
from it without sharing any of the method's code.

Workloads (heads x tokens x head_dim, block size 64):

* ``tiny``     2 x 1024 x 64, fp32, 4x16x16 grid in raster order, top-k 4.
* ``flux``     24 x 4608 x 128, bf16, 512 text tokens then a 64x64 image grid,
               density 0.15 (top-k 11 of 72 blocks).
* ``wan``      40 x 32760 x 128, bf16, 21x30x52 latent grid in Morton order,
               4 outlier channels x8, density 0.125 (top-k 64 of 512).
* ``hunyuan``  24 x 65536 x 128, bf16, 16x64x64 grid in Morton order,
               8 outlier channels x8, density 0.125 (top-k 128 of 1024).
* ``long``     16 x 131072 x 128, bf16, 32x64x64 grid in Morton order,
               density 0.0625 (top-k 128 of 2048).

The shapes follow the models named in "PISA: Piecewise Sparse Attention Is
Wiser for Efficient Diffusion Transformers" (Section 4.1, Table 1: Wan2.1-14B,
HunyuanVideo, FLUX.1) and the protocol of the Piecewise-Taylor-Attention
README (block 64, density 0.125, +-1 exact band, Morton tile order).

Recipe per head (every head has its own ``SeedSequence([1000 + cfg_id, h])``
stream, so one head can be regenerated without the others):

1. outlier channels (if any): ``rng.choice(d, n_outliers, replace=False)``,
   shared by q and k;
2. for q, then k: wave-vector indices ``integers(0, 26, (d, 8))``, phases
   ``uniform(0, 2pi, (d, 8))``, noise ``0.5 * standard_normal((n_img, d),
   float32)``;
3. v: ``standard_normal((n, d), float32)``;
4. text tokens (flux only): q then k, ``standard_normal((n_text, d), float32)``.

Field of channel c at token (t, y, x) on a T x Y x X grid:
``(1/sqrt(8)) * sum_s sin(2 pi (a_s t/T + b_s y/Y + g_s x/X) + phi_s)`` with
(a, b, g) in {0,1,2}^3 minus the zero vector (26 wave vectors), i.e. a field
with the power of one unit-amplitude sinusoid. q and k get independent fields
plus the noise; outlier channels are multiplied by 8 after the noise; tiny and
flux multiply q and k by 1/sqrt(d). The result is rounded once to the
workload dtype (round-to-nearest-even for bf16) and returned as float32 arrays
holding exactly representable values.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    heads: int
    n: int
    d: int
    topk: int
    band: int
    dtype: str  # "f32" or "bf16"
    grid: tuple  # (T, Y, X) of the image/video tokens
    order: str  # "raster" or "morton"
    n_text: int = 0
    n_outliers: int = 0
    outlier_gain: float = 8.0
    prescale: bool = False
    density: float | None = None
    block: int = BLOCK

    @property
    def nb(self) -> int:
        return -(-self.n // self.block)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def max_sel(self) -> int:
        return min(self.nb, self.topk + 2 * self.band + 1)


def topk_from_density(density: float, nb: int) -> int:
    """Blocks computed exactly besides the band: ceil(density * n_blocks)."""
    return int(math.ceil(density * nb - 1e-12))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1024, 64, 4, 1, "f32", (4, 16, 16), "raster",
                     prescale=True),
    "flux": Workload("flux", 2, 24, 4608, 128, topk_from_density(0.15, 72), 1,
                     "bf16", (1, 64, 64), "raster", n_text=512, prescale=True,
                     density=0.15),
    "wan": Workload("wan", 3, 40, 32760, 128, topk_from_density(0.125, 512), 1,
                    "bf16", (21, 30, 52), "morton", n_outliers=4, density=0.125),
    "hunyuan": Workload("hunyuan", 4, 24, 65536, 128,
                        topk_from_density(0.125, 1024), 1, "bf16", (16, 64, 64),
                        "morton", n_outliers=8, density=0.125),
    "long": Workload("long", 5, 16, 131072, 128, topk_from_density(0.0625, 2048),
                     1, "bf16", (32, 64, 64), "morton", density=0.0625),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 holding the rounded values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _morton_key(t, y, x, bits):
    key = np.zeros(t.shape, dtype=np.int64)
    for b in range(bits):
        key |= ((t >> b) & 1).astype(np.int64) << (3 * b + 2)
        key |= ((y >> b) & 1).astype(np.int64) << (3 * b + 1)
        key |= ((x >> b) & 1).astype(np.int64) << (3 * b)
    return key


def token_coords(grid, order):
    """(t, y, x) integer coordinates of the grid tokens in sequence order."""
    T, Y, X = grid
    t, y, x = np.meshgrid(np.arange(T), np.arange(Y), np.arange(X), indexing="ij")
    t, y, x = t.ravel(), y.ravel(), x.ravel()
    if order == "morton":
        bits = max(int(math.ceil(math.log2(max(T, Y, X, 2)))), 1)
        perm = np.argsort(_morton_key(t, y, x, bits), kind="stable")
        t, y, x = t[perm], y[perm], x[perm]
    elif order != "raster":
        raise ValueError(order)
    return t, y, x


_WAVES = np.array([(a, b, g) for a in range(3) for b in range(3) for g in range(3)
                   if (a, b, g) != (0, 0, 0)], dtype=np.float64)


def _wave_basis(grid, order):
    T, Y, X = grid
    t, y, x = token_coords(grid, order)
    theta = 2.0 * np.pi * (np.outer(_WAVES[:, 0], t / T) + np.outer(_WAVES[:, 1], y / Y)
                           + np.outer(_WAVES[:, 2], x / X))
    return np.sin(theta), np.cos(theta)  # [26, n_img]


def _field(rng, d, basis):
    sin_t, cos_t = basis
    waves = rng.integers(0, len(_WAVES), size=(d, 8))
    phases = rng.uniform(0.0, 2.0 * np.pi, size=(d, 8))
    amp = 1.0 / math.sqrt(8.0)
    cs = np.zeros((d, len(_WAVES)))
    cc = np.zeros((d, len(_WAVES)))
    rows = np.repeat(np.arange(d), 8)
    # sin(theta + phi) = sin(theta) cos(phi) + cos(theta) sin(phi)
    np.add.at(cs, (rows, waves.ravel()), amp * np.cos(phases.ravel()))
    np.add.at(cc, (rows, waves.ravel()), amp * np.sin(phases.ravel()))
    return (cs @ sin_t + cc @ cos_t).T  # [n_img, d]


_BASIS_CACHE: dict = {}


def make_head(wl: Workload, h: int, seed_offset: int = 0):
    """Q, K, V of head ``h`` as float32 [n, d] arrays whose values are exact in
    the workload dtype."""
    key = (wl.grid, wl.order)
    if key not in _BASIS_CACHE:
        _BASIS_CACHE.clear()
        _BASIS_CACHE[key] = _wave_basis(wl.grid, wl.order)
    basis = _BASIS_CACHE[key]
    n_img = basis[0].shape[1]
    assert n_img + wl.n_text == wl.n, (wl.name, n_img, wl.n_text, wl.n)
    rng = np.random.default_rng(np.random.SeedSequence([1000 + wl.cfg_id + seed_offset, h]))
    outl = rng.choice(wl.d, wl.n_outliers, replace=False) if wl.n_outliers else None
    qk = []
    for _ in range(2):
        f = _field(rng, wl.d, basis)
        f += 0.5 * rng.standard_normal((n_img, wl.d), dtype=np.float32)
        qk.append(f)
    v = rng.standard_normal((wl.n, wl.d), dtype=np.float32)
    out = []
    for img in qk:
        if wl.n_text:
            txt = rng.standard_normal((wl.n_text, wl.d), dtype=np.float32).astype(np.float64)
            img = np.concatenate([txt, img], axis=0)
        if outl is not None:
            img[:, outl] *= wl.outlier_gain
        if wl.prescale:
            img = img / math.sqrt(wl.d)
        out.append(img)
    q, k = out
    res = []
    for a in (q, k, v):
        a = np.asarray(a, dtype=np.float32)
        if wl.dtype == "bf16":
            a = round_to_bf16(a)
        res.append(np.ascontiguousarray(a))
    return tuple(res)


def make_inputs(wl: Workload, heads=None, seed_offset: int = 0):
    """Stacked [H, n, d] float32 arrays for the requested heads (default all)."""
    hs = range(wl.heads) if heads is None else heads
    qs, ks, vs = [], [], []
    for h in hs:
        q, k, v = make_head(wl, h, seed_offset)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return np.stack(qs), np.stack(ks), np.stack(vs)


def small_case(heads, n, d, seed, dtype="bf16", spread=1.0, mean_scale=1.0):
    """Generic random case for parity/edge tests: q, k = per-block smooth mean
    plus noise, v ~ N(0, 1). Returns float32 arrays exact in ``dtype``."""
    rng = np.random.default_rng(np.random.SeedSequence([7, seed, heads, n, d]))
    nb = -(-n // BLOCK)
    out = []
    for _ in range(2):
        centers = mean_scale * rng.standard_normal((heads, nb, d))
        x = np.repeat(centers, BLOCK, axis=1)[:, :n]
        x = x + spread * rng.standard_normal((heads, n, d))
        out.append(x)
    out.append(rng.standard_normal((heads, n, d)))
    res = []
    for a in out:
        a = np.asarray(a, dtype=np.float32)
        if dtype == "bf16":
            a = round_to_bf16(a)
        res.append(np.ascontiguousarray(a))
    return tuple(res)
