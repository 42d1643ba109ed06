"""Seeded synthetic video-DiT attention inputs.

This module is shared by the oracle-side tests and the CUDA path. It only
draws random numbers and lays them out; it holds none of the method's
arithmetic (no reordering, pooling, selection or attention).

Workloads stand in for the video latents the pages measure on (Wan2.2 I2V,
"mlsift.com tag listing", sequence-parallelism entry; MovieGen-like training
data, "Dynamic Sparsity in Large-Scale Video DiT Training", trade-offs), which
are not available here. Each head gets:

* a smooth locality field F: 8 random Fourier features over the normalised
  (t, y, x) position, with unit expected squared norm;
* a shared direction u ~ N(0, I/d) added to every query, and added with
  weight 2*s_h to the keys of n_hot "hot" key tiles, so that a few key blocks
  draw attention from everywhere (the power-law, non-local critical pairs of
  "Dynamic Sparsity in Large-Scale Video DiT Training", prior-work section);
* i.i.d. N(0, 1) noise for Q, K and V.

Tokens are laid out raster-major, [B, N, H, d] with N = T*Y*X and x fastest.
Hot tiles are axis-aligned (a, b, c) boxes on the tile lattice of the grid.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d: int
    T: int
    Y: int
    X: int
    ta: int
    tb: int
    tc: int
    dtype: str            # "f32" or "bf16"
    estimator: str        # "mean" or "lowrank"
    top_p: float
    k_floor: int
    P: int
    n_hot: int
    skew: bool            # per-head concentration scale log-uniform in [0.25, 8]
    backward: bool        # forward + backward (dO drawn)
    seed: int
    rank: int = 16

    @property
    def N(self) -> int:
        return self.T * self.Y * self.X

    @property
    def Bt(self) -> int:
        return self.ta * self.tb * self.tc

    @property
    def nb(self) -> int:
        return self.N // self.Bt

    @property
    def tiles(self) -> tuple[int, int, int]:
        return (self.T // self.ta, self.Y // self.tb, self.X // self.tc)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS: dict[str, Workload] = {
    # 1,024 tokens, 16 blocks of 64, fp32, forward only.
    "tiny": Workload("tiny-1k-fp32", 1, 2, 64, 4, 16, 16, 4, 4, 4, "f32", "mean",
                     0.9, 2, 2, 2, False, False, 1),
    # 8,192 tokens, 128 blocks of 64, bf16, forward only.
    "medium": Workload("medium-8k-bf16", 1, 12, 64, 8, 32, 32, 4, 4, 4, "bf16", "mean",
                       0.9, 4, 4, 4, False, False, 2),
    # Wan-14B attention-layer shape: 30,720 tokens, 240 blocks of 128, 40 heads.
    "wan": Workload("wan14b-layer-30k-bf16", 1, 40, 128, 20, 32, 48, 2, 8, 8, "bf16", "mean",
                    0.95, 8, 8, 8, False, False, 3),
    # Same shape, per-head hot-block strength log-uniform in [0.25, 8].
    "skewed": Workload("skewed-30k-bf16", 1, 40, 128, 20, 32, 48, 2, 8, 8, "bf16", "mean",
                       0.9, 4, 8, 8, True, False, 4),
    # Training shape: 65,536 tokens, 512 blocks of 128, rank-16 predictor, Top-k only.
    "training": Workload("training-64k-bf16", 1, 24, 128, 16, 64, 64, 2, 8, 8, "bf16", "lowrank",
                         0.0, 52, 8, 8, False, True, 5),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bfloat16 (ties to even), kept as float32.

    Works in place on a float32 array (returns it); other inputs are copied first.
    """
    if not (isinstance(x, np.ndarray) and x.dtype == np.float32 and x.flags.c_contiguous):
        x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.isfinite(x).all():
        raise ValueError("round_bf16 expects finite values")
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return x


def _fourier_params(rng: np.random.Generator, d: int):
    """Draw one head's 8 Fourier features: integer frequencies, phases, coefficients."""
    omega = np.zeros((8, 3), dtype=np.int64)
    for m in range(8):
        while True:
            w = rng.integers(-2, 3, size=3)
            if np.any(w != 0):
                omega[m] = w
                break
    phi = rng.uniform(0.0, 2.0 * math.pi, size=8)
    c = rng.normal(0.0, 1.0 / math.sqrt(4.0 * d), size=(8, d))
    return omega, phi, c


def _fourier_eval(wl: Workload, params) -> np.ndarray:
    """[N, d] locality field for one head, raster order (x fastest)."""
    omega, phi, c = params
    t = np.arange(wl.T, dtype=np.float64) / wl.T
    y = np.arange(wl.Y, dtype=np.float64) / wl.Y
    x = np.arange(wl.X, dtype=np.float64) / wl.X
    tt, yy, xx = np.meshgrid(t, y, x, indexing="ij")
    pos = np.stack([tt.ravel(), yy.ravel(), xx.ravel()], axis=1)       # [N, 3]
    phase = 2.0 * math.pi * (pos @ omega.T.astype(np.float64)) + phi    # [N, 8]
    return (np.cos(phase) @ c).astype(np.float32)                       # [N, d]


def _hot_token_mask(wl: Workload, hot_tiles: np.ndarray) -> np.ndarray:
    """Boolean [N] raster mask of the tokens inside the chosen hot tiles.

    A tile id enumerates the tile lattice with the x tile index fastest.
    """
    nT, nY, nX = wl.tiles
    mask = np.zeros((wl.T, wl.Y, wl.X), dtype=bool)
    for tid in hot_tiles:
        bt, rem = divmod(int(tid), nY * nX)
        by, bx = divmod(rem, nX)
        mask[bt * wl.ta:(bt + 1) * wl.ta, by * wl.tb:(by + 1) * wl.tb, bx * wl.tc:(bx + 1) * wl.tc] = True
    return mask.ravel()


def make(wl: Workload, with_noise: bool = True) -> dict[str, np.ndarray]:
    """Draw the workload's tensors (float32 numpy, raster layout [B, N, H, d]).

    Draw order: per (b, h): Fourier field, u, hot tiles, strength s_h; then the
    noise Z_q, Z_k, Z_v; then (backward workloads) dO; then (low-rank
    workloads) Wq, Wk. bf16 workloads round Q, K, V and dO to bf16 once; both
    sides consume the rounded values.
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, H, N, d = wl.B, wl.H, wl.N, wl.d
    params = {}
    u_all = np.zeros((B, H, d), dtype=np.float32)
    hot = np.zeros((B, H, wl.n_hot), dtype=np.int64)
    strength = np.ones((B, H), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            params[b, h] = _fourier_params(rng, d)
            u_all[b, h] = rng.normal(0.0, 1.0 / math.sqrt(d), size=d)
            hot[b, h] = np.sort(rng.choice(wl.nb, size=wl.n_hot, replace=False))
            if wl.skew:
                strength[b, h] = math.exp(rng.uniform(math.log(0.25), math.log(8.0)))
    shape = (B, N, H, d)
    if with_noise:
        q = rng.standard_normal(shape, dtype=np.float32)
        k = rng.standard_normal(shape, dtype=np.float32)
        v = rng.standard_normal(shape, dtype=np.float32)
    else:
        q, k, v = (np.zeros(shape, np.float32) for _ in range(3))
    for b in range(B):
        for h in range(H):
            field = _fourier_eval(wl, params[b, h])
            q[b, :, h, :] += field + u_all[b, h]
            k[b, :, h, :] += field
            mask = _hot_token_mask(wl, hot[b, h])
            k[b, mask, h, :] += np.float32(2.0 * strength[b, h]) * u_all[b, h]
    out = {"q": q, "k": k, "v": v, "hot": hot, "strength": strength}
    if wl.backward:
        out["do"] = rng.standard_normal((B, N, H, d), dtype=np.float32)
    if wl.estimator == "lowrank":
        out["wq"] = rng.normal(0.0, 1.0 / math.sqrt(d), size=(H, d, wl.rank)).astype(np.float32)
        out["wk"] = rng.normal(0.0, 1.0 / math.sqrt(d), size=(H, d, wl.rank)).astype(np.float32)
    if wl.dtype == "bf16":
        for key in ("q", "k", "v", "do"):
            if key in out:
                out[key] = round_bf16(out[key])
    return out


def random_scores(seed: int, rows: int, nb: int, scale: float = 1.0) -> np.ndarray:
    """A float32 [rows, nb] score matrix for selection-only tests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal((rows, nb)) * scale).astype(np.float32)


def micro(seed: int = 7) -> tuple[Workload, dict[str, np.ndarray]]:
    """A 32-token case (T=2, Y=4, X=4, 2x2x2 tiles, d=8) for finite-difference checks."""
    wl = Workload("micro-32-f64", 1, 2, 8, 2, 4, 4, 2, 2, 2, "f32", "mean", 0.7, 1, 2, 1, False, True, seed)
    return wl, make(wl)
