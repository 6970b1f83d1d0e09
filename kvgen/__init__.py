"""Seeded synthetic KV-cache tensors and random draws.

This module is the single source of inputs shared by the float64 oracle, the
CUDA library's tests and the benchmark.  It holds none of the compression
method's arithmetic: it only synthesises data with the shapes and spectral
structure of the workloads the JoLT pages describe (Mistral-7B-v0.3 GQA and
LLaMA-2-13B MHA caches; "A JoLT for the KV cache", abstract and Results), and
the random numbers the method itself consumes (the rotation's sign vector and
the FlashJoLT Gaussian sketch), so that both sides receive identical values.

Generator (all arithmetic in float64):
  * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014), used in counter form: draw i of stream k is
    mix64(k + (i + 1) * GAMMA).
  * 53-bit uniforms u = (z >> 11) * 2^-53; Box-Muller normals from pairs.
  * Unit tensor X[h, t, d] = S * sum_i i^-alpha a_i[h] b_i[t] c_i[d] with
    a, b, c i.i.d. N(0, 1) and unit-normalised, S giving unit RMS per entry;
    K tensors get a RoPE-like rotation of adjacent channel pairs
    (2p, 2p+1) by angle t * 10000^(-2p/D); N(0, sigma^2) noise is added; K
    tensors then have fixed outlier channels scaled by 8; the result is
    rounded to fp32 (RNE) and, for bf16 workloads, on to bf16 (RNE).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence, Tuple

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

FULL = -1  # grid sentinel: keep the mode untruncated (rank = T or rank = D)


# --------------------------------------------------------------------------
# SplitMix64, scalar and vectorised
# --------------------------------------------------------------------------
def mix64(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(*parts: int) -> int:
    """Derive a 64-bit stream key from a tuple of small integers."""
    k = 0
    for p in parts:
        k = mix64((k ^ (int(p) & MASK64)) + GAMMA)
    return k


def splitmix64_counter(key: int, start: int, n: int) -> np.ndarray:
    """Draws start .. start+n-1 of stream `key` as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(key) + i * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform53(key: int, start: int, n: int) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits."""
    z = splitmix64_counter(key, start, n)
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(key: int, n: int) -> np.ndarray:
    """n standard normals by Box-Muller from consecutive uniform pairs."""
    m = (n + 1) // 2
    u = uniform53(key, 0, 2 * m)
    u1 = 1.0 - u[0::2]  # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:n]


# --------------------------------------------------------------------------
# rounding helpers (data synthesis only)
# --------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int          # 1-based id used in stream keys
    n_groups: int
    H: int
    T: int
    D: int
    dtype: str           # "f32" or "bf16"
    cp_rank: int
    noise: float
    outliers: Tuple[int, ...]
    rope: bool
    rT: Tuple[int, ...]  # FULL = untruncated
    rd: Tuple[int, ...]
    bits: Tuple[int, ...]
    block: int
    budget_ratio: float  # compression ratio vs fp16 storage of all units
    token_mode: str      # "exact" or "randomized"
    oversample: int = 8
    power_iters: int = 2
    seed: int = 0

    @property
    def n_units(self) -> int:
        return 2 * self.n_groups

    @property
    def elems_per_unit(self) -> int:
        return self.H * self.T * self.D

    @property
    def fp16_bytes(self) -> int:
        return 2 * self.elems_per_unit * self.n_units

    @property
    def budget_bytes(self) -> int:
        return int(self.fp16_bytes // self.budget_ratio)

    def unit_label(self, u: int) -> str:
        return f"g{u // 2}{'KV'[u % 2]}"


_GRID = dict(rT=(4, 8, 16, 32, FULL), rd=(4, 8, 16, 32, FULL), bits=(0, 2, 4, 8))

WORKLOADS = {
    # 2 groups x {K,V} of fp32 [4, 64, 32]; rank-16 CP, noise 0.01, block 32
    "tiny": Workload("tiny", 1, 2, 4, 64, 32, "f32", 16, 0.01, (3, 17), False,
                     (4, 8, 16, 32, FULL), (4, 8, 16, FULL), (0, 2, 4, 8), 32, 2.0,
                     "exact"),
    # Mistral-7B-v0.3: 32 layers x 8 KV heads, groups of 4 layers -> H = 32
    "mistral_t1024": Workload("mistral_t1024", 2, 8, 32, 1024, 128, "bf16", 64, 0.02,
                              (3, 17, 67, 81), True, **_GRID, block=128,
                              budget_ratio=2.0, token_mode="exact"),
    "mistral_t2048": Workload("mistral_t2048", 3, 8, 32, 2048, 128, "bf16", 64, 0.02,
                              (3, 17, 67, 81), True, **_GRID, block=128,
                              budget_ratio=3.0, token_mode="exact"),
    # LLaMA-2-13B: 40 layers x 40 heads, groups of 4 layers -> H = 160
    "llama_t1024": Workload("llama_t1024", 4, 10, 160, 1024, 128, "bf16", 64, 0.02,
                            (3, 17, 67, 81), True, **_GRID, block=128,
                            budget_ratio=2.0, token_mode="exact"),
    # FlashJoLT long context: randomized token mode
    "flash_t4096": Workload("flash_t4096", 5, 8, 32, 4096, 128, "bf16", 64, 0.02,
                            (3, 17, 67, 81), True, **_GRID, block=128,
                            budget_ratio=2.0, token_mode="randomized"),
}


def custom_workload(base: str, **kw) -> Workload:
    """A workload with the generator and grid of `base` and other sizes."""
    return dataclasses.replace(WORKLOADS[base], **kw)


def _unit_norm_cols(m: np.ndarray) -> np.ndarray:
    return m / np.linalg.norm(m, axis=0, keepdims=True)


def make_unit_f64(w: Workload, u: int) -> np.ndarray:
    """Unit u's tensor in float64 before the final dtype rounding."""
    g, c = divmod(u, 2)
    H, T, D, R = w.H, w.T, w.D, w.cp_rank
    alpha = 1.0 if c == 0 else 0.5
    a = _unit_norm_cols(normals(stream_key(w.seed, w.cfg_id, g, c, 1), H * R).reshape(H, R))
    b = _unit_norm_cols(normals(stream_key(w.seed, w.cfg_id, g, c, 2), T * R).reshape(T, R))
    cc = _unit_norm_cols(normals(stream_key(w.seed, w.cfg_id, g, c, 3), D * R).reshape(D, R))
    wts = np.arange(1, R + 1, dtype=np.float64) ** (-alpha)
    x = np.empty((H, T, D), dtype=np.float64)
    bw = b * wts[None, :]
    for h in range(H):
        x[h] = (bw * a[h][None, :]) @ cc.T
    x *= math.sqrt(H * T * D / float(np.sum(x * x)))
    if c == 0 and w.rope:
        p = np.arange(D // 2, dtype=np.float64)
        ang = np.arange(T, dtype=np.float64)[:, None] * (10000.0 ** (-2.0 * p / D))[None, :]
        cs, sn = np.cos(ang), np.sin(ang)
        x0 = x[:, :, 0::2].copy()
        x1 = x[:, :, 1::2].copy()
        x[:, :, 0::2] = x0 * cs - x1 * sn
        x[:, :, 1::2] = x0 * sn + x1 * cs
    x += w.noise * normals(stream_key(w.seed, w.cfg_id, g, c, 4), H * T * D).reshape(H, T, D)
    if c == 0:
        for ch in w.outliers:
            if ch < D:
                x[:, :, ch] *= 8.0
    return x


def make_unit(w: Workload, u: int) -> np.ndarray:
    """Unit tensor as stored for the device: float32 array for "f32"
    workloads, uint16 bf16 bit patterns for "bf16" workloads."""
    x32 = make_unit_f64(w, u).astype(np.float32)
    if w.dtype == "f32":
        return x32
    return round_to_bf16(x32)


def unit_values_f64(w: Workload, stored: np.ndarray) -> np.ndarray:
    """Exact float64 values of a stored unit tensor (f32 or bf16 bits)."""
    if w.dtype == "f32":
        return stored.astype(np.float64)
    return bf16_to_f32(stored).astype(np.float64)


def make_signs(w: Workload, u: int) -> np.ndarray:
    """diag(sigma) of the rotation for unit u: int8 entries in {-1, +1}."""
    g, c = divmod(u, 2)
    z = splitmix64_counter(stream_key(w.seed, w.cfg_id, g, c, 5), 0, w.D)
    return np.where((z >> np.uint64(63)) == 1, -1, 1).astype(np.int8)


def sketch_width(w: Workload) -> int:
    """Columns of the Gaussian sketch: largest truncated r_T plus oversampling."""
    return max(r for r in w.rT if r != FULL) + w.oversample


def make_sketch(w: Workload, u: int) -> np.ndarray:
    """FlashJoLT Gaussian test matrix for unit u, float32 [H][D][ell].
    The sketch used for feature rank r_d is the slice [:, :r_d, :]."""
    g, c = divmod(u, 2)
    ell = sketch_width(w)
    om = normals(stream_key(w.seed, w.cfg_id, g, c, 6), w.H * w.D * ell)
    return om.reshape(w.H, w.D, ell).astype(np.float32)


def make_all(w: Workload, units: Sequence[int] | None = None) -> List[np.ndarray]:
    units = range(w.n_units) if units is None else units
    return [make_unit(w, u) for u in units]
