"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only makes inputs: Gaussian Q/K/V rounded to the stated 16-bit
type, the per-key raised-cosine skirt bias, the tile-64 block mask with its
validity vector, and the per-(head, channel) V scale. It holds none of the
quantisation or attention arithmetic, and it imports neither the CUDA binding
nor the oracle.

Workloads (shapes from the pages' measurements; values are N(0,1) stand-ins
for activations that are not available here):

* ``tiny``        B1 H2  S256          D64  bf16, seed 0, per-token scales
* ``sdxl``        B1 H10 S4096         D64  fp16, seed 1, per-64-row-block
                  scales, K plus a per-(head, channel) offset drawn with
                  standard deviation 2 (stresses the K mean-centring)
* ``anima4k``     B1 H16 S4096         D128 bf16, seed 2, per-token, V scale
* ``anima9k``     B1 H16 S9216         D128 bf16, seed 2, per-token, V scale
* ``banded``      B1 H56 Q4096 K33600  D128 bf16, seed 3, per-key skirt bias
* ``sparse``      B1 H24 S65536        D128 bf16, seed 4, tile-64 block mask
                  (a band of 64 key tiles plus 16 random ones per query
                  tile), last tile 37 of 64 rows valid, pads zeroed
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

TILE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    dtype: str                 # "bf16" | "fp16" (Q, K, V and the output)
    seed: int
    granularity: str = "token"  # "token" | "block64"
    k_offset_sigma: float = 0.0
    v_scale: bool = False
    bias: str | None = None      # None | "skirt"
    skirt_width: int = 0         # keys of fade on each side of the core
    sparse: bool = False
    band_tiles: int = 64
    random_tiles: int = 16
    last_tile_valid: int = 64
    notes: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 256, 256, 64, "bf16", 0),
    "sdxl": Workload("sdxl", 1, 10, 4096, 4096, 64, "fp16", 1,
                     granularity="block64", k_offset_sigma=2.0),
    "anima4k": Workload("anima4k", 1, 16, 4096, 4096, 128, "bf16", 2, v_scale=True),
    "anima9k": Workload("anima9k", 1, 16, 9216, 9216, 128, "bf16", 2, v_scale=True),
    "banded": Workload("banded", 1, 56, 4096, 33600, 128, "bf16", 3,
                       bias="skirt", skirt_width=6720),
    "sparse": Workload("sparse", 1, 24, 65536, 65536, 128, "bf16", 4,
                       sparse=True, last_tile_valid=37),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """N(0,1) samples drawn in fp32 from a seeded torch generator, rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    return x.to(dtype)


def skirt_bias(Sk: int, width: int) -> np.ndarray:
    """Per-key additive bias of the banded-window workload, fp32 ``[Sk]``.

    The central ``Sk - 2*width`` keys get 0. Over ``width`` keys on each side a
    raised-cosine weight w = (1 + cos(pi*u))/2 falls from 1 towards 0 as u goes
    from 0 to 1, and the bias is ln(max(w, 1e-4)), so the outermost key sits at
    ln(1e-4). Computed in float64, rounded once to float32.
    """
    j = np.arange(Sk, dtype=np.float64)
    lo, hi = width, Sk - width
    u = np.zeros(Sk)
    left = j < lo
    right = j >= hi
    u[left] = (lo - j[left]) / width
    u[right] = (j[right] - (hi - 1)) / width
    w = 0.5 * (1.0 + np.cos(np.pi * u))
    b = np.log(np.maximum(w, 1e-4))
    b[~(left | right)] = 0.0
    return b.astype(np.float32)


def band_random_mask(H: int, T: int, band: int, n_random: int, seed: int) -> np.ndarray:
    """Tile-64 block mask ``[1, H, T, T]`` (bool).

    Query tile i keeps the band of ``band`` key tiles starting at
    clamp(i - band/2, 0, T - band) plus ``n_random`` distinct tiles drawn
    uniformly from outside the band (numpy PCG64 seeded with ``seed``; rows are
    drawn in (h, i) order).
    """
    rng = np.random.default_rng(seed)
    m = np.zeros((1, H, T, T), dtype=bool)
    all_tiles = np.arange(T)
    for h in range(H):
        for i in range(T):
            start = min(max(i - band // 2, 0), T - band)
            m[0, h, i, start:start + band] = True
            outside = np.concatenate([all_tiles[:start], all_tiles[start + band:]])
            pick = rng.choice(outside, size=min(n_random, outside.size), replace=False)
            m[0, h, i, pick] = True
    return m


def rope_tables(positions: int, D: int, base: float = 10000.0):
    """cos / sin tables fp32 ``[positions, D/2]`` of the usual rotary
    frequencies: angle(p, i) = p * base^(-2i/D), computed in float64 and
    rounded once to float32 (an input of the RoPE prologue, as a model's
    position embedding is)."""
    p = np.arange(positions, dtype=np.float64)[:, None]
    i = np.arange(D // 2, dtype=np.float64)[None, :]
    ang = p * base ** (-2.0 * i / D)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def norm_weight(D: int, seed: int) -> np.ndarray:
    """A seeded RMSNorm weight fp32 ``[D]``: 1 + N(0, 0.1)."""
    g = np.random.default_rng(seed)
    return (1.0 + 0.1 * g.standard_normal(D)).astype(np.float32)


def validity_vector(T: int, last_valid: int) -> np.ndarray:
    """int32 ``[T]``: 64 valid rows per tile except the last one."""
    v = np.full(T, TILE, dtype=np.int32)
    v[-1] = last_valid
    return v


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    v_scale: torch.Tensor | None = None      # fp32 [H, D]
    bias: torch.Tensor | None = None         # fp32 [Sk]
    block_mask: torch.Tensor | None = None   # bool [B, H, Tq, Tk]
    kv_valid: torch.Tensor | None = None     # int32 [Tk]


def make_inputs(wl: Workload, device="cpu") -> Inputs:
    """All inputs of one workload on ``device`` (torch tensors, BHSD, contiguous)."""
    B, H, Sq, Sk, D = wl.B, wl.H, wl.Sq, wl.Sk, wl.D
    dt = wl.torch_dtype
    s = wl.seed * 16
    q = normal((B, H, Sq, D), s + 1, dt, device)
    k32 = torch.randn((B, H, Sk, D), generator=_gen(device, s + 2), device=device,
                      dtype=torch.float32)
    if wl.k_offset_sigma:
        off = torch.randn((1, H, 1, D), generator=_gen(device, s + 3), device=device,
                          dtype=torch.float32) * wl.k_offset_sigma
        k32 = k32 + off
    k = k32.to(dt)
    del k32
    inp = Inputs(wl, q, k, None)
    if wl.v_scale:
        v32 = torch.randn((B, H, Sk, D), generator=_gen(device, s + 4), device=device,
                          dtype=torch.float32)
        vs = v32.abs().amax(dim=(0, 2))                  # [H, D]
        inp.v = (v32 / vs[None, :, None, :]).to(dt)
        inp.v_scale = vs.contiguous()
        del v32
    else:
        inp.v = normal((B, H, Sk, D), s + 4, dt, device)
    if wl.bias == "skirt":
        inp.bias = torch.from_numpy(skirt_bias(Sk, wl.skirt_width)).to(device)
    if wl.sparse:
        T = Sk // TILE
        inp.block_mask = torch.from_numpy(
            band_random_mask(H, T, wl.band_tiles, wl.random_tiles, wl.seed)).to(device)
        vbs = validity_vector(T, wl.last_tile_valid)
        inp.kv_valid = torch.from_numpy(vbs).to(device)
        # Tile pads are zero by contract.
        pad_from = (T - 1) * TILE + wl.last_tile_valid
        for t in (inp.q, inp.k, inp.v):
            t[:, :, pad_from:, :] = 0
    return inp


def algorithmic_ops(wl: Workload, kept_tiles_per_row: float | None = None) -> float:
    """4*B*H*Sq*Sk*D (QK^T and PV multiply-adds, 2 ops each); for the block-sparse
    workload only kept 64x64 tiles count."""
    if wl.sparse:
        T = wl.Sq // TILE
        kept = kept_tiles_per_row if kept_tiles_per_row is not None else (
            wl.band_tiles + wl.random_tiles)
        return float(wl.B * wl.H * T * kept * TILE * TILE * wl.D * 4)
    return float(4 * wl.B * wl.H * wl.Sq * wl.Sk * wl.D)


def small_variant(wl: Workload, **kw) -> Workload:
    """The same workload recipe at a size the oracle finishes in seconds."""
    return wl.with_(**kw)


__all__ = ["Workload", "WORKLOADS", "Inputs", "make_inputs", "normal", "skirt_bias",
           "band_random_mask", "validity_vector", "algorithmic_ops", "small_variant",
           "TILE"]
