"""Pins of the oracle's K mean and INT8 quantiser (CPU only).

Each check compares the oracle with something other than itself: values
derived by hand from the definition, exact rational arithmetic, numpy's own
float64 mean, closed forms and invariants. The definition followed is the one
in "minimax_h3_sparse_int8" (FastVideo API page: per-token scales, K centred
by its sequence mean) with the symmetric [-127, 127] range of
"[attention-int8] Multiple build issues and numerical accuracy problem"
(maintainer's point 1).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import k_mean, quantize, row_validity

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_values(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    return x.to(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------- hand cases

def load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            xs, codes, scale = line.split("|")
            rows.append(([float(t) for t in xs.split()], [int(t) for t in codes.split()],
                         float.fromhex(scale.strip())))
    return rows


def test_hand_derived_rows():
    """tests/golden/quantize_hand.txt: rows whose codes follow by hand from
    code = rne(x * (127/amax)), each with the reasoning in the fixture."""
    for xs, codes, scale in load_golden("quantize_hand.txt"):
        x = np.array(xs, dtype=np.float32).reshape(1, 1, 1, -1)
        c, s = quantize(x)
        assert c.reshape(-1).tolist() == codes, (xs, c.reshape(-1).tolist(), codes)
        assert s.reshape(-1)[0] == np.float32(scale), (xs, s, scale)


def test_ties_round_half_even():
    # amax = 127 makes 127/amax exactly 1, so x = k + 1/2 lands on a tie.
    xs = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5], dtype=np.float32)
    c, s = quantize(xs.reshape(1, 1, 1, -1))
    assert c.reshape(-1).tolist() == [127, 0, 2, 2, 0, -2, -2, 4, 126]
    assert s.reshape(-1)[0] == np.float32(1.0)


def test_zero_row_gives_zero_scale_and_codes():
    x = np.zeros((1, 1, 3, 8), dtype=np.float32)
    x[0, 0, 1, 3] = 0.25
    c, s = quantize(x)
    assert s[0, 0, 0] == 0 and s[0, 0, 2] == 0
    assert not c[0, 0, 0].any() and not c[0, 0, 2].any()
    assert c[0, 0, 1, 3] == 127 and s[0, 0, 1] == np.float32(0.25) / np.float32(127)


@pytest.mark.parametrize("gran", ["token", "block64"])
def test_amax_maps_to_127_and_error_bound(gran):
    x = bf16_values((2, 3, 150, 64), 11, scale=3.0)
    c, s = quantize(x, granularity=gran)
    assert c.min() >= -127 and c.max() <= 127
    if gran == "token":
        srow = s
        # the largest |x| of every row maps to +-127
        assert (np.abs(c).max(axis=3) == 127).all()
    else:
        srow = np.repeat(s, 64, axis=2)[:, :, :150]
        for t in range(3):
            blk = np.abs(c[:, :, t * 64:(t + 1) * 64])
            assert (blk.max(axis=(2, 3)) == 127).all()
    # |x - code*scale| <= scale/2 up to the fp32 rounding of the reciprocal
    err = np.abs(x.astype(np.float64) - c * srow[..., None].astype(np.float64))
    bound = srow[..., None].astype(np.float64) * (0.5 + 1e-5) + 1e-30
    assert (err <= bound).all()


def test_block64_shares_scale_and_handles_ragged_tail():
    x = bf16_values((1, 2, 100, 16), 5)
    c, s = quantize(x, granularity="block64")
    assert s.shape == (1, 2, 2)
    for h in range(2):
        for t, (lo, hi) in enumerate([(0, 64), (64, 100)]):
            amax = np.abs(x[0, h, lo:hi]).max()
            assert s[0, h, t] == np.float32(amax) / np.float32(127)


def test_validity_rows_are_zero_and_excluded_from_block_amax():
    x = bf16_values((1, 1, 128, 8), 3)
    x[0, 0, 64 + 37:] = 1000.0  # pad rows that must not enter the amax
    vbs = np.array([64, 37], dtype=np.int32)
    assert row_validity(128, vbs).sum() == 101
    c, s = quantize(x, granularity="block64", kv_valid=vbs)
    assert not c[0, 0, 101:].any()
    assert s[0, 0, 1] == np.float32(np.abs(x[0, 0, 64:101]).max()) / np.float32(127)
    c2, s2 = quantize(x, granularity="token", kv_valid=vbs)
    assert not c2[0, 0, 101:].any() and not s2[0, 0, 101:].any()


def test_centring_subtracts_mean_in_fp32():
    x = bf16_values((1, 1, 4, 8), 9)
    mu = np.full((1, 1, 8), 0.1, dtype=np.float32)
    c, s = quantize(x, mu)
    xc = (x - np.float32(0.1)).astype(np.float32)
    c2, s2 = quantize(xc)
    assert (c == c2).all() and (s == s2).all()


# ----------------------------------------------------------------- the K mean

def test_mean_closed_form_ramp():
    S = 1000
    k = np.broadcast_to(np.arange(S, dtype=np.float32)[None, None, :, None], (1, 2, S, 3)).copy()
    mu = k_mean(k)
    assert (mu == np.float32((S - 1) / 2)).all()


def test_mean_exact_rational_on_small_inputs():
    k = bf16_values((1, 2, 300, 4), 21, scale=2.0)
    mu = k_mean(k)
    for h in range(2):
        for d in range(4):
            total = sum(Fraction(float(t)) for t in k[0, h, :, d])
            # exact sum -> float64 -> / n in float64 -> float32
            want = np.float32(float(total) / 300)
            assert mu[0, h, d] == want


def test_mean_matches_numpy_float64_mean():
    k = bf16_values((2, 3, 513, 16), 4)
    mu = k_mean(k)
    ref = k.astype(np.float64).mean(axis=2).astype(np.float32)
    assert (mu == ref).all()


def test_mean_translation_and_valid_count():
    k = bf16_values((1, 1, 128, 8), 8)
    c = np.float32(0.5)
    mu0 = k_mean(k)
    mu1 = k_mean(k + c)
    assert np.allclose(mu1 - mu0, 0.5, atol=1e-6)
    vbs = np.array([64, 10], dtype=np.int32)
    kz = k.copy()
    kz[0, 0, 74:] = 0
    mu2 = k_mean(kz, vbs)
    ref = kz[0, 0, :74].astype(np.float64).mean(axis=0).astype(np.float32)
    assert (mu2[0, 0] == ref).all()
