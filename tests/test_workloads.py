"""The seeded input generators: shapes, determinism and the structure each
workload promises (skirt bias end points, band + random tile counts, pads)."""
import math

import numpy as np
import torch

from workloads import (WORKLOADS, band_random_mask, make_inputs, skirt_bias, validity_vector,
                       algorithmic_ops)


def test_skirt_bias_shape_and_end_points():
    b = skirt_bias(33600, 6720)
    assert b.dtype == np.float32 and b.shape == (33600,)
    assert (b[6720:26880] == 0).all()
    assert b[0] == np.float32(math.log(1e-4)) and b[-1] == np.float32(math.log(1e-4))
    assert (np.diff(b[:6720]) >= 0).all() and (np.diff(b[26880:]) <= 0).all()
    assert b[6719] > -1e-6 and b[26880] > -1e-6


def test_band_random_mask_counts():
    m = band_random_mask(3, 128, 64, 16, seed=4)
    assert m.shape == (1, 3, 128, 128)
    assert (m.sum(axis=-1) == 80).all()
    m2 = band_random_mask(3, 128, 64, 16, seed=4)
    assert (m == m2).all()


def test_validity_vector():
    v = validity_vector(1024, 37)
    assert v.dtype == np.int32 and v[-1] == 37 and (v[:-1] == 64).all()


def test_make_inputs_tiny_and_small_sparse():
    inp = make_inputs(WORKLOADS["tiny"])
    assert inp.q.shape == (1, 2, 256, 64) and inp.q.dtype == torch.bfloat16
    again = make_inputs(WORKLOADS["tiny"])
    assert torch.equal(inp.k, again.k)
    wl = WORKLOADS["sparse"].with_(H=2, Sq=512, Sk=512, band_tiles=4, random_tiles=2)
    sp = make_inputs(wl)
    assert sp.block_mask.shape == (1, 2, 8, 8) and sp.kv_valid[-1] == 37
    assert (sp.k[:, :, 7 * 64 + 37:] == 0).all()
    sd = make_inputs(WORKLOADS["sdxl"].with_(Sq=128, Sk=128))
    assert sd.k.dtype == torch.float16
    an = make_inputs(WORKLOADS["anima4k"].with_(Sq=128, Sk=128))
    assert an.v_scale.shape == (16, 128) and an.v.abs().max() <= 1.0


def test_algorithmic_ops():
    assert algorithmic_ops(WORKLOADS["banded"]) == 4 * 56 * 4096 * 33600 * 128
    assert algorithmic_ops(WORKLOADS["sparse"]) == 24 * 1024 * 80 * 64 * 64 * 128 * 4
