"""Pins of the oracle's attention, exact attention and merge (CPU only).

References used, none of them the oracle itself:
* torch.nn.functional.scaled_dot_product_attention in float64 on CPU (a
  library routine; "[attention-int8] ..." section 5 uses SDPA as the yardstick),
* scipy.special.logsumexp for the LSE,
* pure-Python brute force on tiny inputs,
* closed forms: one key, zero queries, a constant bias, a fully masked row,
* invariants stated on the pages: K centring is a softmax-invariant shift
  ("minimax_h3_sparse_int8", module description) and two partial softmaxes
  merge exactly through their LSEs ("int8_attention: masked path costs ~1.8x
  unmasked, ...", Question 2; "Add optional forward LSE output", split-K
  combine).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import attention, exact_attention, merge, quantize, k_mean, quantize_and_attend


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def sdpa64(q, k, v, sm_scale, bias=None, allowed=None):
    """torch SDPA in float64 with an additive mask (bias and -inf)."""
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(t, dtype=np.float64)) for t in (q, k, v))
    mask = torch.zeros(q.shape[2], k.shape[2], dtype=torch.float64)
    if bias is not None:
        mask = mask + torch.from_numpy(np.asarray(bias, np.float64))[None, :]
    if allowed is not None:
        mask = mask.masked_fill(~torch.from_numpy(allowed), float("-inf"))
    return F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=sm_scale).numpy()


def codes_as_values(shape, seed):
    return np.random.default_rng(seed).integers(-127, 128, size=shape).astype(np.int8)


@pytest.mark.parametrize("D", [8, 64])
def test_attention_equals_sdpa_when_scales_are_one(D):
    qc = codes_as_values((1, 2, 40, D), 1)
    kc = codes_as_values((1, 2, 70, D), 2)
    v = rnd((1, 2, 70, D), 3)
    one_q = np.ones((1, 2, 40), np.float32)
    one_k = np.ones((1, 2, 70), np.float32)
    bias = rnd(70, 4)
    sm = 1.0 / 997.0
    o, lse = attention(qc, one_q, kc, one_k, v, sm_scale=sm, bias=bias)
    ref = sdpa64(qc, kc, v, sm, bias)
    assert np.abs(o - ref).max() < 1e-12
    logits = sm * np.einsum("bhid,bhjd->bhij", qc.astype(np.float64), kc.astype(np.float64)) + bias
    assert np.abs(lse - scipy.special.logsumexp(logits, axis=-1)).max() < 1e-12


def test_attention_brute_force_python_loops():
    qc = codes_as_values((1, 1, 3, 2), 7)
    kc = codes_as_values((1, 1, 5, 2), 8)
    qs = np.array([[[0.01, 0.02, 0.005]]], np.float32)
    ks = np.array([[[0.03, 0.01, 0.02, 0.015, 0.04]]], np.float32)
    v = rnd((1, 1, 5, 2), 9)
    vsc = np.array([[2.0, 0.5]])
    bias = [0.0, -1.0, 0.5, -3.0, 0.25]
    sm = 0.7
    o, lse = attention(qc, qs, kc, ks, v, sm_scale=sm, bias=bias, v_scale=vsc)
    for i in range(3):
        logits = []
        for j in range(5):
            dot = sum(float(qc[0, 0, i, d]) * float(qs[0, 0, i]) * float(kc[0, 0, j, d]) *
                      float(ks[0, 0, j]) for d in range(2))
            logits.append(sm * dot + bias[j])
        m = max(logits)
        w = [math.exp(t - m) for t in logits]
        tot = sum(w)
        for d in range(2):
            want = vsc[0, d] * sum(w[j] * v[0, 0, j, d] for j in range(5)) / tot
            assert abs(o[0, 0, i, d] - want) < 1e-12
        assert abs(lse[0, 0, i] - (m + math.log(tot))) < 1e-12


def test_per_block_scales_expand_to_rows():
    qc = codes_as_values((1, 1, 100, 16), 1)
    kc = codes_as_values((1, 1, 130, 16), 2)
    v = rnd((1, 1, 130, 16), 3)
    qsb = np.array([[[0.01, 0.02]]], np.float32)
    ksb = np.array([[[0.03, 0.01, 0.02]]], np.float32)
    o, lse = attention(qc, qsb, kc, ksb, v, granularity="block64")
    qst = np.repeat(qsb, 64, axis=2)[:, :, :100]
    kst = np.repeat(ksb, 64, axis=2)[:, :, :130]
    o2, lse2 = attention(qc, qst, kc, kst, v, granularity="token")
    assert np.abs(o - o2).max() < 1e-14 and np.abs(lse - lse2).max() < 1e-12


def test_single_key_gives_that_value():
    qc = codes_as_values((1, 1, 4, 8), 1)
    kc = codes_as_values((1, 1, 1, 8), 2)
    qs = np.full((1, 1, 4), 0.01, np.float32)
    ks = np.full((1, 1, 1), 0.02, np.float32)
    v = rnd((1, 1, 1, 8), 3)
    vsc = np.abs(rnd((1, 8), 4)) + 0.5
    o, lse = attention(qc, qs, kc, ks, v, sm_scale=0.3, v_scale=vsc)
    assert np.abs(o - v * vsc[0]).max() < 1e-14
    s00 = 0.3 * (qc[0, 0].astype(np.float64) * np.float64(np.float32(0.01))) @ (
        kc[0, 0, 0].astype(np.float64) * np.float64(np.float32(0.02)))
    assert np.abs(lse[0, 0] - s00).max() < 1e-12


def test_zero_query_gives_mean_of_v_and_log_count():
    qc = np.zeros((1, 1, 3, 8), np.int8)
    kc = codes_as_values((1, 1, 37, 8), 2)
    v = rnd((1, 1, 37, 8), 3)
    o, lse = attention(qc, np.ones((1, 1, 3), np.float32), kc, np.ones((1, 1, 37), np.float32), v)
    assert np.abs(o - v.mean(axis=2, keepdims=True)).max() < 1e-14
    assert np.abs(lse - math.log(37)).max() < 1e-13


def test_constant_bias_shifts_lse_only():
    qc = codes_as_values((1, 2, 9, 16), 1)
    kc = codes_as_values((1, 2, 33, 16), 2)
    v = rnd((1, 2, 33, 16), 3)
    qs = np.full((1, 2, 9), 0.01, np.float32)
    ks = np.full((1, 2, 33), 0.01, np.float32)
    o0, l0 = attention(qc, qs, kc, ks, v)
    o1, l1 = attention(qc, qs, kc, ks, v, bias=np.full(33, -2.5))
    assert np.abs(o1 - o0).max() < 1e-13
    assert np.abs(l1 - (l0 - 2.5)).max() < 1e-12


def test_fully_masked_rows_give_zero_and_minus_inf():
    qc = codes_as_values((1, 1, 128, 8), 1)
    kc = codes_as_values((1, 1, 128, 8), 2)
    v = rnd((1, 1, 128, 8), 3)
    bm = np.ones((1, 1, 2, 2), bool)
    bm[0, 0, 1, :] = False          # second query tile sees nothing
    bm[0, 0, 0, 1] = False          # first query tile sees only key tile 0
    s1 = np.full((1, 1, 128), 0.01, np.float32)
    o, lse = attention(qc, s1, kc, s1, v, block_mask=bm)
    assert (o[0, 0, 64:] == 0).all() and np.isneginf(lse[0, 0, 64:]).all()
    ref, _ = attention(qc[:, :, :64], s1[:, :, :64], kc[:, :, :64], s1[:, :, :64], v[:, :, :64])
    assert np.abs(o[0, 0, :64] - ref[0, 0]).max() < 1e-14


def test_validity_masks_partial_key_tile_and_pads_query_rows():
    qc = codes_as_values((1, 1, 128, 8), 1)
    kc = codes_as_values((1, 1, 128, 8), 2)
    v = rnd((1, 1, 128, 8), 3)
    s1 = np.full((1, 1, 128), 0.02, np.float32)
    vbs = np.array([64, 37], np.int32)
    o, lse = attention(qc, s1, kc, s1, v, kv_valid=vbs)
    ref, lref = attention(qc[:, :, :101], s1[:, :, :101], kc[:, :, :101], s1[:, :, :101],
                          v[:, :, :101])
    assert np.abs(o[0, 0, :101] - ref[0, 0]).max() < 1e-14
    assert np.abs(lse[0, 0, :101] - lref[0, 0]).max() < 1e-12
    assert (o[0, 0, 101:] == 0).all() and np.isneginf(lse[0, 0, 101:]).all()


def test_block_mask_matches_sdpa_with_expanded_mask():
    rng = np.random.default_rng(5)
    qc = codes_as_values((1, 2, 192, 8), 1)
    kc = codes_as_values((1, 2, 256, 8), 2)
    v = rnd((1, 2, 256, 8), 3)
    bm = rng.random((1, 2, 3, 4)) < 0.5
    bm[..., 0] = True
    o, _ = attention(qc, np.ones((1, 2, 192), np.float32), kc, np.ones((1, 2, 256), np.float32), v,
                     sm_scale=0.01, block_mask=bm)
    for h in range(2):
        allowed = np.repeat(np.repeat(bm[0, h], 64, axis=0), 64, axis=1)
        ref = sdpa64(qc[:, h:h + 1], kc[:, h:h + 1], v[:, h:h + 1], 0.01, allowed=allowed)
        assert np.abs(o[:, h:h + 1] - ref).max() < 1e-12


def test_exact_attention_matches_sdpa_and_centring_is_invariant():
    q = rnd((1, 2, 30, 16), 1)
    k = rnd((1, 2, 50, 16), 2)
    v = rnd((1, 2, 50, 16), 3)
    mu = rnd((1, 2, 1, 16), 4, 3.0)
    sm = 16 ** -0.5
    o, lse = exact_attention(q, k, v)
    assert np.abs(o - sdpa64(q, k, v, sm)).max() < 1e-12
    oc, lsec = exact_attention(q, k - mu, v)
    assert np.abs(oc - o).max() < 1e-12
    shift = -sm * np.einsum("bhid,bhd->bhi", q, mu[:, :, 0])
    assert np.abs(lsec - (lse + shift)).max() < 1e-11


def test_merge_of_key_split_equals_whole():
    q = rnd((1, 3, 20, 16), 1)
    k = rnd((1, 3, 90, 16), 2)
    v = rnd((1, 3, 90, 16), 3)
    bias = np.log(np.linspace(1.0, 1e-4, 90))
    o, lse = exact_attention(q, k, v, bias=bias)
    core = slice(0, 55)
    skirt = slice(55, 90)
    o1, l1 = exact_attention(q, k[:, :, core], v[:, :, core], bias=bias[core])
    o2, l2 = exact_attention(q, k[:, :, skirt], v[:, :, skirt], bias=bias[skirt])
    om, lm = merge(o1, l1, o2, l2)
    assert np.abs(om - o).max() < 1e-12 and np.abs(lm - lse).max() < 1e-12


def test_merge_with_empty_partials():
    o1 = rnd((1, 1, 4, 8), 1)
    l1 = rnd((1, 1, 4), 2)
    dead = np.full((1, 1, 4), -np.inf)
    om, lm = merge(o1, l1, np.zeros_like(o1), dead)
    assert np.abs(om - o1).max() < 1e-15 and np.abs(lm - l1).max() < 1e-15
    om2, lm2 = merge(np.zeros_like(o1), dead, np.zeros_like(o1), dead)
    assert (om2 == 0).all() and np.isneginf(lm2).all()


def test_quantized_path_is_close_to_exact_attention():
    """The whole INT8 path against exact float64 attention: the mean absolute
    error stays well under the 0.01-0.02 that "[attention-int8] ..." section 5
    expects of INT8 attention."""
    g = torch.Generator().manual_seed(0)
    q = torch.randn(1, 2, 256, 64, generator=g).to(torch.bfloat16).float().numpy()
    k = (torch.randn(1, 2, 256, 64, generator=g) + 2).to(torch.bfloat16).float().numpy()
    v = torch.randn(1, 2, 256, 64, generator=g).to(torch.bfloat16).float().numpy()
    o, lse, _ = quantize_and_attend(q, k, v)
    oe, _ = exact_attention(q, k, v)
    assert np.abs(o - oe).mean() < 2e-3


def test_centring_keeps_output_and_shifts_lse_in_quantized_path():
    g = torch.Generator().manual_seed(1)
    q = torch.randn(1, 1, 64, 32, generator=g).to(torch.bfloat16).float().numpy()
    k = torch.randn(1, 1, 200, 32, generator=g).to(torch.bfloat16).float().numpy()
    v = torch.randn(1, 1, 200, 32, generator=g).to(torch.bfloat16).float().numpy()
    mu = k_mean(k)
    assert mu.shape == (1, 1, 32)
    o1, l1, _ = quantize_and_attend(q, k, v, center_k=True)
    o0, l0, _ = quantize_and_attend(q, k, v, center_k=False)
    # both approximate the same attention; LSEs differ by about -sm*q.mu
    assert np.abs(o1 - o0).mean() < 5e-3
    shift = -(32 ** -0.5) * np.einsum("bhid,bhd->bhi", q.astype(np.float64), mu.astype(np.float64))
    assert np.abs((l1 - l0) - shift).max() < 5e-2
