"""Pins of the oracle's general attention mask (CPU only).

The mask forms are those of "int8_attention: masked path costs ~1.8x
unmasked, and a request for optional return_lse", The measurement: fp32,
bf16 and fp16 additive masks and a bool mask, shaped [1,1,1,K] or expanded
to [1,1,Q,K]; the bool mask is True where a key is kept. References: pure
Python loops, torch float64 SDPA (its bool and float ``attn_mask``), and
closed forms.
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import attention, exact_attention


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def codes(shape, seed):
    return np.random.default_rng(seed).integers(-127, 128, size=shape).astype(np.int8)


def test_full_float_mask_brute_force():
    B, H, Sq, Sk, D = 2, 2, 3, 5, 4
    qc, kc = codes((B, H, Sq, D), 1), codes((B, H, Sk, D), 2)
    qs = np.abs(rnd((B, H, Sq), 3, 0.01)).astype(np.float32) + 1e-3
    ks = np.abs(rnd((B, H, Sk), 4, 0.01)).astype(np.float32) + 1e-3
    v = rnd((B, H, Sk, D), 5)
    mask = rnd((B, H, Sq, Sk), 6, 2.0)
    mask[0, 1, 2, 3] = -np.inf
    sm = 0.45
    o, lse = attention(qc, qs, kc, ks, v, sm_scale=sm, mask=mask)
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                t = []
                for j in range(Sk):
                    dot = sum(float(qc[b, h, i, d]) * float(qs[b, h, i]) * float(kc[b, h, j, d]) *
                              float(ks[b, h, j]) for d in range(D))
                    t.append(sm * dot + float(mask[b, h, i, j]))
                m = max(t)
                w = [math.exp(x - m) for x in t]
                for d in range(D):
                    want = sum(w[j] * v[b, h, j, d] for j in range(Sk)) / sum(w)
                    assert abs(o[b, h, i, d] - want) < 1e-12
                assert abs(lse[b, h, i] - (m + math.log(sum(w)))) < 1e-12


def test_broadcast_forms_match_sdpa():
    """[1,1,1,K], [1,1,Q,K] expanded, [B,1,1,K] and [1,H,Q,K] masks against
    torch SDPA in float64 with the same broadcast attn_mask."""
    B, H, Sq, Sk, D = 2, 3, 17, 29, 8
    q, k, v = rnd((B, H, Sq, D), 1), rnd((B, H, Sk, D), 2), rnd((B, H, Sk, D), 3)
    for shape in [(1, 1, 1, Sk), (1, 1, Sq, Sk), (B, 1, 1, Sk), (1, H, Sq, Sk), (B, H, Sq, Sk)]:
        mask = rnd(shape, 4, 1.5)
        o, lse = exact_attention(q, k, v, sm_scale=0.3, mask=mask)
        ref = F.scaled_dot_product_attention(*(torch.from_numpy(t) for t in (q, k, v)),
                                             attn_mask=torch.from_numpy(mask), scale=0.3).numpy()
        assert np.abs(o - ref).max() < 1e-12, shape
        expanded = np.broadcast_to(mask, (B, H, Sq, Sk))
        s = 0.3 * np.einsum("bhqd,bhkd->bhqk", q, k) + expanded
        want = np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1)) + s.max(-1)
        assert np.abs(lse - want).max() < 1e-12, shape


def test_bool_mask_is_zero_or_minus_inf_and_matches_sdpa():
    B, H, Sq, Sk, D = 1, 2, 9, 40, 8
    q, k, v = rnd((B, H, Sq, D), 1), rnd((B, H, Sk, D), 2), rnd((B, H, Sk, D), 3)
    keep = np.random.default_rng(5).random((1, H, Sq, Sk)) > 0.3
    keep[0, 0, 4, :] = True
    o_b, l_b = exact_attention(q, k, v, mask=keep)
    o_f, l_f = exact_attention(q, k, v, mask=np.where(keep, 0.0, -np.inf))
    assert np.array_equal(o_b, o_f) and np.array_equal(l_b, l_f)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(t) for t in (q, k, v)),
                                         attn_mask=torch.from_numpy(keep)).numpy()
    assert np.abs(o_b - ref).max() < 1e-12


def test_per_key_mask_equals_bias_and_row_constant_shifts_lse():
    qc, kc = codes((1, 2, 7, 16), 1), codes((1, 2, 33, 16), 2)
    qs = np.full((1, 2, 7), 0.01, np.float32)
    ks = np.full((1, 2, 33), 0.02, np.float32)
    v = rnd((1, 2, 33, 16), 3)
    bias = rnd(33, 4)
    o1, l1 = attention(qc, qs, kc, ks, v, bias=bias)
    o2, l2 = attention(qc, qs, kc, ks, v, mask=bias.reshape(1, 1, 1, 33))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o0, l0 = attention(qc, qs, kc, ks, v)
    c = rnd((1, 2, 7, 1), 5, 3.0)
    o3, l3 = attention(qc, qs, kc, ks, v, mask=c)
    assert np.abs(o3 - o0).max() < 1e-13
    assert np.abs(l3 - (l0 + c[..., 0])).max() < 1e-12


def test_all_false_row_gives_zero_and_minus_inf():
    qc, kc = codes((1, 1, 4, 8), 1), codes((1, 1, 70, 8), 2)
    qs = np.full((1, 1, 4), 0.01, np.float32)
    ks = np.full((1, 1, 70), 0.01, np.float32)
    v = rnd((1, 1, 70, 8), 3)
    keep = np.ones((1, 1, 4, 70), bool)
    keep[0, 0, 2] = False
    o, lse = attention(qc, qs, kc, ks, v, mask=keep)
    assert np.all(o[0, 0, 2] == 0.0) and lse[0, 0, 2] == -np.inf
    assert np.all(np.isfinite(lse[0, 0, [0, 1, 3]]))
