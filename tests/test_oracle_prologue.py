"""Pins of the oracle's RMSNorm + RoPE prologue (CPU only).

The prologue is the step "Feature Request: Direct int8 Q/K passthrough
between Comfy Kitchen and SageAttention", maintainer's reply, puts between
the projections and attention (``rms_rope``, ``apply_rope``,
``rms_rope_split_half``). References: torch ``rms_norm`` in float64, complex
multiplication in complex128, and invariants of a rotation.
"""
import numpy as np
import pytest
import torch

from oracle import exact_attention, qk_prologue, quantize_and_attend, round_to_16bit
from workloads import norm_weight, rope_tables


def rnd16(shape, seed, dtype, scale=1.0):
    x = np.random.default_rng(seed).standard_normal(shape).astype(np.float32) * np.float32(scale)
    return round_to_16bit(x, dtype)


def ulp16(x, dtype):
    """Spacing of the 16-bit type at |x| (relative 2^-7 bf16, 2^-10 fp16)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - (7 if dtype == "bf16" else 10))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("scale,eps", [(3.0, 1e-6), (1e-3, 1e-6)])  # eps matters in the second
def test_rmsnorm_matches_torch_float64(dtype, scale, eps):
    x = rnd16((1, 2, 37, 64), 1, dtype, scale)
    w = norm_weight(64, 2)
    y = qk_prologue(x, dtype=dtype, norm_weight=w, eps=eps)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (64,),
                                       weight=torch.from_numpy(w.astype(np.float64)),
                                       eps=eps).numpy()
    assert np.all(np.abs(y - ref) <= ulp16(ref, dtype))           # within one 16-bit ulp
    assert np.mean(y == round_to_16bit(ref.astype(np.float32), dtype)) > 0.99


def test_zero_row_stays_zero_and_scale_invariance():
    x = rnd16((1, 1, 4, 64), 3, "fp16")
    w = np.ones(64, np.float32)
    z = x.copy()
    z[0, 0, 1] = 0
    assert np.all(qk_prologue(z, dtype="fp16", norm_weight=w, eps=1e-6)[0, 0, 1] == 0)
    y = qk_prologue(x, dtype="fp16", norm_weight=w, eps=0.0)
    y2 = qk_prologue(x * np.float32(4.0), dtype="fp16", norm_weight=w, eps=0.0)
    assert np.array_equal(y, y2)  # RMSNorm without eps is invariant to a power-of-two scale


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_interleaved_rope_is_complex_rotation(dtype):
    D, S = 64, 50
    x = rnd16((1, 2, S, D), 4, dtype)
    cos, sin = rope_tables(100, D)
    y = qk_prologue(x, dtype=dtype, rope="interleaved", cos=cos, sin=sin, pos0=7)
    z = (x[..., 0::2].astype(np.float64) + 1j * x[..., 1::2].astype(np.float64)) * \
        (cos[7:7 + S].astype(np.float64) + 1j * sin[7:7 + S].astype(np.float64))
    ref = np.empty_like(y, dtype=np.float64)
    ref[..., 0::2], ref[..., 1::2] = z.real, z.imag
    assert np.all(np.abs(y - ref) <= ulp16(ref, dtype) + 1e-6)


def test_rotation_sign_identity_and_pair_norms():
    D = 16
    x = rnd16((1, 1, 3, D), 5, "fp16")
    one, zero = np.ones((3, D // 2), np.float32), np.zeros((3, D // 2), np.float32)
    assert np.array_equal(qk_prologue(x, dtype="fp16", rope="split_half", cos=one, sin=zero), x)
    q = qk_prologue(x, dtype="fp16", rope="interleaved", cos=zero, sin=one)
    assert np.array_equal(q[..., 0::2], -x[..., 1::2]) and np.array_equal(q[..., 1::2], x[..., 0::2])
    cos, sin = rope_tables(3, D)
    y = qk_prologue(x, dtype="fp16", rope="split_half", cos=cos, sin=sin)
    n0 = x[..., :D // 2].astype(np.float64) ** 2 + x[..., D // 2:].astype(np.float64) ** 2
    n1 = y[..., :D // 2].astype(np.float64) ** 2 + y[..., D // 2:].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=4e-3, atol=1e-6)


def test_split_half_is_interleaved_on_permuted_channels():
    D = 64
    x = rnd16((2, 1, 9, D), 6, "bf16")
    w = norm_weight(D, 7)
    cos, sin = rope_tables(20, D)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # interleaved -> halves
    a = qk_prologue(x, dtype="bf16", norm_weight=w, rope="interleaved", cos=cos, sin=sin, pos0=3)
    b = qk_prologue(x[..., perm], dtype="bf16", norm_weight=w[perm], rope="split_half",
                    cos=cos, sin=sin, pos0=3)
    assert np.array_equal(a[..., perm], b)


def test_prologue_path_close_to_exact_attention_on_normed_roped_inputs():
    D, S = 64, 96
    q, k, v = (rnd16((1, 2, S, D), s, "bf16") for s in (8, 9, 10))
    wq, wk = norm_weight(D, 11), norm_weight(D, 12)
    cos, sin = rope_tables(S, D)
    pro = dict(dtype="bf16", q_norm_weight=wq, k_norm_weight=wk, eps=1e-6, rope="split_half",
               cos=cos, sin=sin)
    o, lse, _ = quantize_and_attend(q, k, v, prologue=pro)

    def ref64(x, w):
        t = torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (D,),
                                         weight=torch.from_numpy(w.astype(np.float64)), eps=1e-6)
        a, b = t[..., :D // 2], t[..., D // 2:]
        c, s = torch.from_numpy(cos.astype(np.float64)), torch.from_numpy(sin.astype(np.float64))
        return torch.cat([a * c - b * s, a * s + b * c], -1).numpy()

    oe, le = exact_attention(ref64(q, wq), ref64(k, wk), v)
    assert np.abs(o - oe).mean() < 1e-2


def test_rmsnorm_uses_the_exact_sum_of_squares():
    """The oracle's RMSNorm is the mathematics: the sum of squares exact,
    rounded once to fp32, then r = 1/sqrt(ss/D + eps) and y = (x r) w in fp32
    and one rounding to the 16-bit type, here written out with Python's exact
    rationals for the sum. On thousands of random fp16 rows it must agree bit
    for bit; a running fp32 sum (the GPU kernels' documented order) gives a
    different 16-bit row on some of them, so the check tells the two apart."""
    from fractions import Fraction
    from kernel_order import prologue_kernel_order
    D, n = 128, 4000
    x = rnd16((1, 1, n, D), 17, "fp16", 2.0)
    w = norm_weight(D, 18)
    eps = np.float32(1e-6)
    ss = np.array([np.float32(float(sum(Fraction(float(v)) ** 2 for v in row)))  # one rounding
                   for row in x.reshape(n, D)], np.float32)
    ms = (ss / np.float32(D)).astype(np.float32)
    r = (np.float32(1) / np.sqrt((ms + eps).astype(np.float32))).astype(np.float32)
    want = round_to_16bit(((x * r.reshape(1, 1, n, 1)).astype(np.float32) * w).astype(np.float32),
                          "fp16")
    got = qk_prologue(x, dtype="fp16", norm_weight=w, eps=1e-6)
    assert np.array_equal(got, want)
    kern = prologue_kernel_order(x, dtype="fp16", norm_weight=w, eps=1e-6)
    assert np.any(kern != want)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_final_rounding_is_the_library_rounding(dtype):
    """With neither norm nor rotation the prologue is its last step alone, the
    rounding to the 16-bit type: it must equal torch's bf16 / numpy's fp16
    conversion bit for bit, ties, subnormals and overflow included."""
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(4096) * np.exp2(rng.integers(-30, 30, 4096))).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65520.0, 7e4, 1e-8, 6.1e-5, 3e-38, 1e38, 3.4e38,
                     1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11],
                    np.float32)
    x = np.concatenate([x, edge, -edge]).reshape(1, 1, -1, 1)
    x = np.repeat(x, 2, axis=-1)                               # D = 2: one rotation pair, unused
    got = qk_prologue(x, dtype=dtype)
    want = round_to_16bit(x, dtype)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_exact_sum_against_rational_arithmetic():
    """The exact summation the K mean and the RMSNorm use, against Python's
    exact rational arithmetic: heavy cancellation, tiny and huge terms."""
    from fractions import Fraction
    from oracle import exact_sum
    rng = np.random.default_rng(7)
    for trial in range(20):
        x = rng.standard_normal(300) * np.exp2(rng.integers(-60, 60, 300))
        x = np.concatenate([x, -x[:150] * (1 + 2.0 ** -40), [2.0 ** -1074, 1e300, -1e300]])
        want = float(sum((Fraction(float(v)) for v in x), Fraction(0)))  # correctly rounded
        assert exact_sum(x, 53) == want
    # binary32: integer sums below 2^53 are exact in float64, then rounded once
    y = np.array([2.0 ** 24, 1.0, 1.0, 1.0], np.float64)
    assert exact_sum(y, 24) == float(np.float32(2.0 ** 24 + 3))
    assert exact_sum(np.array([2.0 ** 24, 1.0]), 24) == 2.0 ** 24     # tie to even
    assert exact_sum(np.array([2.0 ** 24, 3.0]), 24) == 2.0 ** 24 + 4  # tie to even, upward
