"""The RMSNorm + RoPE prologue with the GPU kernels' own fp32 summation order.

This is not the oracle. The oracle (``oracle.qk_prologue``) sums the squares
of a row exactly and rounds once, which is what the method's RMSNorm means.
The kernels sum them in a fixed fp32 order instead, documented in
``include/ia.h`` beside ``ia_qk_prologue`` as part of this library's
contract: the squares of each 8 consecutive channels in index order, then the
D/8 partial sums added pairwise (t with t + n/2) until one remains. This
helper restates that documented order so that a test can check the kernels
against their own specification bit for bit; the parity tests compare them
with the oracle within a stated bound.
"""
import numpy as np

from oracle import round_to_16bit


def prologue_kernel_order(x, *, dtype, norm_weight=None, eps=1e-6, rope=None, cos=None,
                          sin=None, pos0=0):
    """float32 [B,H,S,D] holding 16-bit values -> the kernels' prologue output."""
    B, H, S, D = x.shape
    y = np.asarray(x, dtype=np.float32).copy()
    if norm_weight is not None:
        w = np.asarray(norm_weight, dtype=np.float32)
        sq = (y * y).astype(np.float32)
        part = sq[..., 0::8].copy()
        for j in range(1, 8):
            part = (part + sq[..., j::8]).astype(np.float32)
        n = D // 8
        while n > 1:
            half = n // 2
            part = (part[..., :half] + part[..., half:n]).astype(np.float32)
            n = half
        ms = (part[..., 0] / np.float32(D)).astype(np.float32)
        rr = (np.float32(1) / np.sqrt((ms + np.float32(eps)).astype(np.float32))).astype(np.float32)
        y = ((y * rr[..., None]).astype(np.float32) * w).astype(np.float32)
    if rope is not None:
        c = np.asarray(cos, dtype=np.float32)[pos0:pos0 + S]
        sn = np.asarray(sin, dtype=np.float32)[pos0:pos0 + S]
        if rope == "interleaved":
            a, bb = y[..., 0::2], y[..., 1::2]
        else:
            a, bb = y[..., :D // 2], y[..., D // 2:]
        a2 = ((a * c).astype(np.float32) - (bb * sn).astype(np.float32)).astype(np.float32)
        b2 = ((a * sn).astype(np.float32) + (bb * c).astype(np.float32)).astype(np.float32)
        y = np.empty_like(y)
        if rope == "interleaved":
            y[..., 0::2], y[..., 1::2] = a2, b2
        else:
            y[..., :D // 2], y[..., D // 2:] = a2, b2
    return round_to_16bit(y, dtype)
