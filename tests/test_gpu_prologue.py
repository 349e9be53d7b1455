"""RMSNorm + RoPE prologue on the GPU against the oracle, and against the
library's documented summation order.

The prologue of "Feature Request: Direct int8 Q/K passthrough between Comfy
Kitchen and SageAttention" (maintainer's reply: rms_rope, apply_rope,
rms_rope_split_half) runs inside the quantize kernel and inside the fused-Q
attention kernel.

Against the oracle, whose RMSNorm takes the exact sum of squares rounded once:
the 16-bit rows the kernels quantize lie within one 16-bit ulp of the
oracle's, plus 2^-18 of the row's largest value where the rotation cancels
(the two sums of squares differ by a few fp32 ulps, which moves the fp32
values before the last rounding by about 2^-20 relative); they are the
documented-order rows below, which the kernels are shown to reproduce bit
for bit. Q codes and scales equal the oracle's on
every row (per-64-row block: every block) whose 16-bit values agree with it,
codes are otherwise within two steps and scales within one 16-bit spacing
(relative 2^-7 for bf16, 2^-10 for fp16: one ulp of amax); the K mean moves
by at most the mean ulp of its column; attention output and LSE meet the
spec tolerances. The reason for the bounds: one ulp in x' and in amax
moves x' * 127 / amax by less than two.

Against the library's contract: the kernels sum the squares in the fixed
fp32 order documented in include/ia.h (tests/kernel_order.py restates it);
codes, scales and K mean computed from those rows must match bit for bit.
The fused-Q attention must equal prologue-quantize + attention bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from util import assert_lse_close, assert_out_close, ensure_built, to_np
from kernel_order import prologue_kernel_order
from workloads import WORKLOADS, make_inputs, norm_weight, rope_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


CASES = [
    # name, workload overrides, norm, rope, q_pos0, k_pos0
    ("anima4k", dict(H=2, Sq=700, Sk=1000), True, "split_half", 0, 0),
    ("anima4k", dict(H=2, Sq=300, Sk=900), True, "interleaved", 100, 7),
    ("anima4k", dict(H=2, Sq=333, Sk=500), True, None, 0, 0),
    ("sdxl", dict(H=2, Sq=600, Sk=700), False, "interleaved", 0, 0),
    ("sdxl", dict(H=2, Sq=600, Sk=700, granularity="token"), True, "split_half", 5, 5),
    ("sparse", dict(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2), True, "split_half", 0, 0),
    ("sparse", dict(H=1, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2, granularity="block64",
                    dtype="fp16"), True, "interleaved", 0, 0),
]


def setup(name, kw, norm, rope, qp, kp):
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    P = max(wl.Sq + qp, wl.Sk + kp) + 3
    cos, sin = rope_tables(P, wl.D)
    wq, wk = (norm_weight(wl.D, 21), norm_weight(wl.D, 22)) if norm else (None, None)
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    pro = ia.make_prologue(q_norm_weight=dev(wq), k_norm_weight=dev(wk), eps=1e-6, rope=rope,
                           cos=dev(cos), sin=dev(sin), q_pos0=qp, k_pos0=kp)
    opro = dict(dtype=wl.dtype, q_norm_weight=wq, k_norm_weight=wk, eps=1e-6, rope=rope,
                cos=cos, sin=sin, q_pos0=qp, k_pos0=kp)
    return wl, inp, pro, opro


def _rows(inp, wl, vbs, opro, fn):
    """Q and K rows after the prologue `fn` (the oracle's or the documented
    order), padding rows zero."""
    pr = dict(opro)
    common = dict(dtype=pr["dtype"], eps=pr["eps"], rope=pr["rope"], cos=pr["cos"], sin=pr["sin"])
    qv = fn(to_np(inp.q), norm_weight=pr["q_norm_weight"], pos0=pr["q_pos0"], **common)
    kv = fn(to_np(inp.k), norm_weight=pr["k_norm_weight"], pos0=pr["k_pos0"], **common)
    if vbs is not None:
        kv = np.where(oracle.row_validity(wl.Sk, vbs)[None, None, :, None], kv, 0)
        qv = np.where(oracle.row_validity(wl.Sq, vbs)[None, None, :, None], qv, 0)
    return qv, kv


def _quant(qv, kv, wl, vbs):
    mu = oracle.k_mean(kv, vbs)
    qc, qs = oracle.quantize(qv, None, wl.granularity, vbs if wl.Sq == wl.Sk else None)
    kc, ks = oracle.quantize(kv, mu, wl.granularity, vbs)
    return qc, qs, kc, ks, mu


def _ulp16(x, dtype):
    """Spacing of the 16-bit type at |x| (0 stays 0 apart: the smallest normal's)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** (-126 if dtype == "bf16" else -14))))
    return 2.0 ** (e - (7 if dtype == "bf16" else 10))


def _gpu_quant(wl, inp, pro):
    import int8_qk_quantized_gb300 as ia
    out = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid,
                         return_mean=True, prologue=pro)
    torch.cuda.synchronize()
    return [to_np(t) for t in out]


@pytest.mark.parametrize("name,kw,norm,rope,qp,kp", CASES)
def test_quantize_with_prologue_documented_order(name, kw, norm, rope, qp, kp):
    """Bit for bit against the quantization of the documented-order rows."""
    wl, inp, pro, opro = setup(name, kw, norm, rope, qp, kp)
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    got = _gpu_quant(wl, inp, pro)
    ref = _quant(*_rows(inp, wl, vbs, opro, prologue_kernel_order), wl, vbs)
    for g, r, n in zip(got, ref, ("q codes", "q scales", "k codes", "k scales", "k mean")):
        assert np.array_equal(g, r), f"{n}: {np.count_nonzero(g != r)} mismatches"


@pytest.mark.parametrize("name,kw,norm,rope,qp,kp", CASES)
def test_quantize_with_prologue_against_oracle(name, kw, norm, rope, qp, kp):
    wl, inp, pro, opro = setup(name, kw, norm, rope, qp, kp)
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    qc, qs, kc, ks, mu = _gpu_quant(wl, inp, pro)
    qo, ko = _rows(inp, wl, vbs, opro, oracle.qk_prologue)
    qk, kk = _rows(inp, wl, vbs, opro, prologue_kernel_order)
    # the rows the kernels quantize: within one 16-bit ulp of the oracle's,
    # plus 2^-18 of the row's largest magnitude for the rotation's cancellation
    for a, o in ((qk, qo), (kk, ko)):
        slack = 2.0 ** -18 * np.abs(o).max(axis=-1, keepdims=True)
        assert np.all(np.abs(a.astype(np.float64) - o) <= _ulp16(o, wl.dtype) + slack)
    rqc, rqs, rkc, rks, rmu = _quant(qo, ko, wl, vbs)
    # Q: equal wherever the rows (blocks) agree; otherwise within the bounds
    same = np.all(qk == qo, axis=-1)                                     # [B,H,Sq]
    if wl.granularity == "block64":
        nb = qs.shape[-1]
        pad = nb * 64 - wl.Sq
        same = np.pad(same, ((0, 0), (0, 0), (0, pad)), constant_values=True)
        same_blk = same.reshape(*same.shape[:2], nb, 64).all(-1)
        same_rows = np.repeat(same_blk, 64, axis=-1)[..., :wl.Sq]
        same_scale = same_blk
    else:
        same_rows = same_scale = same
    assert np.array_equal(qc[same_rows], rqc[same_rows])
    assert np.array_equal(qs[same_scale], rqs[same_scale])
    rel = 2.0 ** (-7 if wl.dtype == "bf16" else -10)
    for c, rc, sc, rsc in ((qc, rqc, qs, rqs), (kc, rkc, ks, rks)):
        assert np.abs(c.astype(np.int32) - rc).max() <= 2
        assert np.all(np.abs(sc.astype(np.float64) - rsc) <= rel * np.abs(rsc) + 1e-30)
    # the K mean: each row moves by at most one ulp, so the mean by at most the
    # column's mean ulp (plus the mean's own fp32 rounding)
    n_valid = wl.Sk if vbs is None else int(oracle.row_validity(wl.Sk, vbs).sum())
    bound = _ulp16(ko, wl.dtype).sum(axis=2) / n_valid + 2.0 ** -23 * np.abs(rmu)
    assert np.all(np.abs(mu.astype(np.float64) - rmu) <= bound)


@pytest.mark.parametrize("name,kw,norm,rope,qp,kp", CASES)
def test_fused_q_prologue_equals_two_pass_and_oracle(name, kw, norm, rope, qp, kp):
    import int8_qk_quantized_gb300 as ia
    wl, inp, pro, opro = setup(name, kw, norm, rope, qp, kp)
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity,
                                    kv_valid=inp.kv_valid, prologue=pro)
    args = dict(block_mask=inp.block_mask, v_scale=inp.v_scale, kv_valid=inp.kv_valid,
                granularity=wl.granularity, return_lse=True, kv_splits=1)
    o2, l2 = ia.attention(q8, k8, qs, ks, inp.v, **args)
    o1, l1 = ia.attention_quant_q(inp.q, k8, ks, inp.v, prologue=pro, **args)
    ia.device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    ro, rl, _ = oracle.quantize_and_attend(
        to_np(inp.q), to_np(inp.k), to_np(inp.v), granularity=wl.granularity, kv_valid=vbs,
        block_mask=None if inp.block_mask is None else to_np(inp.block_mask),
        v_scale=None if inp.v_scale is None else to_np(inp.v_scale), prologue=opro)
    valid = None if vbs is None else oracle.row_validity(wl.Sq, vbs)
    assert_out_close(to_np(o1), ro, valid=valid)
    assert_lse_close(to_np(l1), rl, valid=valid)
