"""RMSNorm + RoPE prologue on the GPU against the oracle.

The prologue of "Feature Request: Direct int8 Q/K passthrough between Comfy
Kitchen and SageAttention" (maintainer's reply: rms_rope, apply_rope,
rms_rope_split_half) runs inside the quantize kernel and inside the fused-Q
attention kernel. Codes, scales and the K mean must equal the oracle's bit for
bit (the oracle follows the kernels' fixed fp32 order); the fused attention
must equal prologue-quantize + attention bit for bit and meet the oracle's
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from util import assert_lse_close, assert_out_close, ensure_built, to_np
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


@pytest.mark.parametrize("name,kw,norm,rope,qp,kp", CASES)
def test_quantize_with_prologue_bit_exact(name, kw, norm, rope, qp, kp):
    import int8_qk_quantized_gb300 as ia
    wl, inp, pro, opro = setup(name, kw, norm, rope, qp, kp)
    q8, qs, k8, ks, mu = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity,
                                        kv_valid=inp.kv_valid, return_mean=True, prologue=pro)
    torch.cuda.synchronize()
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    rqc, rqs, rkc, rks, rmu = _oracle_quant(inp, wl, vbs, opro)
    for got, ref, n in ((q8, rqc, "q codes"), (qs, rqs, "q scales"), (k8, rkc, "k codes"),
                        (ks, rks, "k scales"), (mu, rmu, "k mean")):
        g = to_np(got)
        assert np.array_equal(g, ref), f"{n}: {np.count_nonzero(g != ref)} mismatches"


def _oracle_quant(inp, wl, vbs, opro):
    pr = dict(opro)
    common = dict(dtype=pr["dtype"], eps=pr["eps"], rope=pr["rope"], cos=pr["cos"], sin=pr["sin"])
    qv = oracle.qk_prologue(to_np(inp.q), norm_weight=pr["q_norm_weight"], pos0=pr["q_pos0"], **common)
    kv = oracle.qk_prologue(to_np(inp.k), norm_weight=pr["k_norm_weight"], pos0=pr["k_pos0"], **common)
    if vbs is not None:
        kv = np.where(oracle.row_validity(wl.Sk, vbs)[None, None, :, None], kv, 0)
        qv = np.where(oracle.row_validity(wl.Sq, vbs)[None, None, :, None], qv, 0)
    mu = oracle.k_mean(kv, vbs)
    qc, qs = oracle.quantize(qv, None, wl.granularity, vbs if wl.Sq == wl.Sk else None)
    kc, ks = oracle.quantize(kv, mu, wl.granularity, vbs)
    return qc, qs, kc, ks, mu


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
