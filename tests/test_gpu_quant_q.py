"""Attention with Q quantized inside the kernel, against the two-pass path
and the oracle.

``ia_attention_fwd_quant_q`` quantizes each Q row (or 64-row block) in shared
memory with the same IEEE steps as ``ia_quantize_qk`` ("minimax_h3_sparse_int8",
FastVideo API page, quant_qk_int8), so its output and LSE must equal those of
quantize-then-attend bit for bit, and meet the oracle's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from util import assert_lse_close, assert_out_close, ensure_built, to_np
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


CASES = [
    ("tiny", {}),
    ("sdxl", dict(H=2, Sq=700, Sk=900)),
    ("anima4k", dict(H=2, Sq=1000, Sk=1300)),
    ("banded", dict(H=2, Sq=300, Sk=2500, skirt_width=500)),
    ("sparse", dict(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4)),
    ("sparse", dict(H=1, Sq=1024, Sk=1024, D=64, dtype="fp16", band_tiles=4, random_tiles=2,
                    granularity="block64")),
]


def _run(wl, inp, q=None, **kw):
    import int8_qk_quantized_gb300 as ia
    q = inp.q if q is None else q
    q8, qs, k8, ks = ia.quantize_qk(q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid)
    args = dict(bias=inp.bias, block_mask=inp.block_mask, v_scale=inp.v_scale,
                kv_valid=inp.kv_valid, granularity=wl.granularity, return_lse=True, **kw)
    o2, l2 = ia.attention(q8, k8, qs, ks, inp.v, **args)
    o1, l1 = ia.attention_quant_q(q, k8, ks, inp.v, **args)
    ia.device_status()
    return (o1, l1), (o2, l2)


def _oracle(wl, inp, q=None):
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    o, lse, _ = oracle.quantize_and_attend(
        to_np(inp.q if q is None else q), to_np(inp.k), to_np(inp.v), granularity=wl.granularity,
        kv_valid=vbs, bias=None if inp.bias is None else to_np(inp.bias),
        block_mask=None if inp.block_mask is None else to_np(inp.block_mask),
        v_scale=None if inp.v_scale is None else to_np(inp.v_scale))
    valid = None if inp.kv_valid is None else oracle.row_validity(wl.Sq, vbs)
    return o, lse, valid


@pytest.mark.parametrize("name,kw", CASES)
def test_fused_q_equals_two_pass_and_oracle(name, kw):
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    (o1, l1), (o2, l2) = _run(wl, inp, kv_splits=1)
    assert torch.equal(o1, o2), "fused-Q output differs from quantize + attention"
    assert torch.equal(l1, l2), "fused-Q LSE differs from quantize + attention"
    ro, rl, valid = _oracle(wl, inp)
    assert_out_close(to_np(o1), ro, valid=valid)
    assert_lse_close(to_np(l1), rl, valid=valid)


def test_fused_q_degenerate_rows_and_split():
    """All-zero rows (amax 0: codes and scale 0), one row far larger than the
    rest, a single-row tail, and the key split on top of the fused prologue."""
    wl = WORKLOADS["anima4k"].with_(H=2, Sq=129, Sk=1500, v_scale=False)
    inp = make_inputs(wl, "cuda")
    q = inp.q.clone()
    q[0, 0, 5] = 0
    q[0, 1, 128] = 0
    q[0, 0, 7] *= 1000
    for splits in (1, 3):
        (o1, l1), (o2, l2) = _run(wl, inp, q=q, kv_splits=splits)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl, _ = _oracle(wl, inp, q=q)
    assert_out_close(to_np(o1), ro)
    assert_lse_close(to_np(l1), rl)
    # a zero query row attends uniformly: O is the mean of V, LSE = ln Sk
    assert abs(float(l1[0, 0, 5]) - np.log(wl.Sk)) < 1e-4 * np.log(wl.Sk)


def test_fused_q_block64_padding_rows_excluded():
    """Per-64-row-block scales skip the padded query rows of the last tile:
    garbage there must not change the block's scale."""
    wl = WORKLOADS["sparse"].with_(H=1, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2,
                                   granularity="block64")
    inp = make_inputs(wl, "cuda")
    q = inp.q.clone()
    q[:, :, 1024 - 64 + 37:] = 1000.0  # rows past the last tile's valid count
    (o1, l1), (o2, l2) = _run(wl, inp, q=q, kv_splits=1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    (o3, l3), _ = _run(wl, inp, kv_splits=1)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
