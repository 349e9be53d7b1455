"""GPU attention against the oracle.

Output within max-abs 2e-2 and mean-abs 2e-3 of the same-quantisation float64
oracle and within mean-abs 1e-2 of exact float64 attention; LSE within 1e-4
relative, -inf exactly where the oracle has -inf. Small cases compare every
element; the full-size workloads compare seeded samples of query rows that
cover every query tile of every head, in the launch configuration the
benchmark times."""
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


def run_gpu(inp, wl, sm_scale=None, v=None, return_codes=False):
    import int8_qk_quantized_gb300 as ia
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity,
                                    kv_valid=inp.kv_valid)
    out, lse = ia.attention(q8, k8, qs, ks, inp.v if v is None else v, bias=inp.bias,
                            block_mask=inp.block_mask, sm_scale=sm_scale, v_scale=inp.v_scale,
                            kv_valid=inp.kv_valid, granularity=wl.granularity, return_lse=True)
    ia.device_status()
    res = (to_np(out), to_np(lse))
    return res + ((q8, qs, k8, ks),) if return_codes else res


def run_oracle(inp, wl, rows=None, sm_scale=None, exact=True):
    vbs = None if inp.kv_valid is None else inp.kv_valid.cpu().numpy()
    kw = dict(sm_scale=sm_scale,
              bias=None if inp.bias is None else to_np(inp.bias),
              block_mask=None if inp.block_mask is None else to_np(inp.block_mask),
              v_scale=None if inp.v_scale is None else to_np(inp.v_scale), rows=rows)
    qn, kn, vn = to_np(inp.q), to_np(inp.k), to_np(inp.v)
    o, lse, _ = oracle.quantize_and_attend(qn, kn, vn, granularity=wl.granularity,
                                           kv_valid=vbs, **kw)
    oe = None
    if exact:
        oe, _ = oracle.exact_attention(qn, kn, vn, kv_valid=vbs, **kw)
    return o, lse, oe


def query_valid(inp, wl):
    if inp.kv_valid is None or wl.Sq != wl.Sk:
        return None
    return oracle.row_validity(wl.Sq, inp.kv_valid.cpu().numpy())


SMALL = [
    ("tiny", {}),
    ("sdxl", dict(H=2, Sq=1000, Sk=1000)),
    ("anima4k", dict(H=2, Sq=1000, Sk=1000)),
    ("anima4k", dict(H=2, Sq=300, Sk=777, v_scale=False, dtype="fp16")),
    ("banded", dict(H=2, Sq=300, Sk=2000, skirt_width=400)),
    ("banded", dict(H=2, Sq=257, Sk=1100, skirt_width=300, D=64, dtype="fp16")),
    ("sparse", dict(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4)),
    ("sparse", dict(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2, D=64,
                    granularity="block64")),
]


@pytest.mark.parametrize("name,kw", SMALL)
def test_attention_small(name, kw):
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    o, lse = run_gpu(inp, wl)
    ro, rl, re = run_oracle(inp, wl)
    valid = query_valid(inp, wl)
    assert_out_close(o, ro, re, valid=valid)
    assert_lse_close(lse, rl)
    if valid is not None:
        assert (o[:, :, ~valid] == 0).all()


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (5, 64), (129, 127), (256, 129), (130, 4000)])
def test_attention_edge_shapes(Sq, Sk):
    wl = WORKLOADS["anima4k"].with_(H=1, Sq=Sq, Sk=Sk, v_scale=False)
    inp = make_inputs(wl, "cuda")
    o, lse = run_gpu(inp, wl, sm_scale=0.1)
    ro, rl, re = run_oracle(inp, wl, sm_scale=0.1)
    assert_out_close(o, ro, re)
    assert_lse_close(lse, rl)


def test_attention_fully_masked_rows_and_empty_tiles():
    """A query tile whose mask row is empty gives O = 0 and LSE = -inf; a CTA
    whose two query tiles keep nothing still writes both."""
    wl = WORKLOADS["sparse"].with_(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2)
    inp = make_inputs(wl, "cuda")
    inp.block_mask[0, 0, 3] = False       # one empty query tile
    inp.block_mask[0, 1, 4:6] = False     # both tiles of one CTA empty
    o, lse = run_gpu(inp, wl)
    ro, rl, re = run_oracle(inp, wl, exact=False)
    assert_out_close(o, ro, valid=query_valid(inp, wl))
    assert_lse_close(lse, rl)
    assert np.isneginf(lse[0, 0, 192:256]).all() and (o[0, 0, 192:256] == 0).all()
    assert np.isneginf(lse[0, 1, 256:384]).all()


def test_attention_strided_v_and_out():
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["anima4k"].with_(H=3, Sq=500, Sk=700, v_scale=False)
    inp = make_inputs(wl, "cuda")
    vb = inp.v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)  # BSHD-backed view
    assert not vb.is_contiguous()
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    ob = torch.empty(1, 500, 3, 128, dtype=torch.bfloat16, device="cuda")
    out = ob.permute(0, 2, 1, 3)
    lse_full = torch.empty(1, 3, 600, device="cuda")
    ia.attention(q8, k8, qs, ks, vb, out=out, lse=lse_full[:, :, :500], return_lse=True)
    ia.device_status()
    ro, rl, re = run_oracle(inp, wl)
    assert_out_close(to_np(out), ro, re)
    assert_lse_close(to_np(lse_full[:, :, :500]), rl)


def test_split_core_skirt_merge_equals_single_call():
    """The comfy-kitchen split: core keys without bias, skirt keys with bias,
    merged through the LSEs, equals one call over all keys with the bias.
    K is quantised once so both partials share one centring frame."""
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["banded"].with_(H=3, Sq=640, Sk=2560, skirt_width=512)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    full_o, full_l = ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, return_lse=True)
    lo, hi = 512, 2048
    core_o, core_l = ia.attention(q8, k8[:, :, lo:hi], qs, ks[:, :, lo:hi], inp.v[:, :, lo:hi],
                                  return_lse=True)
    idx = torch.cat([torch.arange(0, lo), torch.arange(hi, 2560)]).cuda()
    sk8, sks, sv = k8[:, :, idx].contiguous(), ks[:, :, idx].contiguous(), inp.v[:, :, idx].contiguous()
    sb = inp.bias[idx].contiguous()
    sk_o, sk_l = ia.attention(q8, sk8, qs, sks, sv, bias=sb, return_lse=True)
    mo, ml = ia.merge_lse(core_o, core_l, sk_o, sk_l)
    ia.device_status()
    d = (mo.float() - full_o.float()).abs()
    assert d.max().item() < 1e-2 and d.mean().item() < 1e-3
    assert ((ml - full_l).abs() / full_l.abs().clamp_min(1)).max().item() < 1e-5
    ro, rl, re = run_oracle(inp, wl)
    assert_out_close(to_np(mo), ro, re)
    assert_lse_close(to_np(ml), rl)


def sample_rows(Sq, seed, per_tile=2):
    rng = np.random.default_rng(seed)
    rows = {0, Sq - 1}
    for t in range(0, Sq, 128):
        for r in rng.integers(t, min(Sq, t + 128), size=per_tile):
            rows.add(int(r))
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["anima4k", "anima9k", "banded", "sparse", "sdxl"])
def test_attention_full_size_sampled(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda")
    o, lse = run_gpu(inp, wl)
    rows = sample_rows(wl.Sq, 11, per_tile=1 if wl.Sq > 20000 else 2)
    ro, rl, re = run_oracle(inp, wl, rows=rows)
    valid = query_valid(inp, wl)
    v = None if valid is None else valid[rows]
    assert_out_close(o[:, :, rows], ro, re, valid=v)
    assert_lse_close(lse[:, :, rows], rl)


def test_banded_split_step_full_size_sampled():
    """The benchmark's step at full size: quantize Q and K once, the unmasked
    core and the two biased skirts as key sub-range views with their LSEs, two
    exact merges ("int8_attention: masked path costs ~1.8x unmasked, ...",
    Question 2), against the oracle's single call over all keys on sampled
    rows."""
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["banded"]
    inp = make_inputs(wl, "cuda")
    lo, hi = wl.skirt_width, wl.Sk - wl.skirt_width
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    parts = []
    for a, b, bias in ((lo, hi, None), (0, lo, inp.bias[:lo]), (hi, wl.Sk, inp.bias[hi:])):
        parts.append(ia.attention(q8, k8[:, :, a:b], qs, ks[:, :, a:b], inp.v[:, :, a:b],
                                  bias=bias, return_lse=True))
    o, l = ia.merge_lse(*parts[0], *parts[1])
    o, l = ia.merge_lse(o, l, *parts[2], out=o, lse_out=l)
    ia.device_status()
    rows = sample_rows(wl.Sq, 12)
    ro, rl, re = run_oracle(inp, wl, rows=rows)
    assert_out_close(to_np(o)[:, :, rows], ro, re)
    assert_lse_close(to_np(l)[:, :, rows], rl)


@pytest.mark.parametrize("name", ["anima4k", "anima9k"])
def test_fused_q_full_size(name):
    """The fused Q quantization at the Anima sizes: equal to quantize + attention
    everywhere, and within the oracle's tolerance on sampled rows."""
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    o2, l2 = ia.attention(q8, k8, qs, ks, inp.v, v_scale=inp.v_scale, return_lse=True)
    o1, l1 = ia.attention_quant_q(inp.q, k8, ks, inp.v, v_scale=inp.v_scale, return_lse=True)
    ia.device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rows = sample_rows(wl.Sq, 13, per_tile=1)
    ro, rl, re = run_oracle(inp, wl, rows=rows)
    assert_out_close(to_np(o1)[:, :, rows], ro, re)
    assert_lse_close(to_np(l1)[:, :, rows], rl)
