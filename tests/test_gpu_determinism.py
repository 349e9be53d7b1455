"""Run-to-run equality of the attention kernels on the GPU.

Every call of the path is a fixed sequence of exact integer products and
fp32 operations in a fixed order, so repeated calls on the same inputs must
give bit-identical outputs and LSE. A difference can only come from a race
between the kernel's warps and the tensor core (a TMEM or shared-memory
buffer reused too early); a race that corrupts a few rows may stay inside the
oracle tolerances, but not inside this check. The shapes cover each kernel:
the dense CTA pairs (unmasked, per-key bias, in-kernel Q quantization, key
splits), the block-sparse kernel and the per-row mask kernel.
"""
import pytest
import torch

from util import ensure_built
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

REPEATS = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def assert_repeatable(fn):
    import int8_qk_quantized_gb300 as ia
    o0, l0 = (t.clone() for t in fn())
    for _ in range(REPEATS - 1):
        o, l = fn()
        bad = (o != o0).any(-1)
        assert not bad.any(), f"{int(bad.sum())} output rows differ between identical calls"
        assert torch.equal(torch.nan_to_num(l, neginf=0.0), torch.nan_to_num(l0, neginf=0.0)), \
            "LSE differs between identical calls"
    ia.device_status()


def test_dense_pairs_repeatable():
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["banded"].with_(H=6)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    assert_repeatable(lambda: ia.attention(q8, k8, qs, ks, inp.v, return_lse=True))
    assert_repeatable(lambda: ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, return_lse=True))
    assert_repeatable(lambda: ia.attention_quant_q(inp.q, k8, ks, inp.v, bias=inp.bias,
                                                   return_lse=True))
    assert_repeatable(lambda: ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, return_lse=True,
                                           kv_splits=3))


def test_block_sparse_repeatable():
    import int8_qk_quantized_gb300 as ia
    for wl in (WORKLOADS["sparse"].with_(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4),
               WORKLOADS["sparse"].with_(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2,
                                         D=64, granularity="block64")):
        inp = make_inputs(wl, "cuda")
        q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, kv_valid=inp.kv_valid,
                                        granularity=wl.granularity)
        assert_repeatable(lambda: ia.attention(q8, k8, qs, ks, inp.v, block_mask=inp.block_mask,
                                               kv_valid=inp.kv_valid, granularity=wl.granularity,
                                               return_lse=True))


def test_row_mask_repeatable():
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["anima4k"].with_(H=4, Sq=2048, Sk=3000)
    inp = make_inputs(wl, "cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    mask = (torch.rand(1, 1, wl.Sq, wl.Sk, device="cuda", generator=g) * -6.0).to(torch.bfloat16)
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    assert_repeatable(lambda: ia.attention(q8, k8, qs, ks, inp.v, mask=mask, return_lse=True))
