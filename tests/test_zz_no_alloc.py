"""The allocation-free attention entry point against the allocating one.

``ia_attention_fwd_static_workspace`` runs the same kernels as
``ia_attention_fwd`` but takes the key-split partials from a fixed scratch
array inside the library. Each check makes two calls in a row, so the second
one finds the first one's partials in the shared scratch; both must match the
allocating entry point within the parity tolerance.
"""
import gc

import pytest
import torch

from util import O_MAX_ABS, O_MEAN_ABS, LSE_REL, ensure_built
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


CASES = [
    ("anima4k", dict(H=3, Sq=700, Sk=3000), 3),
    ("sdxl", dict(H=2, Sq=500, Sk=2000), 5),
    ("banded", dict(H=2, Sq=300, Sk=2500, skirt_width=500), 4),
    ("sparse", dict(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4), 2),
    ("anima4k", dict(H=2, Sq=300, Sk=1000), 1),
]


def _prepare(name, kw):
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid)
    vsc = None if inp.v_scale is None else inp.v_scale.to(torch.float32).contiguous()
    kvv = None if inp.kv_valid is None else inp.kv_valid.to(torch.int32).contiguous()
    args = dict(bias=inp.bias, block_mask=inp.block_mask, v_scale=vsc, kv_valid=kvv,
                granularity=wl.granularity)
    return (q8, k8, qs, ks, inp.v), args


def _close(o, l, ro, rl):
    d = (o.float() - ro.float()).abs()
    assert d.max().item() <= O_MAX_ABS and d.mean().item() <= O_MEAN_ABS
    fin = torch.isfinite(rl)
    assert torch.equal(torch.isneginf(l), torch.isneginf(rl))
    rel = (l[fin] - rl[fin]).abs() / rl[fin].abs().clamp_min(1.0)
    assert rel.numel() == 0 or rel.max().item() <= LSE_REL


def _both(tensors, args, splits):
    import int8_qk_quantized_gb300 as ia
    q8, k8, qs, ks, v = tensors
    ro, rl = ia.attention(q8, k8, qs, ks, v, kv_splits=splits, return_lse=True, **args)
    out = torch.full_like(ro, float("nan"))
    lse = torch.full_like(rl, float("nan"))
    o, l = ia.attention_static_workspace(q8, k8, qs, ks, v, out, lse=lse, kv_splits=splits, **args)
    ia.device_status()
    return o, l, ro, rl


def test_two_calls_in_a_row_different_shapes():
    prepared = [(_prepare(n, kw), s) for n, kw, s in CASES]
    for (tensors, args), splits in prepared:
        o, l, ro, rl = _both(tensors, args, splits)
        _close(o, l, ro, rl)
        # deterministic kernels and the same split: the results agree exactly
        assert torch.equal(o, ro) and torch.equal(l, rl)


@pytest.mark.parametrize("name,kw,splits", CASES[:2])
def test_two_calls_in_a_row_same_shape(name, kw, splits):
    tensors, args = _prepare(name, kw)
    for _ in range(2):
        o, l, ro, rl = _both(tensors, args, splits)
        _close(o, l, ro, rl)


def test_rejects_more_than_the_fixed_scratch():
    import int8_qk_quantized_gb300 as ia
    tensors, args = _prepare("anima4k", dict(H=16, Sq=4096, Sk=4096))
    out = torch.empty_like(tensors[4])
    with pytest.raises(ia.IAError, match="fixed workspace"):
        ia.attention_static_workspace(*tensors, out, kv_splits=8, **args)


def test_allocates_no_device_memory():
    """The property the entry point exists for: a call with a key split takes
    no device memory. After one warm-up call (which may load the kernels'
    module), the device's free memory is the same before and after a call,
    and torch's allocator holds the same bytes."""
    import int8_qk_quantized_gb300 as ia
    tensors, args = _prepare("anima4k", dict(H=3, Sq=700, Sk=3000))
    q8, k8, qs, ks, v = tensors
    out = torch.empty_like(v[:, :, :700])
    lse = torch.empty((1, 3, 700), dtype=torch.float32, device="cuda")
    ia.attention_static_workspace(q8, k8, qs, ks, v, out, lse=lse, kv_splits=4, **args)
    torch.cuda.synchronize()
    gc.collect()  # tensors of earlier tests are not freed during the measurement
    free0, held0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for splits in (4, 2, 4):
        ia.attention_static_workspace(q8, k8, qs, ks, v, out, lse=lse, kv_splits=splits, **args)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    # torch's allocator gave the calls nothing (a collection may still free
    # unrelated tensors, never add any)
    assert torch.cuda.memory_allocated() <= held0
    ia.device_status()


def test_balanced_segments_through_the_fixed_workspace():
    """Head dim 64 with two key ranges and at least one query tile per SM runs
    the balanced segments; through the allocation-free entry point the partials
    live in the fixed workspace, and the result equals the allocating call."""
    import int8_qk_quantized_gb300 as ia
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = -(-sms // 3) + 1  # 3 query tiles of 256 rows per head
    tensors, args = _prepare("sdxl", dict(H=H, Sq=700, Sk=1000))
    q8, k8, qs, ks, v = tensors
    ref, rl = ia.attention(q8, k8, qs, ks, v, kv_splits=2, return_lse=True, **args)
    out = torch.empty_like(ref)
    lse = torch.empty_like(rl)
    o, l = ia.attention_static_workspace(q8, k8, qs, ks, v, out, lse=lse, kv_splits=2, **args)
    ia.device_status()
    assert torch.equal(o, ref) and torch.equal(l, rl)
