"""Out-of-bounds write checks, standing in for compute-sanitizer (closed on this pool).

Every output a kernel writes (codes, scales, the K mean, attention output and
LSE, the key-split workspace, merged outputs) is placed inside a larger device
buffer whose other bytes hold a fixed pattern. After the call the pattern must
be intact everywhere the output does not reach: 4 KiB before and after a
contiguous output, and, for strided outputs, every byte of the parent buffer
outside the view. The results inside must also equal those of the same call
on freshly allocated outputs, so a write that lands in the wrong place inside
the buffer shows as well. The shapes take every edge the kernels have: ragged
query and key tails, a CTA-pair grid rounded up past Sq, key sub-range views,
head-interleaved (BSHD) outputs, key splits, a partial last 64-row tile under
a validity vector, per-row masks, and the fused-Q and allocation-free entry
points. All calls go through the C ABI.
"""
import ctypes

import numpy as np
import pytest
import torch

from util import ensure_built
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
PAT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


class Guarded:
    """A device buffer of `nbytes` between two guard regions, all bytes PAT."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), PAT, dtype=torch.uint8, device="cuda")

    def tensor(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        g = torch.cat([self.buf[:GUARD], self.buf[GUARD + self.n:]])
        bad = int((g != PAT).sum())
        assert bad == 0, f"{what}: {bad} guard bytes overwritten"


def guarded_like(shape, dtype):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    g = Guarded(n)
    return g, g.tensor(dtype, shape)


def strided_in_parent(parent_shape, dtype, make_view):
    """A parent buffer full of PAT and a strided view of it; returns (parent
    bytes, view, mask of the parent's bytes the view covers)."""
    es = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(parent_shape))
    raw = torch.full((n * es,), PAT, dtype=torch.uint8, device="cuda")
    parent = raw.view(dtype).view(parent_shape)
    view = make_view(parent)
    cover = torch.zeros(parent_shape, dtype=torch.int32, device="cuda")
    make_view(cover).fill_(1)
    cover_bytes = cover.reshape(-1, 1).repeat(1, es).reshape(-1).bool()
    return raw, view, cover_bytes


def check_outside(raw, cover, what):
    torch.cuda.synchronize()
    bad = int((raw[~cover] != PAT).sum())
    assert bad == 0, f"{what}: {bad} bytes outside the view overwritten"


# ------------------------------------------------------------------- quantize
QUANT_CASES = [
    ("anima4k", dict(H=2, Sq=300, Sk=777)),                                   # ragged, D 128
    ("sdxl", dict(H=2, Sq=130, Sk=191)),                                      # D 64, per block
    ("sparse", dict(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2)),    # partial last tile
    ("sparse", dict(H=1, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2, D=64,
                    granularity="block64")),
]


@pytest.mark.parametrize("with_mean", [True, False], ids=["mean_out", "no_mean_out"])
@pytest.mark.parametrize("name,kw", QUANT_CASES + [
    # K between 32 and 64 MiB: one launch for Q and K (cluster mean, then codes)
    ("banded", dict(H=2, Sq=200, Sk=66001, skirt_width=600)),
    ("sparse", dict(H=1, Sq=135168, Sk=135168, band_tiles=4, random_tiles=2, granularity="block64")),
    # K above 64 MiB: with a mean output, the mean kernel and the code kernel
    ("banded", dict(H=4, Sq=200, Sk=66001, skirt_width=600)),
    ("sparse", dict(H=2, Sq=135168, Sk=135168, band_tiles=4, random_tiles=2, granularity="block64")),
])
def test_quantize_outputs_stay_in_bounds(name, kw, with_mean):
    """A K above 64 MiB with a mean output runs the mean and code kernels;
    otherwise Q and K go in one launch (the fused kernel for K)."""
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    B, H, D = wl.B, wl.H, wl.D
    ns = (lambda S: S) if wl.granularity == "token" else (lambda S: (S + 63) // 64)
    ref = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid,
                         return_mean=True)
    outs = [guarded_like((B, H, wl.Sq, D), torch.int8), guarded_like((B, H, ns(wl.Sq)), torch.float32),
            guarded_like((B, H, wl.Sk, D), torch.int8), guarded_like((B, H, ns(wl.Sk)), torch.float32),
            guarded_like((B, H, D), torch.float32)]
    L = ia.load_library()
    qst = (ctypes.c_int64 * 3)(*[inp.q.stride(i) for i in range(3)])
    kst = (ctypes.c_int64 * 3)(*[inp.k.stride(i) for i in range(3)])
    kvv = None if inp.kv_valid is None else inp.kv_valid.to(torch.int32).contiguous()
    st = L.ia_quantize_qk(inp.q.data_ptr(), inp.k.data_ptr(), ia._dtype_code(inp.q.dtype), B, H,
                          wl.Sq, wl.Sk, D, qst, kst, ia._gran_code(wl.granularity), 1,
                          None if kvv is None else kvv.data_ptr(), None,
                          *[t.data_ptr() for _, t in (outs[0], outs[2], outs[1], outs[3])],
                          outs[4][1].data_ptr() if with_mean else None,
                          torch.cuda.current_stream().cuda_stream)
    assert st == 0, ia.load_library().ia_last_error_message()
    n_out = 5 if with_mean else 4
    for (g, t), r, n in zip(outs[:n_out], ref, ("q codes", "q scales", "k codes", "k scales", "k mean")):
        g.check(n)
        assert torch.equal(t, r), n


# ------------------------------------------------------------------ attention
ATTN_CASES = [
    ("anima4k", dict(H=2, Sq=257, Sk=1100, v_scale=False), {}),              # pair grid past Sq
    ("anima4k", dict(H=1, Sq=129, Sk=65, v_scale=False), {}),
    ("sdxl", dict(H=2, Sq=333, Sk=1000), {}),                                 # D 64
    ("banded", dict(H=2, Sq=300, Sk=2500, skirt_width=500), dict(bias=True)),
    ("anima4k", dict(H=2, Sq=200, Sk=3000, v_scale=False), dict(kv_splits=3)),
    ("sdxl", dict(H=2, Sq=100, Sk=2048), dict(kv_splits=4)),
    # two key ranges over >= one 256-row query tile per SM: balanced segments
    ("sdxl", dict(H=60, Sq=700, Sk=1000), dict(kv_splits=2, segments=True)),
    ("sparse", dict(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2), {}),
    ("sparse", dict(H=1, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2, D=64,
                    granularity="block64"), dict(kv_splits=2)),
    ("anima4k", dict(H=1, Sq=300, Sk=512, v_scale=False), dict(row_mask=True)),
]


def _attn_args(wl, inp, extra):
    args = dict(block_mask=inp.block_mask, v_scale=inp.v_scale, kv_valid=inp.kv_valid,
                granularity=wl.granularity, return_lse=True, kv_splits=extra.get("kv_splits", 1))
    if extra.get("bias"):
        args["bias"] = inp.bias
    if extra.get("row_mask"):
        g = torch.Generator(device="cuda").manual_seed(3)
        args["mask"] = torch.rand((1, 1, wl.Sq, wl.Sk), generator=g, device="cuda") > 0.3
    return args


@pytest.mark.parametrize("name,kw,extra", ATTN_CASES)
def test_attention_outputs_and_workspace_stay_in_bounds(name, kw, extra):
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid)
    args = _attn_args(wl, inp, extra)
    ro, rl = ia.attention(q8, k8, qs, ks, inp.v, **args)
    go, out = guarded_like(tuple(ro.shape), ro.dtype)
    gl, lse = guarded_like(tuple(rl.shape), torch.float32)
    ws = None
    if args["kv_splits"] > 1:
        p = ia.AttnParams()
        ia.load_library().ia_attn_params_init(ctypes.byref(p), wl.B, wl.H, wl.Sq, wl.Sk, wl.D, 0, 0)
        p.kv_splits = args["kv_splits"]
        need = ia.load_library().ia_attention_workspace_size(ctypes.byref(p))
        gw = Guarded(need)
        ws = gw.tensor(torch.uint8, (need,))
    o, l = ia.attention(q8, k8, qs, ks, inp.v, out=out, lse=lse, workspace=ws, **args)
    ia.device_status()
    go.check("out")
    gl.check("lse")
    if ws is not None:
        gw.check("key-split workspace")
    assert torch.equal(o, ro) and torch.equal(l, rl)
    # the fused-Q entry point (Q quantized in the kernel) on the same guards
    if not extra.get("row_mask"):
        out.fill_(0)
        o2, l2 = ia.attention_quant_q(inp.q, k8, ks, inp.v, out=out, lse=lse, workspace=ws, **args)
        ia.device_status()
        go.check("fused-Q out")
        gl.check("fused-Q lse")
        if extra.get("segments"):
            # the int8-Q call split the keys in balanced segments, the fused-Q
            # call (no segments) in two equal ranges: equal up to the merge's
            # rounding
            assert (o2.float() - ro.float()).abs().max().item() < 2e-3
            assert (l2 - rl).abs().max().item() < 1e-4
        else:
            assert torch.equal(o2, ro) and torch.equal(l2, rl)


def test_key_subrange_views_and_bshd_outputs_stay_in_bounds():
    """The core/skirt split's key sub-range views with outputs written into
    head-interleaved parents (BSHD, padded rows) and an LSE view with a padded
    row stride: every byte of the parents outside the views keeps the pattern."""
    import int8_qk_quantized_gb300 as ia
    for D, name in ((128, "banded"), (64, "sdxl")):
        wl = WORKLOADS[name].with_(H=3, Sq=257, Sk=1500, D=D)
        inp = make_inputs(wl, "cuda")
        q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity)
        a, b = 320, 1216  # whole 64-row tiles, so that per-block scales slice with them
        ksr = ks[:, :, a:b] if wl.granularity == "token" else ks[:, :, a // 64:b // 64]
        ref = ia.attention(q8, k8[:, :, a:b], qs, ksr, inp.v[:, :, a:b],
                           granularity=wl.granularity, return_lse=True)
        raw_o, out, cov_o = strided_in_parent(
            (1, wl.Sq, wl.H + 1, D + 8), inp.v.dtype,
            lambda t: t[:, :, :wl.H, :D].permute(0, 2, 1, 3))
        raw_l, lse, cov_l = strided_in_parent(
            (1, wl.H, wl.Sq + 7), torch.float32, lambda t: t[:, :, 3:3 + wl.Sq])
        o, l = ia.attention(q8, k8[:, :, a:b], qs, ksr, inp.v[:, :, a:b], out=out,
                            lse=lse, granularity=wl.granularity, return_lse=True)
        ia.device_status()
        check_outside(raw_o, cov_o, f"BSHD out D={D}")
        check_outside(raw_l, cov_l, f"strided lse D={D}")
        assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])


def test_merge_outputs_stay_in_bounds():
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["banded"].with_(H=2, Sq=301, Sk=1000, skirt_width=200)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    parts = [ia.attention(q8, k8[:, :, a:b], qs, ks[:, :, a:b], inp.v[:, :, a:b], return_lse=True)
             for a, b in ((0, 300), (300, 700), (700, 1000))]
    ro, rl = ia.merge_lse(*parts[0], *parts[1])
    go, out = guarded_like(tuple(ro.shape), ro.dtype)
    gl, lse = guarded_like(tuple(rl.shape), torch.float32)
    o, l = ia.merge_lse(*parts[0], *parts[1], out=out, lse_out=lse)
    go.check("merge out")
    gl.check("merge lse")
    assert torch.equal(o, ro) and torch.equal(l, rl)
    rno, rnl = ia.merge_lse_n([p[0] for p in parts], [p[1] for p in parts])
    go2, out2 = guarded_like(tuple(rno.shape), rno.dtype)
    gl2, lse2 = guarded_like(tuple(rnl.shape), torch.float32)
    o, l = ia.merge_lse_n([p[0] for p in parts], [p[1] for p in parts], out=out2, lse_out=lse2)
    go2.check("merge_n out")
    gl2.check("merge_n lse")
    assert torch.equal(o, rno) and torch.equal(l, rnl)


def test_static_workspace_entry_outputs_stay_in_bounds():
    import int8_qk_quantized_gb300 as ia
    wl = WORKLOADS["anima4k"].with_(H=2, Sq=300, Sk=2000, v_scale=False)
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k)
    ro, rl = ia.attention(q8, k8, qs, ks, inp.v, return_lse=True, kv_splits=3)
    go, out = guarded_like(tuple(ro.shape), ro.dtype)
    gl, lse = guarded_like(tuple(rl.shape), torch.float32)
    o, l = ia.attention_static_workspace(q8, k8, qs, ks, inp.v, out, lse=lse, kv_splits=3)
    ia.device_status()
    go.check("static-workspace out")
    gl.check("static-workspace lse")
    assert torch.equal(o, ro) and torch.equal(l, rl)
