"""GPU quantiser against the oracle: codes, scales and the K mean bit for bit.

Covers the fused kernel (with Q in the same launch for a K of at most 64 MiB)
and, for a larger K, the two-kernel path (mean pass, then codes), per-token and per-64-row-block scales, bf16 and fp16, D 64
and 128,
ragged tails, the validity vector, strided (BSHD-backed) inputs, an external
mean, no centring, and the full-size K of the banded and block-sparse
workloads."""
import numpy as np
import pytest
import torch

import oracle
from util import ensure_built, to_np
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def gpu_quant(q, k, gran, kv_valid=None, center=True, k_mean=None, two_pass=True):
    """two_pass: the library's mean-then-codes kernels (it is given a buffer for
    the mean, which is returned); False: the fused kernel (no mean buffer, so
    only codes and scales come back)."""
    import int8_qk_quantized_gb300 as ia
    res = ia.quantize_qk(q, k, granularity=gran, center_k=center, kv_valid=kv_valid,
                         k_mean=k_mean, return_mean=center and two_pass, two_pass=two_pass)
    torch.cuda.synchronize()
    return [None if t is None else to_np(t) for t in res]


def oracle_quant(q, k, gran, kv_valid=None, center=True, k_mean=None):
    vbs = None if kv_valid is None else kv_valid.cpu().numpy()
    qn, kn = to_np(q), to_np(k)
    mu = None
    if center:
        mu = oracle.k_mean(kn, vbs) if k_mean is None else k_mean.cpu().numpy()
    qc, qs = oracle.quantize(qn, None, gran, vbs if q.shape[2] == k.shape[2] else None)
    kc, ks = oracle.quantize(kn, mu, gran, vbs)
    return [qc, qs, kc, ks] + ([mu] if center else [])


def assert_same(got, ref):
    names = ["q codes", "q scales", "k codes", "k scales", "k mean"]
    for g, r, n in zip(got, ref, names):
        assert g.shape == r.shape, (n, g.shape, r.shape)
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)
            raise AssertionError(f"{n}: {len(bad)} mismatches, first at {bad[0].tolist()}: "
                                 f"{g[tuple(bad[0])]} vs {r[tuple(bad[0])]}")


SMALL = [
    ("tiny", {}),
    ("sdxl", dict(H=3, Sq=1000, Sk=1000)),
    ("sdxl", dict(H=2, Sq=4096, Sk=4096, granularity="token")),
    ("anima4k", dict(H=3, Sq=777, Sk=1000)),
    ("anima4k", dict(H=2, granularity="block64", dtype="fp16")),
    ("banded", dict(H=2, Sq=300, Sk=3000, skirt_width=600)),
    ("sparse", dict(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4)),
    ("sparse", dict(H=2, Sq=2048, Sk=2048, band_tiles=8, random_tiles=4, granularity="block64")),
    # a Q more than twice as long as K: Q's code kernel and K's cluster kernel
    # run as two launches (in one launch Q would get only K's chunk count)
    ("anima4k", dict(H=2, Sq=5000, Sk=700)),
    ("anima4k", dict(H=2, Sq=3001, Sk=640, granularity="block64", dtype="fp16")),
]


@pytest.mark.parametrize("name,kw", SMALL)
def test_quantize_bit_exact(name, kw):
    wl = WORKLOADS[name].with_(**kw)
    inp = make_inputs(wl, "cuda")
    got = gpu_quant(inp.q, inp.k, wl.granularity, inp.kv_valid)
    ref = oracle_quant(inp.q, inp.k, wl.granularity, inp.kv_valid)
    assert_same(got, ref)


# A K between 32 and 64 MiB takes the one-pass cluster form with Q in the same
# launch; above 64 MiB, with a mean buffer, the library runs the mean kernel and
# the code kernel, without one the fused kernel. All against the oracle (ragged
# tail, validity vector, per-token and per-block scales).
LARGE = [
    ("banded", dict(H=2, Sq=300, Sk=70001, skirt_width=600)),   # 35.8 MB: one pass
    ("sparse", dict(H=1, Sq=140032, Sk=140032, band_tiles=8, random_tiles=4, granularity="block64")),
    ("banded", dict(H=4, Sq=300, Sk=70001, skirt_width=600)),   # 71.7 MB: two kernels
    ("sparse", dict(H=2, Sq=140032, Sk=140032, band_tiles=8, random_tiles=4, granularity="block64")),
]


@pytest.mark.parametrize("two_pass", [True, False], ids=["two_pass", "fused"])
@pytest.mark.parametrize("name,kw", LARGE)
def test_quantize_large_k_both_paths(name, kw, two_pass):
    wl = WORKLOADS[name].with_(**kw)
    assert wl.B * wl.H * wl.Sk * wl.D * 2 > 32 << 20
    inp = make_inputs(wl, "cuda")
    got = gpu_quant(inp.q, inp.k, wl.granularity, inp.kv_valid, two_pass=two_pass)
    ref = oracle_quant(inp.q, inp.k, wl.granularity, inp.kv_valid)
    assert_same(got, ref)


@pytest.mark.parametrize("D,gran", [(64, "token"), (128, "block64")])
def test_quantize_strided_bshd_views(D, gran):
    g = torch.Generator(device="cuda").manual_seed(7)
    B, S, H = 2, 700, 3
    qb = torch.randn(B, S, H, D, generator=g, device="cuda").to(torch.bfloat16)
    kb = (torch.randn(B, S, H, D, generator=g, device="cuda") * 3 + 1).to(torch.bfloat16)
    q, k = qb.permute(0, 2, 1, 3), kb.permute(0, 2, 1, 3)
    assert not q.is_contiguous()
    assert_same(gpu_quant(q, k, gran), oracle_quant(q, k, gran))


def test_quantize_external_mean_and_no_centring():
    wl = WORKLOADS["sdxl"].with_(H=2, Sq=640, Sk=640)
    inp = make_inputs(wl, "cuda")
    mu = torch.randn(1, 2, 64, generator=torch.Generator(device="cuda").manual_seed(3),
                     device="cuda")
    got = gpu_quant(inp.q, inp.k, "token", k_mean=mu)
    ref = oracle_quant(inp.q, inp.k, "token", k_mean=mu)
    assert_same(got, ref)
    got = gpu_quant(inp.q, inp.k, "block64", center=False)
    ref = oracle_quant(inp.q, inp.k, "block64", center=False)
    assert_same(got, ref)


def test_quantize_degenerate_rows():
    """All-zero rows, a constant K (centred to zero) and a single row."""
    q = torch.zeros(1, 1, 130, 128, dtype=torch.bfloat16, device="cuda")
    q[0, 0, 5, 7] = 3.0
    k = torch.full((1, 1, 130, 128), 0.5, dtype=torch.bfloat16, device="cuda")
    assert_same(gpu_quant(q, k, "token"), oracle_quant(q, k, "token"))
    assert_same(gpu_quant(q, k, "block64"), oracle_quant(q, k, "block64"))
    q1 = torch.randn(1, 2, 1, 64, device="cuda").to(torch.float16)
    k1 = torch.randn(1, 2, 1, 64, device="cuda").to(torch.float16)
    assert_same(gpu_quant(q1, k1, "token"), oracle_quant(q1, k1, "token"))


@pytest.mark.parametrize("name", ["banded", "sparse"])
def test_quantize_full_size(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda")
    got = gpu_quant(inp.q, inp.k, wl.granularity, inp.kv_valid)
    ref = oracle_quant(inp.q, inp.k, wl.granularity, inp.kv_valid)
    assert_same(got, ref)
