"""GPU LSE merge against the float64 oracle merge, including empty partials
(-inf), in-place output and both 16-bit types."""
import numpy as np
import pytest
import torch

import oracle
from util import ensure_built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("D,dt,rows", [(128, torch.bfloat16, 777), (64, torch.float16, 4096)])
def test_merge_matches_oracle(D, dt, rows):
    import int8_qk_quantized_gb300 as ia
    g = torch.Generator(device="cuda").manual_seed(1)
    o1 = torch.randn(1, 3, rows, D, generator=g, device="cuda").to(dt)
    o2 = torch.randn(1, 3, rows, D, generator=g, device="cuda").to(dt)
    l1 = torch.randn(1, 3, rows, generator=g, device="cuda") * 4 + 8
    l2 = torch.randn(1, 3, rows, generator=g, device="cuda") * 4 + 8
    l1[0, 0, :10] = float("-inf")
    l2[0, 1, 5:15] = float("-inf")
    l1[0, 2, 20:30] = float("-inf")
    l2[0, 2, 20:30] = float("-inf")
    o, l = ia.merge_lse(o1, l1, o2, l2)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(to_np(o1), to_np(l1), to_np(o2), to_np(l2))
    # one rounding to the output type (half an ulp: 2^-8 relative for bf16,
    # 2^-11 for fp16) on top of fp32 arithmetic
    rel = 2.0 ** -8 if dt == torch.bfloat16 else 2.0 ** -11
    assert (np.abs(to_np(o) - ro) <= rel * np.abs(ro) + 1e-5).all()
    got_l = to_np(l)
    assert (np.isneginf(got_l) == np.isneginf(rl)).all()
    fin = np.isfinite(rl)
    assert np.abs(got_l[fin] - rl[fin]).max() < 1e-5 * np.abs(rl[fin]).max() + 1e-5
    assert (to_np(o)[0, 2, 20:30] == 0).all()
    # in place over the first partial
    ia.merge_lse(o1, l1, o2, l2, out=o1, lse_out=l1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o) and torch.equal(l1, l)
