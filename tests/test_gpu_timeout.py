"""The bounded-wait path of the attention kernel, without a GPU fault.

The test hook makes the MMA issuer of every CTA wait on a barrier that nothing
signals, with a 20 ms limit. The call must come back, the device status must
report IA_ERR_TIMEOUT exactly once, and the same context must then run a
normal call correctly (no fault, no hang, TMEM released)."""
import numpy as np
import pytest
import torch

from util import ensure_built, to_np
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("kind", ["dense", "sparse", "segments"])
def test_wait_timeout_reports_status_and_context_survives(kind):
    """`segments`: head dim 64 with two key ranges over >= one query tile per
    SM, so each CTA runs a loop of segments; after the timeout in its first
    segment the CTA leaves the loop instead of starting the next one."""
    import time

    import int8_qk_quantized_gb300 as ia
    splits = 1
    if kind == "sparse":
        wl = WORKLOADS["sparse"].with_(H=2, Sq=1024, Sk=1024, band_tiles=4, random_tiles=2)
    elif kind == "dense":
        wl = WORKLOADS["anima4k"].with_(H=2, Sq=512, Sk=640)
    else:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        wl = WORKLOADS["sdxl"].with_(H=-(-sms // 3) + 1, Sq=700, Sk=1000)
        splits = 2
    inp = make_inputs(wl, "cuda")
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, kv_valid=inp.kv_valid, granularity=wl.granularity)
    args = dict(block_mask=inp.block_mask, kv_valid=inp.kv_valid, v_scale=inp.v_scale,
                granularity=wl.granularity, kv_splits=splits)
    ref = ia.attention(q8, k8, qs, ks, inp.v, **args)
    ia.device_status()
    t0 = time.perf_counter()
    ia.attention(q8, k8, qs, ks, inp.v, wait_timeout_ns=20_000_000, debug_stall=True, **args)
    with pytest.raises(ia.IAError) as e:
        ia.device_status()
    assert e.value.status == 4
    assert time.perf_counter() - t0 < 30.0
    ia.device_status()  # cleared by the read
    out = ia.attention(q8, k8, qs, ks, inp.v, **args)
    ia.device_status()
    assert torch.equal(out, ref)
