"""Helpers shared by the tests (no method arithmetic here)."""
import os
import re

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ia.h")

# Tolerances of the parity bar (output against the same-quantisation float64
# oracle; output against exact float64 attention; LSE relative).
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
O_EXACT_MEAN_ABS = 1e-2
LSE_REL = 1e-4


def ensure_built():
    from int8_qk_quantized_gb300 import build_lib
    return build_lib.build()


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a 16-bit tensor (or plain copy of others) on the host."""
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.detach().float().cpu().numpy()
    return t.detach().cpu().numpy()


def declared_symbols():
    """Names of the functions include/ia.h declares with IA_API."""
    src = open(HEADER).read()
    return sorted(set(re.findall(r"IA_API\s+[\w\s\*]+?\b(ia_\w+)\s*\(", src)))


def assert_lse_close(got, ref, valid=None):
    """LSE within LSE_REL relative of the reference, -inf exactly where it is
    -inf. Reading of "1e-4 relative": the error is divided by max(|LSE|, 1), so
    it is relative for |LSE| >= 1 and an absolute 1e-4 below (an LSE near 0
    would otherwise make any bound vanish; LSE is ln of a sum of exponentials,
    so 1e-4 absolute there is a relative 1e-4 on that sum)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if valid is not None:
        got, ref = got[..., valid], ref[..., valid]
    inf_ref = np.isneginf(ref)
    assert (np.isneginf(got) == inf_ref).all(), "-inf rows differ"
    g, r = got[~inf_ref], ref[~inf_ref]
    err = np.abs(g - r) / np.maximum(np.abs(r), 1.0)
    assert err.size == 0 or err.max() <= LSE_REL, f"LSE rel err {err.max():.3e}"


def assert_out_close(got, ref, exact=None, valid=None, max_abs=O_MAX_ABS, mean_abs=O_MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if valid is not None:
        got, ref = got[..., valid, :], ref[..., valid, :]
        if exact is not None:
            exact = np.asarray(exact)[..., valid, :]
    d = np.abs(got - ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert d.max() <= max_abs, f"max abs err {d.max():.3e}"
    assert d.mean() <= mean_abs, f"mean abs err {d.mean():.3e}"
    if exact is not None:
        de = np.abs(got - np.asarray(exact, dtype=np.float64)).mean()
        assert de <= O_EXACT_MEAN_ABS, f"mean abs err vs exact attention {de:.3e}"
    return d.max(), d.mean()
