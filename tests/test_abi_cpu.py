"""The C ABI on the host, no GPU: the library builds and loads, it exports
every function include/ia.h declares, the ctypes mirror of ia_attn_params
matches the C layout, and argument errors are reported before any launch."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

from util import HEADER, ROOT, declared_symbols, ensure_built

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="CUDA toolkit not available")


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import int8_qk_quantized_gb300 as ia
    return ia.load_library()


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"ia_quantize_qk", "ia_attention_fwd", "ia_merge_lse"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libia.so does not export {n}"


def test_params_struct_layout_matches_header(lib):
    import int8_qk_quantized_gb300 as ia
    src = r'''
#include <stddef.h>
#include <stdio.h>
#include "ia.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(ia_attn_params), offsetof(ia_attn_params, q_strides),
         offsetof(ia_attn_params, lse_strides), offsetof(ia_attn_params, v_scale),
         offsetof(ia_attn_params, kv_valid), offsetof(ia_attn_params, mask),
         offsetof(ia_attn_params, mask_strides), offsetof(ia_attn_params, q_prologue));
  printf("%zu %zu %zu %zu\n", sizeof(ia_qk_prologue), offsetof(ia_qk_prologue, eps),
         offsetof(ia_qk_prologue, rope_stride), offsetof(ia_qk_prologue, k_pos0));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    P = ia.AttnParams
    Q = ia.QKPrologue
    assert [int(x) for x in out] == [ctypes.sizeof(P), P.q_strides.offset, P.lse_strides.offset,
                                     P.v_scale.offset, P.kv_valid.offset, P.mask.offset,
                                     P.mask_strides.offset, P.q_prologue.offset,
                                     ctypes.sizeof(Q), Q.eps.offset, Q.rope_stride.offset,
                                     Q.k_pos0.offset]


def test_params_init_contiguous_strides(lib):
    import int8_qk_quantized_gb300 as ia
    p = ia.AttnParams()
    lib.ia_attn_params_init(ctypes.byref(p), 2, 3, 100, 200, 64, ia.PER_BLOCK64, ia.FP16)
    assert list(p.q_strides) == [3 * 100 * 64, 100 * 64, 64]
    assert list(p.k_strides) == [3 * 200 * 64, 200 * 64, 64]
    assert list(p.qs_strides) == [3 * 2, 2] and list(p.ks_strides) == [3 * 4, 4]
    assert list(p.lse_strides) == [300, 100]
    assert p.sm_scale != p.sm_scale  # NaN selects D^-1/2


def test_status_strings(lib):
    assert lib.ia_status_string(0) == b"ok"
    assert lib.ia_status_string(4) == b"device wait timed out"
    assert lib.ia_version().count(b".") == 2


def _params(lib, D=128, Sq=256, Sk=256):
    import int8_qk_quantized_gb300 as ia
    p = ia.AttnParams()
    lib.ia_attn_params_init(ctypes.byref(p), 1, 2, Sq, Sk, D, ia.PER_TOKEN, ia.BF16)
    return p


def test_argument_errors_reported_before_any_launch(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    null = None
    p = _params(lib, D=96)
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, null, null, fake, null,
                                ctypes.byref(p), null) == 1
    assert b"D must be 64 or 128" in lib.ia_last_error_message()
    assert lib.ia_get_last_error() == 1
    p = _params(lib)
    assert lib.ia_attention_fwd(null, fake, fake, fake, fake, null, null, fake, null,
                                ctypes.byref(p), null) == 1
    mis = ctypes.c_void_p(0x1008)
    assert lib.ia_attention_fwd(fake, fake, fake, fake, mis, null, null, fake, null,
                                ctypes.byref(p), null) == 1
    p.v_strides[2] = 100  # 200 bytes: not a multiple of 16
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, null, null, fake, null,
                                ctypes.byref(p), null) == 1
    p = _params(lib, Sk=100)
    p.kv_valid = 0x1000
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, null, null, fake, null,
                                ctypes.byref(p), null) == 1
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, null, null, fake, null, None,
                                null) == 1
    assert lib.ia_merge_lse(fake, fake, fake, fake, fake, null, 1, 1, 4, 32, 0, null) == 1
    assert lib.ia_merge_lse(fake, fake, fake, fake, fake, null, 1, 1, 4, 64, 7, null) == 1
    st = (ctypes.c_int64 * 3)(128, 128, 128)
    assert lib.ia_quantize_qk(null, null, 0, 1, 1, 8, 8, 128, st, st, 0, 1, null, null, null,
                              null, null, null, null, null) == 1
    assert lib.ia_quantize_qk(fake, null, 0, 1, 1, 8, 8, 128, st, st, 0, 1, null, null, null,
                              null, null, null, null, null) == 1  # q without outputs


def test_empty_problems_are_no_ops(lib):
    fake = ctypes.c_void_p(0x1000)
    p = _params(lib, Sq=0)
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 0
    assert lib.ia_merge_lse(fake, fake, fake, fake, fake, None, 1, 0, 4, 64, 0, None) == 0


def test_no_device_is_a_cuda_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    fake = ctypes.c_void_p(0x1000)
    p = _params(lib)
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 3


def test_binding_raises_when_library_missing(tmp_path, monkeypatch):
    import int8_qk_quantized_gb300 as ia
    monkeypatch.setattr(ia, "_lib", None)
    monkeypatch.setattr(ia, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ia.load_library()


def test_static_workspace_limit_checked_before_any_work(lib):
    import re
    import int8_qk_quantized_gb300 as ia
    m = re.search(r"#define IA_STATIC_WORKSPACE_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(HEADER).read())
    assert m and int(m.group(1)) << int(m.group(2)) == ia.STATIC_WORKSPACE_BYTES
    fake = ctypes.c_void_p(0x1000)
    p = _params(lib, Sq=4096, Sk=4096)
    p.H = 16
    p.kv_splits = 8  # 8 * 16 * 4096 * 129 * 4 bytes of partials > the fixed scratch
    assert lib.ia_attention_workspace_size(ctypes.byref(p)) > ia.STATIC_WORKSPACE_BYTES
    assert lib.ia_attention_fwd_static_workspace(fake, fake, fake, fake, fake, None, None, fake,
                                                 None, ctypes.byref(p), None) == 1
    assert b"fixed workspace" in lib.ia_last_error_message()
    assert lib.ia_attention_fwd_static_workspace(fake, fake, fake, fake, fake, None, None, fake,
                                                 None, None, None) == 1


def test_workspace_holds_the_partials(lib):
    """Key-split scratch: the fp32 O and LSE of every key range."""
    for B, H, Sq, D, n in [(1, 2, 256, 128, 2), (2, 3, 1000, 64, 2), (1, 1, 33, 64, 5),
                           (3, 5, 4097, 64, 3), (1, 1, 1, 64, 2)]:
        p = _params(lib, D=D, Sq=Sq)
        p.B, p.H, p.kv_splits = B, H, n
        assert lib.ia_attention_workspace_size(ctypes.byref(p)) == n * B * H * Sq * (D + 1) * 4
    p.kv_splits = 1
    assert lib.ia_attention_workspace_size(ctypes.byref(p)) == 0


def test_mask_argument_errors(lib):
    fake = ctypes.c_void_p(0x1000)
    p = _params(lib)
    p.mask = 0x1000
    p.mask_strides[:] = [0, 0, 256, 1]
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, fake, None, fake, None,
                                ctypes.byref(p), None) == 1
    assert b"either" in lib.ia_last_error_message()
    p.mask_dtype = 9
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 1
    p.mask_dtype = 0
    p.mask_strides[:] = [0, 0, 256, 2]
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 1
    assert b"key stride" in lib.ia_last_error_message()
    p.mask_strides[:] = [0, 0, 255, 1]  # per-row rows of 1020 bytes: not 16-byte aligned
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 1
    assert b"16-byte" in lib.ia_last_error_message()
    p.mask_strides[:] = [0, 0, 256, 1]
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, fake, fake, None,
                                ctypes.byref(p), None) == 2  # per-row mask with a block mask


def test_prologue_argument_errors(lib):
    import int8_qk_quantized_gb300 as ia
    fake = ctypes.c_void_p(0x1000)
    st = (ctypes.c_int64 * 3)(128 * 64, 64 * 128, 128)
    pr = ia.QKPrologue()
    pr.eps = -1.0
    args = (fake, fake, 0, 1, 1, 64, 64, 128, st, st, 0, 1, None, None, fake, fake, fake, fake, None)
    assert lib.ia_quantize_qk_prologue(*args, ctypes.byref(pr), None) == 1
    assert b"eps" in lib.ia_last_error_message()
    pr.eps = 1e-6
    pr.rope = 2  # split half without tables
    assert lib.ia_quantize_qk_prologue(*args, ctypes.byref(pr), None) == 1
    pr.rope_cos = pr.rope_sin = 0x2000
    pr.rope_stride = 64
    pr.rope_positions = 50  # 64 rows past a 50-position table
    assert lib.ia_quantize_qk_prologue(*args, ctypes.byref(pr), None) == 1
    assert b"rope" in lib.ia_last_error_message()
    pr.rope_positions = 64
    pr.rope_stride = 30  # < D/2
    assert lib.ia_quantize_qk_prologue(*args, ctypes.byref(pr), None) == 1
    p = _params(lib)
    p.q_prologue = ctypes.addressof(pr)
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 1
    assert b"quant_q" in lib.ia_last_error_message()


def test_grid_limits_reported(lib):
    fake = ctypes.c_void_p(0x1000)
    p = _params(lib)
    p.H = 70000
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 2
    p = _params(lib)
    p.B, p.kv_splits = 20000, 4
    p.workspace, p.workspace_bytes = 0x1000, 1 << 62
    assert lib.ia_attention_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                                ctypes.byref(p), None) == 2
    st = (ctypes.c_int64 * 3)(128, 128, 128)
    assert lib.ia_quantize_qk(fake, None, 0, 1, 70000, 8, 8, 128, st, None, 0, 0, None, None,
                              fake, None, fake, None, None, None) == 2
