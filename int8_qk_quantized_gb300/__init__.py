"""INT8-QK quantised attention for GB300 (sm_103a): Python binding of libia.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI in ``include/ia.h``. Torch is used for device memory
and the current stream. If ``libia.so`` has not been built, the first call
raises; there is no fallback implementation.

    q8, qs, k8, ks = quantize_qk(q, k)                  # int8 codes + fp32 scales
    out, lse = attention(q8, k8, qs, ks, v, bias=b, return_lse=True)
    out, lse = merge_lse(o1, l1, o2, l2)
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["quantize_qk", "attention", "merge_lse", "merge_lse_n", "device_status", "IAError", "lib_path",
           "load_library", "AttnParams", "BF16", "FP16", "PER_TOKEN", "PER_BLOCK64"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libia.so")
_lib = None

BF16, FP16 = 0, 1
PER_TOKEN, PER_BLOCK64 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "timeout"}


class IAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


ROPE_LAYOUTS = {None: 0, "none": 0, "interleaved": 1, "split_half": 2}


class QKPrologue(ctypes.Structure):
    """Mirror of ``ia_qk_prologue`` (RMSNorm + RoPE before quantization)."""
    _fields_ = [
        ("q_norm_weight", ctypes.c_void_p), ("k_norm_weight", ctypes.c_void_p),
        ("eps", ctypes.c_float), ("rope", ctypes.c_int),
        ("rope_cos", ctypes.c_void_p), ("rope_sin", ctypes.c_void_p),
        ("rope_stride", ctypes.c_int64), ("rope_positions", ctypes.c_int),
        ("q_pos0", ctypes.c_int), ("k_pos0", ctypes.c_int),
    ]


def make_prologue(q_norm_weight=None, k_norm_weight=None, eps: float = 1e-6, rope=None,
                  cos=None, sin=None, q_pos0: int = 0, k_pos0: int = 0):
    """An ``ia_qk_prologue`` from device tensors: fp32 ``[D]`` norm weights,
    ``rope`` in (None, "interleaved", "split_half") with fp32 ``[P, D/2]``
    cos / sin tables. Returns (struct, tensors kept alive with it)."""
    pr = QKPrologue()
    keep = []
    for name, t in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
        if t is not None:
            if t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous fp32 tensor")
            setattr(pr, name, t.data_ptr())
            keep.append(t)
    pr.eps = float(eps)
    pr.rope = ROPE_LAYOUTS[rope]
    if rope not in (None, "none"):
        if cos is None or sin is None or cos.shape != sin.shape:
            raise ValueError("rope needs cos and sin tables of one shape [P, D/2]")
        for t in (cos, sin):
            if t.dtype != torch.float32 or t.dim() != 2 or t.stride(1) != 1:
                raise ValueError("rope tables must be fp32 [P, D/2] with contiguous rows")
        if cos.stride(0) != sin.stride(0):
            raise ValueError("cos and sin must share the row stride")
        pr.rope_cos, pr.rope_sin = cos.data_ptr(), sin.data_ptr()
        pr.rope_stride = cos.stride(0)
        pr.rope_positions = cos.shape[0]
        keep += [cos, sin]
    pr.q_pos0, pr.k_pos0 = int(q_pos0), int(k_pos0)
    return pr, keep


class AttnParams(ctypes.Structure):
    """Mirror of ``ia_attn_params``."""
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("Sq", ctypes.c_int), ("Sk", ctypes.c_int),
        ("D", ctypes.c_int), ("sm_scale", ctypes.c_float), ("granularity", ctypes.c_int),
        ("v_dtype", ctypes.c_int),
        ("q_strides", ctypes.c_int64 * 3), ("k_strides", ctypes.c_int64 * 3),
        ("qs_strides", ctypes.c_int64 * 2), ("ks_strides", ctypes.c_int64 * 2),
        ("v_strides", ctypes.c_int64 * 3), ("o_strides", ctypes.c_int64 * 3),
        ("lse_strides", ctypes.c_int64 * 2),
        ("v_scale", ctypes.c_void_p), ("kv_valid", ctypes.c_void_p),
        ("kv_splits", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("wait_timeout_ns", ctypes.c_uint64), ("debug_stall", ctypes.c_int),
        ("mask", ctypes.c_void_p), ("mask_dtype", ctypes.c_int),
        ("mask_strides", ctypes.c_int64 * 4), ("q_prologue", ctypes.c_void_p),
    ]


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libia.so (built by ``build_lib.build()``) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "int8_qk_quantized_gb300.build_lib.build() first")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)
    L.ia_quantize_qk.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i64p, i64p, i32, i32,
                                 vp, vp, vp, vp, vp, vp, vp, vp]
    L.ia_quantize_qk.restype = i32
    L.ia_quantize_qk_prologue.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i64p, i64p, i32,
                                          i32, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.POINTER(QKPrologue), vp]
    L.ia_quantize_qk_prologue.restype = i32
    L.ia_attention_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   ctypes.POINTER(AttnParams), vp]
    L.ia_attention_fwd.restype = i32
    L.ia_attention_fwd_quant_q.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(AttnParams), vp]
    L.ia_attention_fwd_quant_q.restype = i32
    L.ia_attention_fwd_static_workspace.argtypes = L.ia_attention_fwd.argtypes
    L.ia_attention_fwd_static_workspace.restype = i32
    L.ia_merge_lse.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    L.ia_merge_lse.restype = i32
    L.ia_merge_lse_n.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, vp, i32, i32,
                                 i32, i32, i32, vp]
    L.ia_merge_lse_n.restype = i32
    L.ia_attention_workspace_size.argtypes = [ctypes.POINTER(AttnParams)]
    L.ia_attention_workspace_size.restype = ctypes.c_size_t
    L.ia_attention_default_splits.argtypes = [ctypes.POINTER(AttnParams), i32]
    L.ia_attention_default_splits.restype = i32
    L.ia_attn_params_init.argtypes = [ctypes.POINTER(AttnParams), i32, i32, i32, i32, i32, i32, i32]
    L.ia_attn_params_init.restype = None
    L.ia_device_status.argtypes = [vp]
    L.ia_device_status.restype = i32
    L.ia_status_string.argtypes = [i32]
    L.ia_status_string.restype = ctypes.c_char_p
    L.ia_last_error_message.argtypes = []
    L.ia_last_error_message.restype = ctypes.c_char_p
    L.ia_get_last_error.argtypes = []
    L.ia_get_last_error.restype = i32
    L.ia_version.argtypes = []
    L.ia_version.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int):
    if status != 0:
        msg = load_library().ia_last_error_message().decode(errors="replace")
        raise IAError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float16:
        return FP16
    raise TypeError(f"16-bit float tensors expected (bf16 or fp16), got {dt}")


def _gran_code(g):
    return {"token": PER_TOKEN, "block64": PER_BLOCK64}[g]


def _strides3(t):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a [B,H,S,D] tensor with a contiguous last dimension")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def quantize_qk(q, k, granularity: str = "token", center_k: bool = True, kv_valid=None,
                k_mean=None, return_mean: bool = False, stream=None, prologue=None,
                two_pass: bool = True):
    """Quantise Q (may be None) and K to INT8 with symmetric fp32 scales.

    ``prologue`` (from ``make_prologue``) applies RMSNorm + RoPE to each row
    first, in the same kernel (``ia_quantize_qk_prologue``). ``two_pass``
    (default) hands the library a buffer for the K mean, which selects its
    mean-then-codes kernels; False leaves it out unless ``return_mean``, which
    selects the single fused kernel (same results).
    Returns ``(q8, q_scale, k8, k_scale)`` (``None`` for a skipped input), plus
    the K mean ``[B,H,D]`` that was used when ``return_mean``.
    """
    L = load_library()
    ref = k if k is not None else q
    B, H, _, D = ref.shape
    dt = _dtype_code(ref.dtype)
    g = _gran_code(granularity)
    dev = ref.device

    def nscale(S):
        return S if g == PER_TOKEN else (S + 63) // 64

    q8 = qs = k8 = ks = None
    Sq = Sk = 0
    if q is not None:
        Sq = q.shape[2]
        q8 = torch.empty((B, H, Sq, D), dtype=torch.int8, device=dev)
        qs = torch.empty((B, H, nscale(Sq)), dtype=torch.float32, device=dev)
    if k is not None:
        Sk = k.shape[2]
        k8 = torch.empty((B, H, Sk, D), dtype=torch.int8, device=dev)
        ks = torch.empty((B, H, nscale(Sk)), dtype=torch.float32, device=dev)
    mu = None
    if k is not None and center_k and (two_pass or return_mean):
        mu = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    if kv_valid is not None:
        kv_valid = kv_valid.to(device=dev, dtype=torch.int32).contiguous()
    if k_mean is not None:
        k_mean = k_mean.to(device=dev, dtype=torch.float32).contiguous()
    args = (_ptr(q), _ptr(k), dt, B, H, Sq, Sk, D,
            _strides3(q) if q is not None else None, _strides3(k) if k is not None else None,
            g, 1 if center_k else 0, _ptr(kv_valid), _ptr(k_mean),
            _ptr(q8), _ptr(k8), _ptr(qs), _ptr(ks), _ptr(mu))
    if prologue is None:
        _check(L.ia_quantize_qk(*args, _stream(stream)))
    else:
        pr = prologue[0] if isinstance(prologue, tuple) else prologue
        _check(L.ia_quantize_qk_prologue(*args, ctypes.byref(pr), _stream(stream)))
    res = (q8, qs, k8, ks)
    return res + (mu,) if return_mean else res


MASK_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.bool: 3}


def _set_mask(p, mask, B, H, Sq, Sk, device):
    """Fill the general-mask fields of ``p`` from a tensor broadcastable to
    [B,H,Sq,Sk]; broadcast dimensions keep stride 0. Returns the tensor the
    pointer refers to."""
    if mask.dtype not in MASK_DTYPES:
        raise ValueError("mask must be float32, bfloat16, float16 or bool")
    if mask.device != device:
        raise ValueError("mask must be on the device of q/k/v")
    m = mask
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4:
        raise ValueError("mask must have at most 4 dimensions")
    if m.shape[3] != 1 and m.stride(3) != 1:
        m = m.contiguous()
    m = m.expand(B, H, Sq, Sk)
    p.mask = m.data_ptr()
    p.mask_dtype = MASK_DTYPES[m.dtype]
    p.mask_strides[:] = [m.stride(i) if m.shape[i] > 1 else 0 for i in range(3)] + [1]
    return m


def _attn_setup(L, q, k8, q_scale, k_scale, v, bias, block_mask, sm_scale, v_scale, kv_valid,
                granularity, return_lse, out, lse, kv_splits, workspace, wait_timeout_ns,
                debug_stall, mask=None):
    """ia_attn_params and the checked tensors of one attention call."""
    B, H, Sq, D = q.shape
    Sk = k8.shape[2]
    p = AttnParams()
    p.B, p.H, p.Sq, p.Sk, p.D = B, H, Sq, Sk, D
    p.sm_scale = float("nan") if sm_scale is None else float(sm_scale)
    p.granularity = _gran_code(granularity)
    p.v_dtype = _dtype_code(v.dtype)
    p.wait_timeout_ns = int(wait_timeout_ns)
    if kv_splits is None:
        kv_splits = L.ia_attention_default_splits(ctypes.byref(p), 1 if block_mask is not None else 0)
    p.kv_splits = int(kv_splits)
    if p.kv_splits > 1:
        need = L.ia_attention_workspace_size(ctypes.byref(p))
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    p.debug_stall = 1 if debug_stall else 0
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=v.dtype, device=v.device)
    if return_lse and lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=v.device)
    for name, t in (("q_strides", q), ("k_strides", k8), ("v_strides", v), ("o_strides", out)):
        s = _strides3(t)
        getattr(p, name)[:] = list(s)
    for name, t in (("qs_strides", q_scale), ("ks_strides", k_scale)):
        if t is None:
            continue
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("scales must be [B,H,n] with a contiguous last dimension")
        getattr(p, name)[:] = [t.stride(0), t.stride(1)]
    if lse is not None:
        if lse.dim() != 3 or lse.stride(2) != 1:
            raise ValueError("lse must be [B,H,Sq] with a contiguous last dimension")
        p.lse_strides[:] = [lse.stride(0), lse.stride(1)]
    if bias is not None:
        bias = bias.reshape(-1)
        if bias.dtype != torch.float32 or bias.numel() != Sk or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32 tensor with Sk elements")
    if block_mask is not None:
        if block_mask.dtype not in (torch.bool, torch.uint8) or not block_mask.is_contiguous():
            raise ValueError("block_mask must be a contiguous bool/uint8 tensor")
        if tuple(block_mask.shape) != (B, H, (Sq + 63) // 64, (Sk + 63) // 64):
            raise ValueError("block_mask must be [B, H, ceil(Sq/64), ceil(Sk/64)]")
    if v_scale is not None:
        v_scale = v_scale.to(device=v.device, dtype=torch.float32).contiguous()
        if v_scale.shape != (H, D):
            raise ValueError("v_scale must be [H, D]")
        p.v_scale = v_scale.data_ptr()
    if kv_valid is not None:
        kv_valid = kv_valid.to(device=v.device, dtype=torch.int32).contiguous()
        p.kv_valid = kv_valid.data_ptr()
    if mask is not None:
        mask = _set_mask(p, mask, B, H, Sq, Sk, v.device)
    # the tensors are returned so that they stay alive until the launch
    return p, out, lse, bias, block_mask, (workspace, v_scale, kv_valid, mask)


def attention(q8, k8, q_scale, k_scale, v, *, bias=None, block_mask=None, sm_scale=None,
              v_scale=None, kv_valid=None, granularity: str = "token", return_lse: bool = False,
              out=None, lse=None, stream=None, kv_splits=None, workspace=None,
              wait_timeout_ns: int = 0, debug_stall: bool = False, mask=None):
    """Forward attention on INT8 Q/K codes with a 16-bit P.V (see ``ia_attention_fwd``).

    ``bias`` is fp32 ``[Sk]`` (any ``[1,1,1,Sk]`` view), ``block_mask`` bool
    ``[B,H,ceil(Sq/64),ceil(Sk/64)]``, ``v_scale`` fp32 ``[H,D]``, ``kv_valid``
    int32 ``[Sk/64]``. ``mask`` (instead of ``bias``) is a float32/bfloat16/
    float16 additive or bool keep mask broadcastable to ``[B,H,Sq,Sk]``; a
    mask that is the same for every query (stride 0 along queries, e.g.
    ``[1,1,1,Sk]`` or an ``expand``-ed view) runs at the cost of a bias.
    ``kv_splits``: None lets the library choose, 1 disables
    the key split; with a split the scratch comes from ``workspace`` (a device
    tensor of at least ``ia_attention_workspace_size`` bytes) or is allocated
    here. Returns ``out`` or ``(out, lse)``.
    """
    L = load_library()
    p, out, lse, bias, block_mask, _keep = _attn_setup(
        L, q8, k8, q_scale, k_scale, v, bias, block_mask, sm_scale, v_scale, kv_valid,
        granularity, return_lse, out, lse, kv_splits, workspace, wait_timeout_ns, debug_stall,
        mask)
    _check(L.ia_attention_fwd(_ptr(q8), _ptr(k8), _ptr(q_scale), _ptr(k_scale), _ptr(v),
                              _ptr(bias), _ptr(block_mask), _ptr(out), _ptr(lse),
                              ctypes.byref(p), _stream(stream)))
    return (out, lse) if return_lse else out


def attention_quant_q(q, k8, k_scale, v, *, bias=None, block_mask=None, sm_scale=None,
                      v_scale=None, kv_valid=None, granularity: str = "token",
                      return_lse: bool = False, out=None, lse=None, stream=None, kv_splits=None,
                      workspace=None, wait_timeout_ns: int = 0, mask=None, prologue=None):
    """Attention with Q quantized inside the kernel (see ``ia_attention_fwd_quant_q``).

    ``q`` is the 16-bit ``[B,H,Sq,D]`` query of V's dtype; ``k8``/``k_scale``
    come from ``quantize_qk(None, k, ...)`` or ``quantize_qk(q, k, ...)``.
    ``prologue`` (from ``make_prologue``) applies its Q-side RMSNorm + RoPE to
    the Q rows before the in-kernel quantization.
    The other arguments and the result are those of ``attention``.
    """
    L = load_library()
    if q.dtype != v.dtype:
        raise ValueError("q and v must share the 16-bit dtype")
    p, out, lse, bias, block_mask, _keep = _attn_setup(
        L, q, k8, None, k_scale, v, bias, block_mask, sm_scale, v_scale, kv_valid, granularity,
        return_lse, out, lse, kv_splits, workspace, wait_timeout_ns, False, mask)
    if prologue is not None:
        pr = prologue[0] if isinstance(prologue, tuple) else prologue
        p.q_prologue = ctypes.addressof(pr)
    _check(L.ia_attention_fwd_quant_q(_ptr(q), _ptr(k8), _ptr(k_scale), _ptr(v), _ptr(bias),
                                      _ptr(block_mask), _ptr(out), _ptr(lse), ctypes.byref(p),
                                      _stream(stream)))
    return (out, lse) if return_lse else out


STATIC_WORKSPACE_BYTES = 64 << 20  # IA_STATIC_WORKSPACE_BYTES: fixed scratch per device


def attention_static_workspace(q8, k8, q_scale, k_scale, v, out, *, lse=None, bias=None,
                               block_mask=None, sm_scale=None, v_scale=None, kv_valid=None,
                               granularity: str = "token", kv_splits: int = 1, stream=None):
    """``ia_attention_fwd_static_workspace``: attention that allocates nothing.

    For callers that cannot allocate device memory per call (a plugin inside
    a runtime that owns the memory, a latency-critical loop that cannot pay
    for cudaMalloc/cudaFree, a fixed memory budget). With ``kv_splits >= 2``
    the partials go to the library's fixed per-device scratch
    (``IA_STATIC_WORKSPACE_BYTES``) instead of a caller workspace. Nothing is
    allocated here either: ``out`` (and ``lse`` if wanted) are given, and
    ``v_scale`` / ``kv_valid`` must already be contiguous fp32 / int32 device
    tensors. Calls that overlap on the GPU share the scratch and race; calls
    on one stream are safe. The first call on a device looks up the scratch
    address, so make it before any stream capture. Returns ``out`` or
    ``(out, lse)`` when ``lse`` is given.
    """
    L = load_library()
    B, H, Sq, D = q8.shape
    Sk = k8.shape[2]
    p = AttnParams()
    p.B, p.H, p.Sq, p.Sk, p.D = B, H, Sq, Sk, D
    p.sm_scale = float("nan") if sm_scale is None else float(sm_scale)
    p.granularity = _gran_code(granularity)
    p.v_dtype = _dtype_code(v.dtype)
    p.kv_splits = int(kv_splits)
    if out.shape != (B, H, Sq, D) or out.dtype != v.dtype:
        raise ValueError("out must be [B,H,Sq,D] of V's dtype")
    for name, t in (("q_strides", q8), ("k_strides", k8), ("v_strides", v), ("o_strides", out)):
        getattr(p, name)[:] = list(_strides3(t))
    for name, t in (("qs_strides", q_scale), ("ks_strides", k_scale)):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("scales must be [B,H,n] with a contiguous last dimension")
        getattr(p, name)[:] = [t.stride(0), t.stride(1)]
    if lse is not None:
        if lse.shape != (B, H, Sq) or lse.dtype != torch.float32 or lse.stride(2) != 1:
            raise ValueError("lse must be fp32 [B,H,Sq] with a contiguous last dimension")
        p.lse_strides[:] = [lse.stride(0), lse.stride(1)]
    if bias is not None:
        bias = bias.reshape(-1)
        if bias.dtype != torch.float32 or bias.numel() != Sk or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32 tensor with Sk elements")
    if block_mask is not None:
        if block_mask.dtype not in (torch.bool, torch.uint8) or not block_mask.is_contiguous():
            raise ValueError("block_mask must be a contiguous bool/uint8 tensor")
        if tuple(block_mask.shape) != (B, H, (Sq + 63) // 64, (Sk + 63) // 64):
            raise ValueError("block_mask must be [B, H, ceil(Sq/64), ceil(Sk/64)]")
    if v_scale is not None:
        if v_scale.shape != (H, D) or v_scale.dtype != torch.float32 or not v_scale.is_contiguous():
            raise ValueError("v_scale must be a contiguous fp32 [H, D] tensor")
        p.v_scale = v_scale.data_ptr()
    if kv_valid is not None:
        if kv_valid.dtype != torch.int32 or not kv_valid.is_contiguous():
            raise ValueError("kv_valid must be a contiguous int32 tensor")
        p.kv_valid = kv_valid.data_ptr()
    _check(L.ia_attention_fwd_static_workspace(
        _ptr(q8), _ptr(k8), _ptr(q_scale), _ptr(k_scale), _ptr(v), _ptr(bias), _ptr(block_mask),
        _ptr(out), _ptr(lse), ctypes.byref(p), _stream(stream)))
    return out if lse is None else (out, lse)


def merge_lse(o1, lse1, o2, lse2, out=None, lse_out=None, stream=None):
    """Exact merge of two partial attentions through their LSEs (contiguous inputs)."""
    L = load_library()
    B, H, Sq, D = o1.shape
    for t in (o1, o2, lse1, lse2):
        if not t.is_contiguous():
            raise ValueError("merge_lse expects contiguous inputs")
    if out is None:
        out = torch.empty_like(o1)
    if lse_out is None:
        lse_out = torch.empty_like(lse1)
    _check(L.ia_merge_lse(_ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _ptr(out), _ptr(lse_out),
                          B, H, Sq, D, _dtype_code(o1.dtype), _stream(stream)))
    return out, lse_out


def merge_lse_n(outs, lses, out=None, lse_out=None, stream=None):
    """Exact merge of n partial attentions (contiguous, same shapes) through their LSEs."""
    L = load_library()
    n = len(outs)
    B, H, Sq, D = outs[0].shape
    for t in list(outs) + list(lses):
        if not t.is_contiguous():
            raise ValueError("merge_lse_n expects contiguous inputs")
    if out is None:
        out = torch.empty_like(outs[0])
    if lse_out is None:
        lse_out = torch.empty_like(lses[0])
    op = (ctypes.c_void_p * n)(*[t.data_ptr() for t in outs])
    lp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lses])
    _check(L.ia_merge_lse_n(op, lp, n, _ptr(out), _ptr(lse_out), B, H, Sq, D,
                            _dtype_code(outs[0].dtype), _stream(stream)))
    return out, lse_out


def device_status(stream=None):
    """Synchronise the stream and raise if a bounded device wait ran out."""
    _check(load_library().ia_device_status(_stream(stream)))
