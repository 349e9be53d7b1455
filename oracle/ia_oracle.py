"""Plain, slow CPU oracle of INT8-QK quantised attention. TEST INFRASTRUCTURE ONLY.

The arithmetic is C++ (``oracle/ia_oracle.cpp``, built by
``oracle/build_oracle.py`` with g++ into ``oracle/_build/libia_oracle.so``, on
first use if needed); this module marshals numpy arrays into it and composes
the steps. Nothing in the product path imports this module; only the tests,
the smoke check and the benchmark's CPU-baseline legs do. It shares no code
with the CUDA library. Arrays are numpy; 16-bit inputs arrive as float32
arrays holding the exact bf16/fp16 values.

Sources (page title, then the part of the page), restated at each C++
function with the step it defines:

* [FastVideo] "minimax_h3_sparse_int8" (FastVideo API page): the module
  description (per-token Q/K scales, K centring as a softmax-invariant shift,
  one V scale per head and channel applied in the epilogue, BF16 PV with FP32
  accumulation, tile-64 keys with partial key tiles masked) and the source of
  ``sparse_sm89_attention`` (the K mean is the sum over the sequence divided
  by the number of valid rows; codes are int8 ``[B,H,S,D]``, scales fp32
  ``[B,H,S]``; the mask is ``[B,H,S/64,S/64]`` and the validity vector has one
  entry per 64-row tile).
* [Passthrough] "Feature Request: Direct int8 Q/K passthrough between Comfy
  Kitchen and SageAttention": section 2.1 (mean_seq, quant_qk_int8, then an
  int8 QK product with a 16-bit PV), section 3.1 (per-block int8 Q/K with
  fp32 scales) and the maintainer's reply (RMSNorm + RoPE on the 16-bit
  values before quantization).
* [model-kernels] "[attention-int8] Multiple build issues and numerical
  accuracy problem": the maintainer's point 1 (symmetric range [-127, 127]).
* [comfy-kitchen] "int8_attention: masked path costs ~1.8x unmasked, and a
  request for optional return_lse": the opening paragraph (one additive bias
  per key, shape [1,1,1,K]), "The measurement" (fp32, bf16 and fp16 additive
  masks and bool masks, [1,1,1,K] or expanded to [1,1,Q,K]), "Question 2"
  (merging two partial softmaxes exactly through their log-sum-exp) and the
  repro (the bool mask is True where the key's weight is kept).
* [FlyDSL] "Add optional forward LSE output": "Summary" (LSE = sm_scale*m +
  ln l, natural log), "Kernel implementation" (-inf for fully masked rows;
  split-K combine from the combined maximum and denominator) and "Public API"
  (fp32 ``[B,H,Sq]``, includes the softmax scale).

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, library routines or invariants; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build_oracle

TILE = 64

PARITY_STATUS = {
    "k_mean": "pinned (exact rational sum on small inputs, translation property)",
    "quantize": "pinned (hand-derived codes, ties, zero rows, error bound)",
    "attention": "pinned (brute-force softmax, torch fp64 SDPA, special cases)",
    "attention(mask=)": "pinned (brute-force masked softmax, bool = 0/-inf, row shifts)",
    "exact_attention": "pinned (torch fp64 SDPA, centring invariance)",
    "merge": "pinned (split of one softmax equals the whole)",
    "qk_prologue": "pinned (torch rms_norm, exact rational sum of squares, complex rotation, "
                   "pair norms, layout permutation, library 16-bit rounding)",
}

_lib = None
_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_I8P = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_VP = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build_oracle.build())
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        L.or_k_mean.argtypes = [_F32P, i32, i32, i32, i32, _VP, _F32P, i32]
        L.or_quantize.argtypes = [_F32P, i32, i32, i32, i32, _VP, i32, _VP, _I8P, _F32P, i32]
        L.or_qk_prologue.argtypes = [_F32P, i32, i32, i32, i32, i32, _VP, f32, i32, _VP, _VP,
                                     i32, _F32P, i32]
        L.or_attention.argtypes = [i32, i32, i32, i32, i32, _VP, i32, _VP, _VP, i32, _VP, i32,
                                   _VP, i32, f64, _VP, _VP, i32, _VP, _VP, _VP, _VP, i32, _VP,
                                   i64, _F64P, _F64P, i32]
        L.or_merge.argtypes = [_F64P, _F64P, _F64P, _F64P, i64, i32, _F64P, _F64P]
        L.or_exact_sum.argtypes = [_F64P, i64, i32]
        L.or_exact_sum.restype = f64
        L.or_hardware_threads.restype = i32
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


_THREADS = 0  # 0: every hardware thread


def set_threads(n: int) -> None:
    """Threads the oracle's C++ loops use (0: all hardware threads)."""
    global _THREADS
    _THREADS = int(n)


def hardware_threads() -> int:
    """std::thread::hardware_concurrency() as the oracle library sees it."""
    return int(_load().or_hardware_threads())


def exact_sum(x, bits: int = 53) -> float:
    """The exact sum of the float64 values ``x`` rounded once to nearest-even
    binary64 (bits=53) or binary32 (bits=24): the summation the K mean and
    the RMSNorm sum of squares are defined with."""
    x = _c(x, np.float64).reshape(-1)
    return float(_load().or_exact_sum(x, x.size, int(bits)))


# --------------------------------------------------------------------------- #
# Quantisation
# --------------------------------------------------------------------------- #

def row_validity(S: int, kv_valid) -> np.ndarray:
    """bool ``[S]``: row s is valid iff s % 64 < kv_valid[s // 64].

    [FastVideo] ``sparse_sm89_attention``: the validity vector holds the
    number of valid rows of each 64-row tile and S == 64 * len(vbs).
    """
    if kv_valid is None:
        return np.ones(S, dtype=bool)
    vbs = np.asarray(kv_valid, dtype=np.int64)
    assert S == TILE * vbs.size
    s = np.arange(S)
    return (s % TILE) < vbs[s // TILE]


def _vbs(kv_valid, S):
    if kv_valid is None:
        return None
    v = _c(kv_valid, np.int32).reshape(-1)
    assert S == TILE * v.size
    return v


def k_mean(k: np.ndarray, kv_valid=None) -> np.ndarray:
    """K's mean over the sequence, fp32 ``[B,H,D]`` (``or_k_mean``).

    [FastVideo] ``sparse_sm89_attention``: the sum of K over the sequence
    divided by the number of valid rows. Reading: the sum is exact, rounded
    once to float64, divided by the count in float64, rounded once to fp32.
    """
    kk = _c(k, np.float32)
    B, H, S, D = kk.shape
    vbs = _vbs(kv_valid, S)
    mu = np.zeros((B, H, D), dtype=np.float32)
    _load().or_k_mean(kk, B, H, S, D, _ptr(vbs), mu, _THREADS)
    return mu


def quantize(x: np.ndarray, mu: np.ndarray | None = None, granularity: str = "token",
             kv_valid=None):
    """Symmetric INT8 quantisation of Q or K (``or_quantize``).

    Returns (codes int8 ``[B,H,S,D]``, scales fp32 ``[B,H,S]`` per token or
    ``[B,H,ceil(S/64)]`` per 64-row block). Per row or 64-row block: x' =
    fp32(x - mu) (K only); amax = max |x'|; scale = fp32(amax / 127); codes =
    round-half-even(fp32(x' * fp32(127 / amax))) clamped to [-127, 127];
    amax = 0 gives codes 0, scale 0; rows past the validity vector are not
    data ([FastVideo]; [model-kernels] point 1; [Passthrough] 3.1).
    """
    xx = _c(x, np.float32)
    B, H, S, D = xx.shape
    if granularity not in ("token", "block64"):
        raise ValueError(granularity)
    m = None if mu is None else _c(mu, np.float32).reshape(B, H, D)
    vbs = _vbs(kv_valid, S)
    nb = S if granularity == "token" else -(-S // TILE)
    codes = np.zeros((B, H, S, D), dtype=np.int8)
    scales = np.zeros((B, H, nb), dtype=np.float32)
    _load().or_quantize(xx, B, H, S, D, _ptr(m), 0 if granularity == "token" else 1, _ptr(vbs),
                        codes, scales, _THREADS)
    return codes, scales


def round_to_16bit(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to bf16 or fp16 (round-half-to-even) and return the
    rounded values as float32 (exact). A library routine: torch's dtype
    conversion for bf16, numpy's float16 for fp16. The tests build 16-bit
    inputs with it and pin the C++ rounding inside :func:`qk_prologue` to it."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "fp16":
        with np.errstate(over="ignore"):  # values past the fp16 range become inf, as they should
            return x.astype(np.float16).astype(np.float32)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).float().numpy()


def qk_prologue(x: np.ndarray, *, dtype: str, norm_weight=None, eps: float = 1e-6,
                rope: str | None = None, cos=None, sin=None, pos0: int = 0) -> np.ndarray:
    """RMSNorm then rotary embedding of each row of Q or K, rounded to the
    16-bit type (``or_qk_prologue``): the activations the unfused path hands
    to attention ([Passthrough] maintainer's reply).

    Reading (the page gives names, not formulas), per row x of D values:
    ss = the exact sum of x_d^2 rounded once to fp32; ms = fp32(ss / D);
    r = fp32(1 / fp32(sqrt(fp32(ms + eps)))); y_d = fp32(fp32(x_d r) w_d);
    then pair i = (y[2i], y[2i+1]) ("interleaved") or (y[i], y[i + D/2])
    ("split_half") is rotated: a' = fp32(fp32(a c) - fp32(b s)), b' =
    fp32(fp32(a s) + fp32(b c)) with c = cos[p, i], s = sin[p, i] at position
    p = pos0 + row; one rounding to the 16-bit type at the end. ``cos`` /
    ``sin`` are fp32 ``[P, D/2]``. Returns float32 holding 16-bit values.
    """
    xx = _c(x, np.float32)
    B, H, S, D = xx.shape
    w = None if norm_weight is None else _c(norm_weight, np.float32).reshape(D)
    code = {None: 0, "none": 0, "interleaved": 1, "split_half": 2}[rope]
    c = s = None
    if code:
        c = _c(cos, np.float32)
        s = _c(sin, np.float32)
        assert c.shape == s.shape and c.shape[1] == D // 2 and pos0 + S <= c.shape[0]
    y = np.empty_like(xx)
    _load().or_qk_prologue(xx, B, H, S, D, 0 if dtype == "bf16" else 1, _ptr(w), float(eps),
                           code, _ptr(c), _ptr(s), int(pos0), y, _THREADS)
    return y


# --------------------------------------------------------------------------- #
# Attention
# --------------------------------------------------------------------------- #

def _mask_args(mask, B, H, Sq, Sk):
    """A general attention mask broadcastable to [B,H,Sq,Sk] (the [1,1,1,K] and
    [1,1,Q,K] views of [comfy-kitchen] "The measurement") as the C++ call
    takes it: (kind, array, element strides with 0 on broadcast dims). A float
    mask holds additive logit offsets (the exact bf16/fp16/fp32 values, widened
    to float64); a bool mask keeps a key where it is True."""
    if mask is None:
        return 0, None, None
    m = np.asarray(mask)
    while m.ndim < 4:
        m = m[None]
    if m.dtype == np.bool_:
        kind, arr = 2, _c(m, np.uint8)
    else:
        kind, arr = 1, _c(m.astype(np.float64), np.float64)
    full = (B, H, Sq, Sk)
    st = []
    for ax in range(4):
        if arr.shape[ax] == full[ax]:
            st.append(arr.strides[ax] // arr.itemsize)
        elif arr.shape[ax] == 1:
            st.append(0)
        else:
            raise ValueError(f"mask shape {m.shape} does not broadcast to {full}")
    return kind, arr, np.array(st, dtype=np.int64)


def _values(a):
    """A float operand as the C++ call takes it: (kind, array); float32 stays
    float32 (16-bit values are exact in it), anything else becomes float64."""
    a = np.asarray(a)
    if a.dtype == np.float32:
        return 1, _c(a, np.float32)
    return 2, _c(a, np.float64)


def _attend(q, q_kind, q_scale, k, k_kind, k_scale, v, *, sm_scale, bias, block_mask, kv_valid,
            v_scale, granularity, rows, mask, pad_query):
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if sm_scale is None:
        sm_scale = D ** -0.5
    rows = np.arange(Sq, dtype=np.int64) if rows is None else _c(rows, np.int64).reshape(-1)
    v_kind, vv = _values(v)
    bias64 = None if bias is None else _c(bias, np.float64).reshape(-1)
    assert bias64 is None or bias64.size == Sk
    bm = None if block_mask is None else _c(block_mask, np.uint8)
    vbs = _vbs(kv_valid, Sk)
    vs = None if v_scale is None else _c(v_scale, np.float64).reshape(H, D)
    kind, marr, mst = _mask_args(mask, B, H, Sq, Sk)
    out = np.zeros((B, H, rows.size, D), dtype=np.float64)
    lse = np.zeros((B, H, rows.size), dtype=np.float64)
    if rows.size == 0:
        return out, lse
    _load().or_attention(B, H, Sq, Sk, D, _ptr(q), q_kind, _ptr(q_scale), _ptr(k), k_kind,
                         _ptr(k_scale), 0 if granularity == "token" else 1, _ptr(vv), v_kind,
                         float(sm_scale), _ptr(bias64), _ptr(marr), kind, _ptr(mst), _ptr(bm),
                         _ptr(vbs), _ptr(vs), 1 if pad_query else 0, _ptr(rows), rows.size, out,
                         lse, _THREADS)
    return out, lse


def attention(q_codes, q_scale, k_codes, k_scale, v, *, sm_scale=None, bias=None,
              block_mask=None, kv_valid=None, v_scale=None, granularity="token",
              rows=None, row_chunk=256, mask=None):
    """Same-quantisation FP64 attention reference (``or_attention``).

    q_hat = code * scale and k_hat likewise (float64);
    s_ij = sm_scale * <q_hat_i, k_hat_j> + bias_j (+ a float mask), with
    s_ij = -inf where the tile-64 block mask drops key tile j//64 for query
    tile i//64, key row j lies past the validity vector or a bool mask is
    False; O_i = v_scale (*) sum_j softmax_j(s_i.) v_j; LSE_i = m_i +
    ln sum_j e^(s_ij - m_i). A fully masked row gives O = 0, LSE = -inf.

    Readings: the bias and masks enter after the softmax scale (SDPA's
    additive ``attn_mask``, which [comfy-kitchen] compares against); with a
    validity vector and Sq == Sk, query rows past it are padding and give
    O = 0 and LSE = -inf. ``rows`` optionally restricts the query rows (a
    1-D index array). ``row_chunk`` is accepted for compatibility and unused.
    Returns (O float64 [B,H,n,D], LSE float64 [B,H,n]).
    """
    qc = _c(q_codes, np.int8)
    kc = _c(k_codes, np.int8)
    Sq, Sk = qc.shape[2], kc.shape[2]
    return _attend(qc, 0, _c(q_scale, np.float32), kc, 0, _c(k_scale, np.float32), v,
                   sm_scale=sm_scale, bias=bias, block_mask=block_mask, kv_valid=kv_valid,
                   v_scale=v_scale, granularity=granularity, rows=rows, mask=mask,
                   pad_query=kv_valid is not None and Sq == Sk)


def exact_attention(q, k, v, *, sm_scale=None, bias=None, block_mask=None, kv_valid=None,
                    v_scale=None, rows=None, row_chunk=256, mask=None):
    """Textbook softmax attention in float64 on the unquantised inputs (no
    centring, no quantisation): the yardstick the INT8 path is measured
    against ([model-kernels] "5. Numerical accuracy" compares against SDPA).
    Same masking, bias, V scale and LSE conventions as :func:`attention`
    (padding query rows are not zeroed here)."""
    qk, qa = _values(q)
    kk, ka = _values(k)
    return _attend(qa, qk, None, ka, kk, None, v,
                   sm_scale=sm_scale, bias=bias, block_mask=block_mask, kv_valid=kv_valid,
                   v_scale=v_scale, granularity="token", rows=rows, mask=mask, pad_query=False)


def merge(o1, lse1, o2, lse2):
    """Exact merge of two partial softmax attentions over disjoint key sets
    (``or_merge``): M = max(L1, L2); w_k = e^(L_k - M); L = M + ln(w1 + w2);
    O = (w1 O1 + w2 O2) / (w1 + w2); both -inf gives O = 0, L = -inf.
    [comfy-kitchen] "Question 2"; [FlyDSL] "Kernel implementation". float64."""
    a1 = _c(o1, np.float64)
    a2 = _c(o2, np.float64)
    b1 = _c(lse1, np.float64)
    b2 = _c(lse2, np.float64)
    D = a1.shape[-1]
    n = b1.size
    o = np.zeros_like(a1)
    l = np.zeros_like(b1)
    _load().or_merge(a1.reshape(n, D), b1.reshape(n), a2.reshape(n, D), b2.reshape(n), n, D,
                     o.reshape(n, D), l.reshape(n))
    return o, l


def quantize_and_attend(q, k, v, *, granularity="token", center_k=True, kv_valid=None,
                        k_mu=None, prologue=None, **attn_kw):
    """The whole path on CPU: optional RMSNorm + RoPE of Q and K
    (:func:`qk_prologue`; ``prologue`` holds ``dtype``, ``q_norm_weight``,
    ``k_norm_weight``, ``eps``, ``rope``, ``cos``, ``sin``, ``q_pos0``,
    ``k_pos0``), K mean, quantise Q and K, same-quantisation attention.
    Returns (O, LSE, (q_codes, q_scale, k_codes, k_scale, mu))."""
    qv = np.asarray(q, dtype=np.float32)
    kv = np.asarray(k, dtype=np.float32)
    if prologue is not None:
        pr = dict(prologue)
        common = dict(dtype=pr["dtype"], eps=pr.get("eps", 1e-6), rope=pr.get("rope"),
                      cos=pr.get("cos"), sin=pr.get("sin"))
        qv = qk_prologue(qv, norm_weight=pr.get("q_norm_weight"), pos0=pr.get("q_pos0", 0),
                         **common)
        kv = qk_prologue(kv, norm_weight=pr.get("k_norm_weight"), pos0=pr.get("k_pos0", 0),
                         **common)
        if kv_valid is not None:  # padding rows stay zero, as the contract has them
            kv = np.where(row_validity(kv.shape[2], kv_valid)[None, None, :, None], kv, 0)
            if qv.shape[2] == kv.shape[2]:
                qv = np.where(row_validity(qv.shape[2], kv_valid)[None, None, :, None], qv, 0)
    mu = None
    if center_k:
        mu = k_mean(kv, kv_valid) if k_mu is None else np.asarray(k_mu, np.float32)
    qc, qs = quantize(qv, None, granularity, kv_valid if qv.shape[2] == kv.shape[2] else None)
    kc, ks = quantize(kv, mu, granularity, kv_valid)
    o, lse = attention(qc, qs, kc, ks, v, granularity=granularity, kv_valid=kv_valid, **attn_kw)
    return o, lse, (qc, qs, kc, ks, mu)
