"""Plain, slow CPU oracle of INT8-QK quantised attention. TEST INFRASTRUCTURE ONLY.

Nothing in the product path imports this module; only the tests, the smoke
check and the benchmark's CPU-baseline leg do. It shares no code with the CUDA
library. Arrays are numpy; 16-bit inputs arrive as float32 arrays holding the
exact bf16/fp16 values.

Sources (page title, then the part of the page):

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
  int8 QK product with a 16-bit PV) and section 3.1 (per-block int8 Q/K with
  fp32 scales).
* [model-kernels] "[attention-int8] Multiple build issues and numerical
  accuracy problem": the maintainer's point 1 (symmetric range [-127, 127]).
* [comfy-kitchen] "int8_attention: masked path costs ~1.8x unmasked, and a
  request for optional return_lse": the opening paragraph (one additive bias
  per key, shape [1,1,1,K]) and "Question 2" (merging two partial softmaxes
  exactly through their log-sum-exp).
* [comfy-kitchen] "The measurement" (the attn_mask forms callers pass: fp32,
  bf16 and fp16 additive masks and bool masks, shaped [1,1,1,K] or expanded
  to [1,1,Q,K]) and the repro (the bool mask is True where the key's weight
  is kept).
* [Passthrough], the maintainer's reply: RMSNorm + RoPE sit between the
  projections and attention in modern DiTs (``apply_rope``, ``rms_rope``,
  ``rms_rope_split_half``) and must run on the 16-bit values.
* [FlyDSL] "Add optional forward LSE output": "Summary" (LSE = sm_scale*m +
  ln l, natural log), "Kernel implementation" (-inf for fully masked rows;
  split-K combine from the combined maximum and denominator) and "Public API"
  (fp32 ``[B,H,Sq]``, includes the softmax scale).

Readings where the pages leave a step open are stated at each function.

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, library routines or invariants; none is
"parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

TILE = 64
QMAX = np.float32(127.0)

PARITY_STATUS = {
    "k_mean": "pinned (exact rational sum on small inputs, translation property)",
    "quantize": "pinned (hand-derived codes, ties, zero rows, error bound)",
    "attention": "pinned (brute-force softmax, torch fp64 SDPA, special cases)",
    "attention(mask=)": "pinned (brute-force masked softmax, bool = 0/-inf, row shifts)",
    "exact_attention": "pinned (torch fp64 SDPA, centring invariance)",
    "merge": "pinned (split of one softmax equals the whole)",
    "qk_prologue": "pinned (torch rms_norm, complex rotation, pair norms, layout permutation)",
}


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


def k_mean(k: np.ndarray, kv_valid=None) -> np.ndarray:
    """K's mean over the sequence, fp32 ``[B,H,D]``.

    [FastVideo] ``sparse_sm89_attention``: the sum of K over the sequence
    divided by the number of valid rows (tile pads are zero, so the sum over
    all rows is the sum over the valid ones). [Passthrough] 2.1 calls this
    step mean_seq (smooth_k).

    Reading: the page sums in fp32 in an unspecified order. Here the sum is
    exact (``math.fsum`` gives the exact sum rounded once to float64), divided
    by the count in float64 and rounded once to float32.
    """
    B, H, S, D = k.shape
    valid = row_validity(S, kv_valid)
    n = int(valid.sum())
    mu = np.zeros((B, H, D), dtype=np.float32)
    kv = np.asarray(k, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for d in range(D):
                col = kv[b, h, valid, d]
                total = math.fsum(col.tolist())
                mu[b, h, d] = np.float32(total / max(n, 1))
    return mu


def quantize(x: np.ndarray, mu: np.ndarray | None = None, granularity: str = "token",
             kv_valid=None):
    """Symmetric INT8 quantisation of Q or K.

    Returns (codes int8 ``[B,H,S,D]``, scales fp32 ``[B,H,S]`` per token or
    ``[B,H,ceil(S/64)]`` per 64-row block).

    Steps, per row (per token) or per 64-row block:
      1. centre: x' = fp32(x - mu) when ``mu`` is given (K only)
         [FastVideo] module description, K centring;
      2. amax = max |x'| over the row or block (exact);
      3. scale = fp32(amax / 127); codes = round-half-even(fp32(x' * fp32(127 /
         amax))) clamped to [-127, 127] -- symmetric range, [model-kernels]
         maintainer point 1; per-token scales [FastVideo]; per-block scales
         [Passthrough] 3.1.
      4. amax == 0 gives codes 0 and scale 0. Rows past the validity vector
         are not data: codes 0, and they do not enter a block's amax; a
         per-token scale of such a row is 0.

    Reading: the pages fix neither the rounding mode nor divide versus
    reciprocal. This uses round-half-to-even of the product with the
    correctly rounded fp32 reciprocal 127/amax.
    """
    B, H, S, D = x.shape
    xc = np.asarray(x, dtype=np.float32)
    if mu is not None:
        xc = (xc - np.asarray(mu, dtype=np.float32)[:, :, None, :]).astype(np.float32)
    valid = row_validity(S, kv_valid)
    xc = np.where(valid[None, None, :, None], xc, np.float32(0)).astype(np.float32)
    absx = np.abs(xc)
    if granularity == "token":
        amax = absx.max(axis=3)                                   # [B,H,S]
        amax_rows = amax
    elif granularity == "block64":
        nb = -(-S // TILE)
        amax = np.zeros((B, H, nb), dtype=np.float32)
        for t in range(nb):
            amax[:, :, t] = absx[:, :, t * TILE:(t + 1) * TILE, :].max(axis=(2, 3))
        amax_rows = np.repeat(amax, TILE, axis=2)[:, :, :S]
    else:
        raise ValueError(granularity)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1)).astype(np.float32)
    scale = np.where(nz, (safe / QMAX).astype(np.float32), np.float32(0)).astype(np.float32)
    nz_rows = amax_rows > 0
    safe_rows = np.where(nz_rows, amax_rows, np.float32(1)).astype(np.float32)
    inv_rows = (QMAX / safe_rows).astype(np.float32)              # fp32(127 / amax)
    prod = (xc * inv_rows[..., None]).astype(np.float32)         # fp32 product
    codes = np.clip(np.rint(prod), -127, 127)
    codes = np.where(nz_rows[..., None], codes, 0).astype(np.int8)
    return codes, scale


def round_to_16bit(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to bf16 or fp16 (round-half-to-even) and return the
    rounded values as float32 (exact). torch's dtype conversion is the library
    routine used for bf16; numpy's float16 for fp16."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "fp16":
        return x.astype(np.float16).astype(np.float32)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).float().numpy()


def qk_prologue(x: np.ndarray, *, dtype: str, norm_weight=None, eps: float = 1e-6,
                rope: str | None = None, cos=None, sin=None, pos0: int = 0) -> np.ndarray:
    """RMSNorm then rotary embedding of each row of Q or K, rounded to the
    16-bit type: the activations the unfused path hands to attention.

    [Passthrough] maintainer's reply: in modern DiTs the projections go
    through RMSNorm + RoPE before attention (``apply_rope``, ``rms_rope``,
    ``rms_rope_split_half``), and RoPE rotates channel pairs, so it has to run
    on the 16-bit values before they are quantized.

    Reading (the page gives names, not formulas), per row x of D values:
      1. RMSNorm (when ``norm_weight`` is given): ss = the fp32 sum of the
         squares x_d^2 (each exact in fp32 for 16-bit x) in a fixed order --
         the squares of each 8 consecutive channels summed in index order,
         then the D/8 partial sums added pairwise, t with t + n/2, until one
         remains; ms = fp32(ss / D); r = fp32(1 / fp32(sqrt(fp32(ms + eps))));
         y_d = fp32(fp32(x_d * r) * w_d). All fp32 steps are correctly rounded.
         The order is the one the GPU kernels use (the pages fix none), so the
         16-bit results, and the codes decided from them, agree bit for bit.
      2. RoPE (when ``rope`` is "interleaved" or "split_half"): pair i is
         (y[2i], y[2i+1]) or (y[i], y[i + D/2]); with c = cos[p, i],
         s = sin[p, i] for the row's position p = pos0 + row:
         a' = fp32(fp32(a c) - fp32(b s)), b' = fp32(fp32(a s) + fp32(b c)),
         the rotation of (a, b) by the angle whose cosine and sine are given.
      3. one rounding to the 16-bit type.
    ``cos`` / ``sin`` are fp32 ``[P, D/2]`` tables. Returns float32 holding
    16-bit values, same shape as ``x``.
    """
    B, H, S, D = x.shape
    y = np.asarray(x, dtype=np.float32).copy()
    if norm_weight is not None:
        w = np.asarray(norm_weight, dtype=np.float32)
        sq = (y * y).astype(np.float32)                                  # exact squares
        part = sq[..., 0::8].copy()                                      # [B,H,S,D/8]
        for j in range(1, 8):
            part = (part + sq[..., j::8]).astype(np.float32)             # index order
        n = D // 8
        while n > 1:
            half = n // 2
            part = (part[..., :half] + part[..., half:n]).astype(np.float32)
            n = half
        ss = part[..., 0]
        ms = (ss / np.float32(D)).astype(np.float32)
        rr = (np.float32(1) / np.sqrt((ms + np.float32(eps)).astype(np.float32))).astype(np.float32)
        y = ((y * rr[..., None]).astype(np.float32) * w).astype(np.float32)
    if rope is not None:
        c = np.asarray(cos, dtype=np.float32)[pos0:pos0 + S]        # [S, D/2]
        sn = np.asarray(sin, dtype=np.float32)[pos0:pos0 + S]
        if rope == "interleaved":
            a, bb = y[..., 0::2], y[..., 1::2]
        elif rope == "split_half":
            a, bb = y[..., :D // 2], y[..., D // 2:]
        else:
            raise ValueError(rope)
        a2 = ((a * c).astype(np.float32) - (bb * sn).astype(np.float32)).astype(np.float32)
        b2 = ((a * sn).astype(np.float32) + (bb * c).astype(np.float32)).astype(np.float32)
        y = np.empty_like(y)
        if rope == "interleaved":
            y[..., 0::2], y[..., 1::2] = a2, b2
        else:
            y[..., :D // 2], y[..., D // 2:] = a2, b2
    return round_to_16bit(y, dtype)


def dequantize(codes: np.ndarray, scale: np.ndarray, granularity: str) -> np.ndarray:
    """code * scale in float64, ``[B,H,S,D]``."""
    S = codes.shape[2]
    if granularity == "token":
        s = np.asarray(scale, dtype=np.float64)
    else:
        s = np.repeat(np.asarray(scale, dtype=np.float64), TILE, axis=2)[:, :, :S]
    return codes.astype(np.float64) * s[..., None]


# --------------------------------------------------------------------------- #
# Attention
# --------------------------------------------------------------------------- #

def _softmax_rows(s: np.ndarray, v: np.ndarray):
    """Per-row softmax of the logits ``s`` [n, Sk] (natural log units) applied to
    ``v`` [Sk, D]. Returns (O [n, D], LSE [n]). A row whose logits are all -inf
    gives O = 0 and LSE = -inf ([FlyDSL] "Kernel implementation")."""
    m = s.max(axis=1)
    dead = ~np.isfinite(m)
    m_safe = np.where(dead, 0.0, m)
    p = np.exp(s - m_safe[:, None])
    p[dead] = 0.0
    l = p.sum(axis=1)
    o = p @ v
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(dead[:, None], 0.0, o / np.where(dead, 1.0, l)[:, None])
        lse = np.where(dead, -np.inf, m_safe + np.log(np.where(dead, 1.0, l)))
    return o, lse


def _key_mask(b, h, rows, Sk, block_mask, kv_valid):
    """Boolean [len(rows), Sk]: key j is visible to query row i."""
    vis = np.ones((len(rows), Sk), dtype=bool)
    if block_mask is not None:
        bm = np.asarray(block_mask)[b, h]                        # [Tq, Tk]
        tiles = bm[np.asarray(rows) // TILE]                     # [n, Tk]
        vis &= np.repeat(tiles, TILE, axis=1)[:, :Sk]
    if kv_valid is not None:
        vis &= row_validity(Sk, kv_valid)[None, :]
    return vis


def _mask_rows(mask, B, H, Sq, Sk, b, h, rows):
    """Rows ``rows`` of head (b, h) of a general attention mask.

    ``mask`` is broadcastable to [B,H,Sq,Sk] (numpy broadcasting, as the
    [1,1,1,K] and [1,1,Q,K] views of [comfy-kitchen] "The measurement"). A
    float mask holds additive logit offsets (the exact bf16/fp16/fp32 values,
    widened to float64); a bool mask keeps a key where it is True and
    excludes it (logit -inf) where it is False.
    Returns ("add", float64 [n, Sk]) or ("keep", bool [n, Sk])."""
    m = np.asarray(mask)
    while m.ndim < 4:
        m = m[None]
    full = np.broadcast_to(m, (B, H, Sq, Sk))[b, h][np.asarray(rows)]
    if full.dtype == np.bool_:
        return "keep", full
    return "add", full.astype(np.float64)


def _apply_mask(s, kind_rows):
    kind, mr = kind_rows
    if kind == "keep":
        return np.where(mr, s, -np.inf)
    return s + mr


def attention(q_codes, q_scale, k_codes, k_scale, v, *, sm_scale=None, bias=None,
              block_mask=None, kv_valid=None, v_scale=None, granularity="token",
              rows=None, row_chunk=256, mask=None):
    """Same-quantisation FP64 attention reference.

    q_hat = code * scale and k_hat likewise (float64);
    s_ij = sm_scale * <q_hat_i, k_hat_j> + bias_j, with s_ij = -inf where the
    tile-64 block mask drops key tile j//64 for query tile i//64 or key row j
    lies past the validity vector;
    O_i = v_scale (*) sum_j softmax_j(s_i.) v_j;  LSE_i = m_i + ln sum_j e^(s_ij - m_i).

    [Passthrough] 2.1 (int8 QK, 16-bit PV); [FastVideo] module description
    (FP32 accumulation, V scale per head and channel applied once at the end,
    masked partial key tiles) and ``sparse_sm89_attention`` (mask layout);
    [comfy-kitchen] opening paragraph (bias [1,1,1,K]); [FlyDSL] "Summary" and
    "Public API" (LSE in natural log including the softmax scale).

    Reading: the bias is added after the softmax scale, as an additive
    ``attn_mask`` is in SDPA, which [comfy-kitchen] compares against.

    Reading: with a validity vector and Sq == Sk, query rows past it are
    padding; they give O = 0 and LSE = -inf (the pages leave them undefined).

    ``mask`` is the general form of the bias (see :func:`_mask_rows`): a float
    mask broadcastable to [B,H,Sq,Sk] is added where ``bias`` would be; a bool
    mask excludes the keys where it is False.

    ``rows`` optionally restricts the query rows (a 1-D index array); rows are
    independent, so they are processed in chunks of ``row_chunk``.
    Returns (O float64 [B,H,n,D], LSE float64 [B,H,n]).
    """
    B, H, Sq, D = q_codes.shape
    Sk = k_codes.shape[2]
    if sm_scale is None:
        sm_scale = D ** -0.5
    qh = dequantize(q_codes, q_scale, granularity)
    kh = dequantize(k_codes, k_scale, granularity)
    vv = np.asarray(v, dtype=np.float64)
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    out = np.zeros((B, H, len(rows), D))
    lse = np.zeros((B, H, len(rows)))
    bias64 = None if bias is None else np.asarray(bias, dtype=np.float64).reshape(-1)
    for b in range(B):
        for h in range(H):
            for c0 in range(0, len(rows), row_chunk):
                r = rows[c0:c0 + row_chunk]
                s = sm_scale * (qh[b, h, r] @ kh[b, h].T)
                if bias64 is not None:
                    s = s + bias64[None, :]
                if mask is not None:
                    s = _apply_mask(s, _mask_rows(mask, B, H, Sq, Sk, b, h, r))
                vis = _key_mask(b, h, r, Sk, block_mask, kv_valid)
                s = np.where(vis, s, -np.inf)
                o, l = _softmax_rows(s, vv[b, h])
                if v_scale is not None:
                    o = o * np.asarray(v_scale, dtype=np.float64)[h][None, :]
                if kv_valid is not None and Sq == Sk:
                    pad = ~row_validity(Sq, kv_valid)[r]
                    o[pad] = 0.0
                    l[pad] = -np.inf
                out[b, h, c0:c0 + len(r)] = o
                lse[b, h, c0:c0 + len(r)] = l
    return out, lse


def exact_attention(q, k, v, *, sm_scale=None, bias=None, block_mask=None, kv_valid=None,
                    v_scale=None, rows=None, row_chunk=256, mask=None):
    """Textbook softmax attention in float64 on the unquantised inputs (no
    centring, no quantisation): the yardstick the INT8 path is measured
    against ([model-kernels] "5. Numerical accuracy" compares against SDPA).
    Same masking, bias, V scale and LSE conventions as :func:`attention`."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if sm_scale is None:
        sm_scale = D ** -0.5
    qq = np.asarray(q, dtype=np.float64)
    kk = np.asarray(k, dtype=np.float64)
    vv = np.asarray(v, dtype=np.float64)
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    out = np.zeros((B, H, len(rows), D))
    lse = np.zeros((B, H, len(rows)))
    bias64 = None if bias is None else np.asarray(bias, dtype=np.float64).reshape(-1)
    for b in range(B):
        for h in range(H):
            for c0 in range(0, len(rows), row_chunk):
                r = rows[c0:c0 + row_chunk]
                s = sm_scale * (qq[b, h, r] @ kk[b, h].T)
                if bias64 is not None:
                    s = s + bias64[None, :]
                if mask is not None:
                    s = _apply_mask(s, _mask_rows(mask, B, H, Sq, Sk, b, h, r))
                vis = _key_mask(b, h, r, Sk, block_mask, kv_valid)
                s = np.where(vis, s, -np.inf)
                o, l = _softmax_rows(s, vv[b, h])
                if v_scale is not None:
                    o = o * np.asarray(v_scale, dtype=np.float64)[h][None, :]
                out[b, h, c0:c0 + len(r)] = o
                lse[b, h, c0:c0 + len(r)] = l
    return out, lse


def merge(o1, lse1, o2, lse2):
    """Exact merge of two partial softmax attentions over disjoint key sets.

    M = max(L1, L2); w_k = e^(L_k - M); L = M + ln(w1 + w2);
    O = (w1 O1 + w2 O2) / (w1 + w2); if both are -inf, O = 0 and L = -inf.
    [comfy-kitchen] "Question 2"; [FlyDSL] "Kernel implementation" (split-K
    combine from the combined maximum and denominator). float64.
    """
    l1 = np.asarray(lse1, dtype=np.float64)
    l2 = np.asarray(lse2, dtype=np.float64)
    o1 = np.asarray(o1, dtype=np.float64)
    o2 = np.asarray(o2, dtype=np.float64)
    m = np.maximum(l1, l2)
    dead = ~np.isfinite(m)
    ms = np.where(dead, 0.0, m)
    w1 = np.where(np.isfinite(l1), np.exp(l1 - ms), 0.0)
    w2 = np.where(np.isfinite(l2), np.exp(l2 - ms), 0.0)
    den = w1 + w2
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(dead[..., None], 0.0,
                     (w1[..., None] * o1 + w2[..., None] * o2) / np.where(dead, 1.0, den)[..., None])
        lse = np.where(dead, -np.inf, ms + np.log(np.where(dead, 1.0, den)))
    return o, lse


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
