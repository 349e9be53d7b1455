/*
 * ia.h -- C ABI of the INT8-QK attention library (libia.so) for NVIDIA GB300 (sm_103a).
 *
 * Forward softmax attention with symmetric INT8 Q/K, an optional per-key
 * additive bias, an optional tile-64 block-sparse key mask, a 16-bit P.V
 * accumulated in FP32, an optional per-(head, channel) V scale and an optional
 * natural-log LSE output, plus the quantisation pass in front of it and the
 * exact two-partial merge behind it.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers on the current CUDA device unless stated.
 *     The caller owns every buffer; the library allocates nothing on the
 *     device, keeps no per-call state and never synchronises: each call only
 *     enqueues kernels on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and returns.
 *   - Tensors are [B, H, S, D] ("BHSD") with the last dimension contiguous.
 *     Strides are in ELEMENTS of the tensor's own type, ordered (b, h, s).
 *   - Errors in the arguments are detected on the host before anything is
 *     enqueued and returned as IA_ERR_INVALID_ARG / IA_ERR_UNSUPPORTED; a
 *     failed launch returns IA_ERR_CUDA. ia_last_error_message() then holds a
 *     one-line description (thread-local).
 *   - Device-side waits inside the attention kernel are bounded. If one runs
 *     out, the kernel records IA_ERR_TIMEOUT in a device status word and
 *     returns instead of hanging; ia_device_status() reads and clears it.
 *   - Only sm_103 devices are supported (IA_ERR_UNSUPPORTED otherwise).
 */
#ifndef IA_H_
#define IA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define IA_API __attribute__((visibility("default")))
#else
#define IA_API
#endif

typedef enum ia_status {
  IA_OK = 0,
  IA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad shape or stride */
  IA_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement */
  IA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  IA_ERR_TIMEOUT = 4      /* a bounded device-side wait ran out */
} ia_status;

typedef enum ia_dtype { IA_BF16 = 0, IA_FP16 = 1 } ia_dtype;

/* One fp32 scale per row ("per token") or per 64-row block of a head. */
typedef enum ia_granularity { IA_PER_TOKEN = 0, IA_PER_BLOCK64 = 1 } ia_granularity;

/* Channel pairing of a rotary embedding (ia_qk_prologue.rope). */
typedef enum ia_rope_layout {
  IA_ROPE_NONE = 0,        /* no rotation */
  IA_ROPE_INTERLEAVED = 1, /* pairs (2i, 2i+1) */
  IA_ROPE_SPLIT_HALF = 2   /* pairs (i, i + D/2) */
} ia_rope_layout;

/*
 * RMSNorm + RoPE applied to each Q / K row before it is quantized: the step
 * that "Feature Request: Direct int8 Q/K passthrough between Comfy Kitchen
 * and SageAttention" (maintainer's reply) places between the projections and
 * attention in modern DiTs (rms_rope, apply_rope, rms_rope_split_half). Per
 * row x of D values, with every fp32 operation correctly rounded:
 *   RMSNorm (weight given): ss = fp32 sum of x_d^2 in a fixed order (the
 *     squares of each 8 consecutive channels in index order, then the D/8
 *     partial sums added pairwise, t with t + n/2, until one remains),
 *     r = 1 / sqrt(ss / D + eps), y_d = (x_d * r) * w_d;
 *   RoPE (rope != NONE): pair i = (y_a, y_b), c = cos[p][i], s = sin[p][i] at
 *     the row's position p = pos0 + row: y_a' = y_a c - y_b s, y_b' = y_a s + y_b c;
 *   then one rounding to the input's 16-bit type; the K mean and the
 *   quantization then see these values. Padding rows (past kv_valid) stay 0.
 * The fixed order makes the result the same bit for bit in every kernel that
 * applies the prologue (ia_quantize_qk_prologue, ia_attention_fwd_quant_q).
 * The order is this library's choice, not part of the method: the sum of
 * squares itself is exact only up to the fp32 roundings of that order, so a
 * row can come out one 16-bit ulp away from the same steps taken on the exact
 * sum rounded once (and its codes one or two steps away).
 */
typedef struct ia_qk_prologue {
  const float* q_norm_weight; /* fp32 [D] RMSNorm weight of Q rows, or NULL (no norm) */
  const float* k_norm_weight; /* fp32 [D] for K rows, or NULL */
  float eps;                  /* RMSNorm epsilon, >= 0 */
  ia_rope_layout rope;
  const float* rope_cos;      /* fp32 [rope_positions][D/2], row stride rope_stride */
  const float* rope_sin;      /* same layout; both 16-byte aligned */
  int64_t rope_stride;        /* elements between positions: >= D/2, a multiple of 4 */
  int rope_positions;         /* rows of the tables; pos0 + S must not exceed it */
  int q_pos0, k_pos0;         /* position of query row 0 and key row 0 */
} ia_qk_prologue;

/* Element type of a general attention mask (ia_attn_params.mask). */
typedef enum ia_mask_dtype {
  IA_MASK_F32 = 0,  /* additive logit offset */
  IA_MASK_BF16 = 1, /* additive logit offset */
  IA_MASK_F16 = 2,  /* additive logit offset */
  IA_MASK_BOOL = 3  /* one byte: nonzero keeps the key, zero excludes it */
} ia_mask_dtype;

/*
 * ia_quantize_qk -- K mean-centring and symmetric INT8 quantisation of Q and K.
 *
 * Defined by: "minimax_h3_sparse_int8" (FastVideo API page), module
 * description and the source of sparse_sm89_attention (per-token scales; K
 * centred by its mean over the sequence, a softmax-invariant shift; the mean is
 * the sum over the sequence divided by the number of valid rows; int8 codes
 * [B,H,S,D] and fp32 scales [B,H,S]); "Feature Request: Direct int8 Q/K
 * passthrough between Comfy Kitchen and SageAttention", sections 2.1 and 3.1
 * (mean_seq + quant_qk_int8; per-block scales); "[attention-int8] Multiple
 * build issues and numerical accuracy problem", maintainer's point 1
 * (symmetric range [-127, 127]).
 *
 * For each row (IA_PER_TOKEN) or 64-row block (IA_PER_BLOCK64) of a head:
 *   x'    = fp32(x - mu)                 (K only, when centring; Q never)
 *   amax  = max |x'|
 *   scale = fp32(amax / 127)             (0 when amax == 0)
 *   code  = round_half_even(fp32(x' * fp32(127 / amax))), clamped to +-127
 * mu[b,h,d] = fp32(fp64(sum_s k[b,h,s,d]) / n_valid): the sum is accumulated
 * with error-free transformations, exact whenever the float64 sum is.
 *
 *   q, k        16-bit inputs of type in_dtype, [B,H,Sq,D] and [B,H,Sk,D],
 *               strides q_strides / k_strides (b,h,s in elements, d contiguous),
 *               16-byte aligned rows. Either may be NULL to skip it.
 *   D           64 or 128.
 *   center_k    nonzero: subtract mu from K (mu from k_mean_in if non-NULL,
 *               else computed). Ignored when k is NULL.
 *   kv_valid    optional int32 [ceil(Sk/64)]: valid rows of each 64-row tile.
 *               Requires Sk % 64 == 0. Rows past it get code 0 and, per
 *               token, scale 0; they are left out of the mean's count and of
 *               block maxima. When Sq == Sk it applies to Q as well.
 *   k_mean_in   optional fp32 [B,H,D] mean to use instead of computing one
 *               (so that separate calls share one centring frame).
 *   q_i8, k_i8  outputs, int8 contiguous [B,H,Sq,D] / [B,H,Sk,D].
 *   q_scale, k_scale  outputs, fp32 contiguous [B,H,Sq] / [B,H,Sk] per token,
 *               [B,H,ceil(S/64)] per block.
 *   k_mean_out  optional fp32 [B,H,D] output of the mean that was used. When
 *               the mean is computed, k_mean_out is given and K holds more
 *               than 64 MiB, the pass runs as two kernels: the K sum
 *               (clusters of CTAs per head, writing the mean here), then the
 *               codes. Otherwise one fused kernel sums and quantises each
 *               head (for a K of at most 64 MiB and a Q at most twice as
 *               long, with Q's codes in the same launch). The results are the
 *               same bits; on a large K the two-kernel form is faster (K no
 *               longer fits in L2 for the fused kernel's second read, and its
 *               code pass is not held at a cluster barrier).
 * Limits (IA_ERR_UNSUPPORTED): H <= 65535 and B <= 65535.
 */
IA_API ia_status ia_quantize_qk(const void* q, const void* k, ia_dtype in_dtype, int B, int H,
                                int Sq, int Sk, int D, const int64_t q_strides[3],
                                const int64_t k_strides[3], ia_granularity granularity,
                                int center_k, const int32_t* kv_valid, const float* k_mean_in,
                                int8_t* q_i8, int8_t* k_i8, float* q_scale, float* k_scale,
                                float* k_mean_out, void* stream);

/*
 * ia_quantize_qk_prologue -- ia_quantize_qk with an RMSNorm + RoPE prologue
 * (ia_qk_prologue) applied to each Q and K row first, fused into the same
 * kernel: the normed, rotated 16-bit rows are never written to memory. The
 * K mean is taken over the prologue's output. Same arguments and outputs as
 * ia_quantize_qk; prologue may be NULL (then it is ia_quantize_qk). Errors:
 * IA_ERR_INVALID_ARG for a negative eps, a rope layout without tables,
 * misaligned tables, rope_stride < D/2 or not a multiple of 4, or positions
 * past rope_positions.
 */
IA_API ia_status ia_quantize_qk_prologue(const void* q, const void* k, ia_dtype in_dtype, int B,
                                         int H, int Sq, int Sk, int D,
                                         const int64_t q_strides[3], const int64_t k_strides[3],
                                         ia_granularity granularity, int center_k,
                                         const int32_t* kv_valid, const float* k_mean_in,
                                         int8_t* q_i8, int8_t* k_i8, float* q_scale,
                                         float* k_scale, float* k_mean_out,
                                         const ia_qk_prologue* prologue, void* stream);

/* Shapes, strides and options of one attention call. */
typedef struct ia_attn_params {
  int B, H, Sq, Sk, D;          /* D is 64 or 128; Sq, Sk >= 0 */
  float sm_scale;               /* softmax scale; NaN selects D^-1/2 */
  ia_granularity granularity;   /* layout of q_scale / k_scale */
  ia_dtype v_dtype;             /* element type of V, of P and of the output */
  int64_t q_strides[3];         /* q_i8 (b,h,s), elements; rows 16-byte aligned */
  int64_t k_strides[3];         /* k_i8 (b,h,s) */
  int64_t qs_strides[2];        /* q_scale (b,h); s or block index contiguous */
  int64_t ks_strides[2];        /* k_scale (b,h) */
  int64_t v_strides[3];         /* v (b,h,s) */
  int64_t o_strides[3];         /* out (b,h,s) */
  int64_t lse_strides[2];       /* lse (b,h); query index contiguous */
  const float* v_scale;         /* optional fp32 [H, D], applied once to the output */
  const int32_t* kv_valid;      /* optional int32 [Sk/64] valid keys per 64-key tile */
  int kv_splits;                /* 0 or 1: one pass over all keys. n >= 2 (at most 16): the
                                   keys are cut into n ranges of whole key tiles (of the
                                   kept-tile list with a block mask); each range is attended
                                   separately into an fp32 partial (O, LSE) in `workspace`,
                                   and the partials are merged exactly, as ia_merge_lse does,
                                   into out and lse. Helps grids that cover the GPU poorly.
                                   Head dim 64, int8 Q, no mask, n == 2 and at least one
                                   256-row query tile per SM: one CTA per SM takes an equal
                                   share of all (query tile, key tile) pairs, so a query
                                   tile's two ranges meet where a CTA's share ends (unequal,
                                   or one range empty); the merge is the same. */
  void* workspace;              /* device scratch of ia_attention_workspace_size(p) bytes,
                                   used only when kv_splits >= 2; owned by the caller */
  size_t workspace_bytes;       /* its size, checked */
  uint64_t wait_timeout_ns;     /* limit of each device-side wait; 0 selects 2 s */
  int debug_stall;              /* test hook: nonzero makes one internal wait of every CTA
                                   wait for a signal that never comes, so the call ends
                                   through the timeout path (status IA_ERR_TIMEOUT) */
  const void* mask;             /* optional general mask, in place of bias_or_null: logically
                                   [B,H,Sq,Sk], element (b,h,i,j) at mask + b*mask_strides[0]
                                   + h*mask_strides[1] + i*mask_strides[2] + j (elements).
                                   Float masks are added to the scaled logits like the bias;
                                   bool masks exclude the keys where they are zero. A zero
                                   stride broadcasts that dimension ("int8_attention: masked
                                   path costs ~1.8x unmasked, ...", The measurement: fp32/bf16/
                                   fp16/bool, [1,1,1,K] and [1,1,Q,K] expanded). */
  ia_mask_dtype mask_dtype;
  int64_t mask_strides[4];      /* (b, h, q, k); k must be 1. q == 0 (one row of keys per b,h,
                                   shared by all queries) takes the per-key path at the cost
                                   of a bias. q != 0 (a row per query) is read by TMA into
                                   shared memory per key tile: base and the b, h, q strides
                                   16-byte aligned; not combinable with a block mask. With
                                   a mask of at most two bytes per key the CTA runs two
                                   128-row stages (~2.3x unmasked, in both entry points);
                                   fp32 masks run one (~3.5x). */
  const ia_qk_prologue* q_prologue; /* ia_attention_fwd_quant_q only: RMSNorm + RoPE of
                                   the Q rows before the in-kernel quantization (its q_*
                                   fields, eps, rope tables); NULL for none */
} ia_attn_params;

/* Fill p with contiguous BHSD strides for the given shape (no pointers set). */
IA_API void ia_attn_params_init(ia_attn_params* p, int B, int H, int Sq, int Sk, int D,
                                ia_granularity granularity, ia_dtype v_dtype);

/*
 * ia_attention_fwd -- forward attention on INT8 Q/K with a 16-bit P.V.
 *
 * Defined by: "minimax_h3_sparse_int8" (FastVideo API page), module
 * description (INT8 QK with per-token scales, FP32 accumulation, PV in BF16,
 * V scale per head and channel applied once in the epilogue, tile-64 key
 * selection with partial key tiles masked) and sparse_sm89_attention (mask
 * [B,H,S/64,S/64], one validity entry per 64-key tile); "int8_attention:
 * masked path costs ~1.8x unmasked, and a request for optional return_lse",
 * opening paragraph (one fp32 additive bias per key, [1,1,1,K], shared by all
 * heads and queries) and Question 2 (LSE so partial calls merge exactly);
 * "Add optional forward LSE output" (FlyDSL), Summary and Public API
 * (LSE = sm_scale*m + ln l, natural log, fp32 [B,H,Sq], -inf for fully masked
 * rows).
 *
 *   s_ij = sm_scale * q_scale_i * k_scale_j * sum_d q_i8[i,d] * k_i8[j,d] + bias_j
 *   s_ij = -inf where block_mask[b,h,i/64,j/64] == 0 or key j is past kv_valid
 *   O_i  = v_scale[h,:] * sum_j softmax_j(s_i.) v_j       (output dtype = v_dtype)
 *   LSE_i = ln sum_j e^{s_ij}; a row with no visible key gives O = 0, LSE = -inf.
 * Query rows past kv_valid (when Sq == Sk) are padding: O = 0, LSE = -inf.
 *
 *   q_i8, k_i8          int8 codes (from ia_quantize_qk or a caller's GEMM epilogue).
 *   q_scale, k_scale    fp32 scales laid out per p->granularity.
 *   v                   [B,H,Sk,D] of p->v_dtype, strides p->v_strides.
 *   bias_or_null        fp32 [Sk], contiguous: broadcast over B, H and queries.
 *   block_mask_or_null  uint8/bool [B,H,ceil(Sq/64),ceil(Sk/64)], contiguous.
 *   out                 [B,H,Sq,D] of p->v_dtype, strides p->o_strides.
 *   lse_or_null         fp32 [B,H,Sq], strides p->lse_strides.
 * A key sub-range [off, off+len) of larger tensors is a view: pass
 * k_i8 + off*k_strides[2], k_scale + off (per token; off/64 per block, off a
 * multiple of 64), v + off*v_strides[2], bias + off, and Sk = len.
 * Alignment: q_i8, k_i8, v and out 16-byte aligned with 16-byte-multiple row,
 * head and batch strides (in bytes).
 * Limits (IA_ERR_UNSUPPORTED): H <= 65535, B * max(kv_splits, 1) <= 65535,
 * Sk <= 65535 * 64; with a block mask the CTA's key-tile list (2 bytes per
 * 64-key tile) must fit in shared memory.
 */
IA_API ia_status ia_attention_fwd(const int8_t* q_i8, const int8_t* k_i8, const float* q_scale,
                                  const float* k_scale, const void* v, const float* bias_or_null,
                                  const uint8_t* block_mask_or_null, void* out,
                                  float* lse_or_null, const ia_attn_params* p, void* stream);

/*
 * ia_attention_fwd_quant_q -- ia_attention_fwd with the Q quantization fused
 * into the attention kernel: Q arrives as 16-bit rows and never makes the
 * round trip through HBM as int8 codes.
 *
 * Defined by: "minimax_h3_sparse_int8" (FastVideo API page), module
 * description and the quant_qk_int8 step (symmetric INT8 codes with one fp32
 * scale per token or per 64-row block, Q not centred); comfy-kitchen issue
 * #101 (int8 Q/K passthrough), the measurements of the quantization stage's
 * share of attention time and the maintainer's point that the 16-bit
 * activations are the interface. Per row i (or 64-row block) of Q:
 *   amax = max |q_i|, scale_i = fl(amax / 127), code = rne(fl(q * fl(127 / amax))),
 *   amax == 0 gives codes 0 and scale 0;
 * bit-identical to ia_quantize_qk on Q followed by ia_attention_fwd, for the
 * same k_i8 / k_scale (quantize K, with its mean, by ia_quantize_qk with q NULL).
 *
 *   q        [B,H,Sq,D] of p->v_dtype (Q and V share the 16-bit type), strides
 *            p->q_strides in elements; 16-byte aligned base and strides.
 *   others   as ia_attention_fwd; p->granularity sets the layout of both the
 *            in-kernel Q scales and k_scale. Query rows past kv_valid (when
 *            Sq == Sk) are padding: they are excluded from their block's amax.
 *
 * When it pays (GB300, whole path of K quantization + attention against
 * ia_quantize_qk + ia_attention_fwd): dense shapes gain the Q pass (anima 4096
 * and 9216 rows, sdxl: 2-7% faster). With a block mask it loses (65536 rows,
 * 80 kept tiles per query tile: about 2% slower): each CTA quantizes its Q rows
 * before any key tile while the block-sparse CTA has few tiles to hide that
 * behind. With the RMSNorm + RoPE prologue in the kernel (p->q_prologue) it is
 * 2-3% slower as well: the prologue's per-row work in the softmax warps costs
 * more than the separate pass it saves. The two paths give identical results;
 * choose by shape.
 */
IA_API ia_status ia_attention_fwd_quant_q(const void* q, const int8_t* k_i8, const float* k_scale,
                                          const void* v, const float* bias_or_null,
                                          const uint8_t* block_mask_or_null, void* out,
                                          float* lse_or_null, const ia_attn_params* p,
                                          void* stream);

/*
 * ia_attention_workspace_size -- bytes of scratch ia_attention_fwd needs for
 * p->kv_splits (0 when kv_splits <= 1): kv_splits * B*H*Sq * (D + 1) * 4.
 */
IA_API size_t ia_attention_workspace_size(const ia_attn_params* p);

/*
 * ia_attention_fwd_static_workspace -- ia_attention_fwd for callers that must
 * not allocate device memory per call. The paper has no counterpart: it is an
 * integration entry point of this library.
 *
 * Who needs it: a caller embedded in a runtime that owns all device memory
 * and hands out no allocator (a plugin inside an inference server, a C
 * program with its own pool), a latency-critical loop that cannot afford
 * cudaMalloc/cudaFree (both may synchronise the device), or a process whose
 * memory budget is fixed at start-up. Such a caller cannot provide the
 * kv_splits >= 2 workspace that ia_attention_fwd asks for.
 *
 * Same arguments, results and errors as ia_attention_fwd, except that
 * p->workspace and p->workspace_bytes are ignored: with kv_splits >= 2 the
 * fp32 partials go to a fixed scratch array inside the library, of
 * IA_STATIC_WORKSPACE_BYTES per device. A call whose
 * ia_attention_workspace_size(p) exceeds that returns IA_ERR_INVALID_ARG
 * before any work. The call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and caches it together
 * with the ID of the current CUDA context; make that first call before any
 * stream capture. A later call in a different context of the device (after
 * cudaDeviceReset, or once the primary context was released and made again)
 * looks the address up again, so the first call in each new context should
 * also come before any capture.
 *
 * Sharing: every call on a device uses the same array, and the array keeps
 * the last call's contents. Nothing in it needs to start at zero: every entry
 * the merge reads is written earlier in the same call. Calls that overlap on
 * the GPU (different streams, or host threads launching concurrently) race on
 * the array and give wrong results; calls on one stream are ordered and safe.
 */
#define IA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20) /* 64 MiB per device */

IA_API ia_status ia_attention_fwd_static_workspace(
    const int8_t* q_i8, const int8_t* k_i8, const float* q_scale, const float* k_scale,
    const void* v, const float* bias_or_null, const uint8_t* block_mask_or_null, void* out,
    float* lse_or_null, const ia_attn_params* p, void* stream);

/*
 * ia_attention_default_splits -- the key split the library suggests for this
 * shape on the current device, from a cost model: the grid runs in rounds of
 * one CTA per SM (two with a block mask), each CTA costs a fixed prologue and
 * epilogue plus its share of the key tiles, and each split adds an fp32
 * partial written and read back by the merge. A split is suggested only when
 * the model expects it to save at least 5%, which happens when the grid
 * covers the SMs poorly (short queries against long keys); with a block mask
 * only when the grid is under one wave. For head dim 64 without a block mask
 * and with at least one 256-row query tile per SM, two ranges are costed as
 * the balanced schedule ia_attention_fwd then runs (see kv_splits). Returns
 * 1..16.
 * block_mask: nonzero if a block mask will be passed.
 */
IA_API int ia_attention_default_splits(const ia_attn_params* p, int block_mask);

/*
 * ia_merge_lse_n -- exact merge of n partial attentions over disjoint key sets
 * (the many-way form of ia_merge_lse; "Add optional forward LSE output",
 * Kernel implementation: the split-K combine reduces all splits, then stores
 * the LSE from the combined maximum and denominator).
 *
 *   M = max_k L_k, w_k = e^{L_k - M}, L = M + ln sum_k w_k,
 *   O = sum_k w_k O_k / sum_k w_k;  M = -inf gives O = 0, L = -inf.
 * o_parts[k]: [B,H,Sq,D] contiguous of `dtype`; lse_parts[k]: fp32 [B,H,Sq]
 * contiguous; the arrays of pointers live in host memory, 1 <= n <= 16.
 * o_out, lse_out: contiguous; lse_out may be NULL; neither may alias an input.
 * 16-byte aligned pointers.
 */
IA_API ia_status ia_merge_lse_n(const void* const* o_parts, const float* const* lse_parts, int n,
                                void* o_out, float* lse_out, int B, int H, int Sq, int D,
                                ia_dtype dtype, void* stream);

/*
 * ia_merge_lse -- exact merge of two partial attentions over disjoint key sets.
 *
 * Defined by: "int8_attention: masked path costs ~1.8x unmasked, ..." Question 2
 * (a core call and a skirt call merged through their log-sum-exps) and "Add
 * optional forward LSE output", Kernel implementation (split-K combine: LSE
 * from the combined maximum and denominator).
 *
 *   M = max(L1, L2), w_k = e^{L_k - M}, L = M + ln(w1 + w2),
 *   O = (w1 O1 + w2 O2) / (w1 + w2);  M = -inf gives O = 0, L = -inf.
 * o1, o2, o_out: [B,H,Sq,D] contiguous of `dtype`; lse1, lse2, lse_out: fp32
 * [B,H,Sq] contiguous. o_out may alias o1 or o2 and lse_out lse1 or lse2.
 * lse_out may be NULL. All pointers 16-byte aligned; D is 64 or 128.
 */
IA_API ia_status ia_merge_lse(const void* o1, const float* lse1, const void* o2,
                              const float* lse2, void* o_out, float* lse_out, int B, int H,
                              int Sq, int D, ia_dtype dtype, void* stream);

/* Static description of a status code. */
IA_API const char* ia_status_string(ia_status s);

/* Status and message of the last failed call on this host thread; IA_OK after a success. */
IA_API ia_status ia_get_last_error(void);
IA_API const char* ia_last_error_message(void);

/*
 * ia_device_status -- synchronise `stream`, then read and clear the device
 * status word the attention kernel writes when a bounded wait runs out.
 * Returns IA_OK, IA_ERR_TIMEOUT, or IA_ERR_CUDA if the synchronisation failed.
 */
IA_API ia_status ia_device_status(void* stream);

/* Library version as "major.minor.patch". */
IA_API const char* ia_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IA_H_ */
