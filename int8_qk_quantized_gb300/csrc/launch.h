// Internal launchers behind the C ABI. Arguments are already validated.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ia.h"

namespace ia {

struct QuantArgs {
  const void* x;           // 16-bit input
  int64_t sb, sh, ss;      // input strides (elements)
  int B, H, S, D;
  int dtype;               // IA_BF16 / IA_FP16
  int gran_block;          // 1: one scale per 64-row block
  int center;              // subtract the mean (K only)
  const int32_t* valid;    // optional per-64-row valid counts
  const float* mean_in;    // optional [B,H,D] mean to use
  float* mean_out;         // optional [B,H,D] mean that was used
  int8_t* codes;           // [B,H,S,D] contiguous
  float* scales;           // [B,H,S] or [B,H,ceil(S/64)] contiguous
  // RMSNorm + RoPE prologue of each row (ia_qk_prologue); off when norm_w is
  // null and rope is IA_ROPE_NONE
  const float* norm_w;     // fp32 [D], 16-byte aligned
  float eps;
  int rope;                // ia_rope_layout
  const float* rcos;       // fp32 [positions][rstride]
  const float* rsin;
  int64_t rstride;
  int pos0;                // position of row 0
};

cudaError_t launch_quantize(const QuantArgs& a, int num_sms, cudaStream_t st);
// Q (no centring) and K together: one launch when K takes the one-pass
// cluster form (centred, no given mean, small enough to stay in L2) and Q is
// at most twice as long as K, else the two launches of launch_quantize, Q first.
cudaError_t launch_quantize_qk(const QuantArgs& aq, const QuantArgs& ak, int num_sms, cudaStream_t st);

struct MergeArgs {
  const void* o1;
  const float* l1;
  const void* o2;
  const float* l2;
  void* o;
  float* l;
  int64_t rows;  // B*H*Sq
  int D;
  int dtype;
};

cudaError_t launch_merge(const MergeArgs& a, int num_sms, cudaStream_t st);

constexpr int kMaxParts = 16;

// n-way merge of partial attentions: part k is o[k] ([B,H,Sq,D] contiguous,
// fp32 when in_f32 else `dtype`) and l[k] (fp32 [B,H,Sq] contiguous).
struct MergeNArgs {
  const void* o[kMaxParts];
  const float* l[kMaxParts];
  int n;
  int in_f32;
  void* out;                 // `dtype`, strides (b,h,s) in elements
  float* lse;                // optional, strides (b,h)
  int B, H, Sq, D;
  int dtype;
  int64_t o_sb, o_sh, o_ss;
  int64_t l_sb, l_sh;
};

cudaError_t launch_merge_n(const MergeNArgs& a, int num_sms, cudaStream_t st);

struct AttnLaunch {
  void* workspace;  // fp32 partials when p.kv_splits >= 2
  const void* q;    // int8 codes, or 16-bit rows of p.v_dtype when q_raw
  int q_raw;        // quantize Q inside the kernel (q_scale unused)
  const int8_t* k;
  const float* q_scale;
  const float* k_scale;
  const void* v;
  const void* bias;        // per-key offsets (fp32 bias, or a general mask with q stride 0)
  int bias_dtype;          // ia_mask_dtype of `bias`
  int64_t bias_sb, bias_sh;  // element strides of its per-(b,h) rows
  int row_mask;            // p.mask varies per query row: read by TMA (p.mask, p.mask_*)
  const uint8_t* mask;     // block mask
  void* out;
  float* lse;
  ia_attn_params p;
  float sm_scale;
};

// Returns IA_OK or an error status; message via the C ABI's error slot.
ia_status launch_attention(const AttnLaunch& a, int num_sms, cudaStream_t st, const char** msg);

// Reads (and clears) the attention kernel's device status word.
cudaError_t attention_read_device_error(unsigned int* out, cudaStream_t st);

}  // namespace ia
