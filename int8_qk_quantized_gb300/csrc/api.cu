// C ABI of libia.so: argument checking, status codes and dispatch to the
// kernel launchers. Nothing here allocates device memory or synchronises
// (except ia_device_status, which exists to synchronise).
#include <cuda.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "launch.h"

namespace {

thread_local ia_status t_last = IA_OK;
thread_local char t_msg[256] = "";

ia_status fail(ia_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ia_status fail(ia_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  t_last = s;
  return s;
}

ia_status ok() {
  t_last = IA_OK;
  t_msg[0] = '\0';
  return IA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device must be sm_103; caches the SM count per device.
ia_status check_device(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static thread_local int cached_dev = -1, cached_sms = 0, cached_ok = 0;
  if (dev != cached_dev) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(IA_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    cached_dev = dev;
    cached_sms = sms;
    cached_ok = (major == 10 && minor == 3) ? 1 : 0;
    if (!cached_ok) {
      cached_dev = -1;
      return fail(IA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                  major, minor);
    }
  }
  *num_sms = cached_sms;
  return IA_OK;
}

bool strides_ok(const int64_t* st, int n, int64_t esize) {
  for (int i = 0; i < n; ++i)
    if (st[i] < 0 || ((st[i] * esize) & 15) != 0) return false;
  return true;
}

// Fixed scratch of ia_attention_fwd_static_workspace: one array per device,
// shared by every call of that entry point on the device.
static __device__ __align__(256) unsigned char g_static_workspace[IA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The array's address belongs to a CUDA context: a context made later on the
// same device (after cudaDeviceReset, or after the primary context was
// released and created again) maps it elsewhere. The looked-up address is
// therefore kept per device together with the ID of the context it was
// looked up in, and looked up again when the current context differs.
struct StaticWorkspaceSlot {
  unsigned long long ctx_id;  // 0: none
  void* ptr;
};
std::mutex g_static_workspace_mu;
StaticWorkspaceSlot g_static_workspace_slot[kMaxDevices];

// ID of the calling thread's current context through the driver's entry
// points (the library links the runtime statically and not libcuda); false
// when there is none yet or the entry points are unavailable.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of g_static_workspace in the current context of the current
// device: looked up with cudaGetSymbolAddress on the first call in a context
// (which also makes the device's primary context current if nothing had),
// then taken from the cache while that context stays current.
ia_status static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(IA_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_static_workspace_mu);
  StaticWorkspaceSlot& slot = g_static_workspace_slot[dev];
  if (have_id && slot.ctx_id == id && slot.ptr != nullptr) {
    *out = slot.ptr;
    return IA_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_static_workspace);
  if (e != cudaSuccess || ptr == nullptr)
    return fail(IA_ERR_CUDA, "cudaGetSymbolAddress(static workspace): %s", cudaGetErrorString(e));
  if (!have_id) have_id = current_context_id(&id);
  slot.ctx_id = have_id ? id : 0ull;  // without an ID the next call looks the address up again
  slot.ptr = ptr;
  *out = ptr;
  return IA_OK;
}

// Checks an RMSNorm + RoPE prologue for rows of width D: Sq / Sk are the
// row counts it will be applied to (0 when absent). for_quantize: the K half
// applies too (ia_quantize_qk_prologue); otherwise only the Q half.
ia_status check_prologue(const ia_qk_prologue* pro, int D, int Sq, int Sk, bool for_quantize) {
  if (pro == nullptr) return IA_OK;
  if (!(pro->eps >= 0.f) || !std::isfinite(pro->eps))
    return fail(IA_ERR_INVALID_ARG, "prologue eps must be finite and >= 0");
  if (!aligned16(pro->q_norm_weight) || (for_quantize && !aligned16(pro->k_norm_weight)))
    return fail(IA_ERR_INVALID_ARG, "norm weights must be 16-byte aligned");
  if (pro->rope != IA_ROPE_NONE) {
    if (pro->rope != IA_ROPE_INTERLEAVED && pro->rope != IA_ROPE_SPLIT_HALF)
      return fail(IA_ERR_INVALID_ARG, "rope layout");
    if (pro->rope_cos == nullptr || pro->rope_sin == nullptr || !aligned16(pro->rope_cos) ||
        !aligned16(pro->rope_sin))
      return fail(IA_ERR_INVALID_ARG, "rope tables must be given and 16-byte aligned");
    if (pro->rope_stride < D / 2 || (pro->rope_stride % 4) != 0)
      return fail(IA_ERR_INVALID_ARG, "rope_stride must be >= D/2 and a multiple of 4");
    if (pro->q_pos0 < 0 || pro->k_pos0 < 0 || pro->rope_positions < 0)
      return fail(IA_ERR_INVALID_ARG, "negative rope position");
    if (static_cast<int64_t>(pro->q_pos0) + Sq > pro->rope_positions ||
        (for_quantize && static_cast<int64_t>(pro->k_pos0) + Sk > pro->rope_positions))
      return fail(IA_ERR_INVALID_ARG, "rows past the rope tables (rope_positions=%d)",
                  pro->rope_positions);
  }
  return IA_OK;
}

void set_prologue(ia::QuantArgs* a, const ia_qk_prologue* pro, bool is_q) {
  if (pro == nullptr) return;
  a->norm_w = is_q ? pro->q_norm_weight : pro->k_norm_weight;
  a->eps = pro->eps;
  a->rope = pro->rope;
  a->rcos = pro->rope_cos;
  a->rsin = pro->rope_sin;
  a->rstride = pro->rope_stride;
  a->pos0 = is_q ? pro->q_pos0 : pro->k_pos0;
}

// Checks and launch shared by ia_attention_fwd (int8 Q codes and their scales)
// and ia_attention_fwd_quant_q (16-bit Q rows of p->v_dtype, quantized inside
// the kernel; q_scale unused).
ia_status attention(const void* q, bool q_raw, const int8_t* k_i8, const float* q_scale,
                    const float* k_scale, const void* v, const float* bias_or_null,
                    const uint8_t* block_mask_or_null, void* out, float* lse_or_null,
                    const ia_attn_params* p, void* stream) {
  if (p == nullptr) return fail(IA_ERR_INVALID_ARG, "params is NULL");
  if (p->B < 0 || p->H < 0 || p->Sq < 0 || p->Sk < 0) return fail(IA_ERR_INVALID_ARG, "negative shape");
  if (p->D != 64 && p->D != 128) return fail(IA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", p->D);
  if (p->v_dtype != IA_BF16 && p->v_dtype != IA_FP16) return fail(IA_ERR_INVALID_ARG, "v_dtype");
  if (p->granularity != IA_PER_TOKEN && p->granularity != IA_PER_BLOCK64)
    return fail(IA_ERR_INVALID_ARG, "granularity");
  if (p->B == 0 || p->H == 0 || p->Sq == 0) return ok();
  if (q == nullptr || k_i8 == nullptr || (!q_raw && q_scale == nullptr) || k_scale == nullptr ||
      v == nullptr || out == nullptr)
    return fail(IA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k_i8) || !aligned16(v) || !aligned16(out))
    return fail(IA_ERR_INVALID_ARG, "q, k_i8, v and out must be 16-byte aligned");
  if (!strides_ok(p->q_strides, 3, q_raw ? 2 : 1) || !strides_ok(p->k_strides, 3, 1) ||
      !strides_ok(p->v_strides, 3, 2) || !strides_ok(p->o_strides, 3, 2))
    return fail(IA_ERR_INVALID_ARG, "row/head/batch strides must be non-negative multiples of 16 bytes");
  if ((p->q_strides[2] < p->D) || (p->k_strides[2] < p->D) || (p->v_strides[2] < p->D) ||
      (p->o_strides[2] < p->D))
    return fail(IA_ERR_INVALID_ARG, "row stride smaller than D");
  if (p->kv_valid != nullptr && (p->Sk % 64) != 0)
    return fail(IA_ERR_INVALID_ARG, "kv_valid requires Sk to be a multiple of 64 (Sk=%d)", p->Sk);
  if (p->Sk > 65535 * 64)
    return fail(IA_ERR_UNSUPPORTED, "Sk too large (%d)", p->Sk);
  // grid: (query tiles, H, B * kv_splits); the last two are at most 65535
  if (p->H > 65535 || static_cast<int64_t>(p->B) * (p->kv_splits > 1 ? p->kv_splits : 1) > 65535)
    return fail(IA_ERR_UNSUPPORTED, "H (%d) and B * kv_splits must be at most 65535", p->H);
  if (p->kv_splits < 0 || p->kv_splits > ia::kMaxParts)
    return fail(IA_ERR_INVALID_ARG, "kv_splits must be in [0, %d] (got %d)", ia::kMaxParts, p->kv_splits);
  if (p->kv_splits > 1) {
    const size_t need = ia_attention_workspace_size(p);
    if (p->workspace == nullptr || p->workspace_bytes < need)
      return fail(IA_ERR_INVALID_ARG, "kv_splits=%d needs a workspace of %zu bytes (got %zu)",
                  p->kv_splits, need, p->workspace == nullptr ? static_cast<size_t>(0) : p->workspace_bytes);
    if (!aligned16(p->workspace)) return fail(IA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  }
  // General mask: its query stride decides between the per-key path (one row
  // of keys per (b, h)) and the per-row path (mask tiles by TMA).
  bool row_mask = false;
  if (p->mask != nullptr) {
    if (bias_or_null != nullptr)
      return fail(IA_ERR_INVALID_ARG, "pass either bias_or_null or params.mask, not both");
    if (p->mask_dtype < IA_MASK_F32 || p->mask_dtype > IA_MASK_BOOL)
      return fail(IA_ERR_INVALID_ARG, "mask_dtype");
    for (int i = 0; i < 4; ++i)
      if (p->mask_strides[i] < 0) return fail(IA_ERR_INVALID_ARG, "negative mask stride");
    if (p->mask_strides[3] != 1 && p->Sk > 1)
      return fail(IA_ERR_INVALID_ARG, "the mask's key stride must be 1");
    row_mask = p->mask_strides[2] != 0 && p->Sq > 1;
    if (row_mask) {
      const int64_t es = p->mask_dtype == IA_MASK_F32 ? 4 : p->mask_dtype == IA_MASK_BOOL ? 1 : 2;
      if (!aligned16(p->mask) || !strides_ok(p->mask_strides, 3, es))
        return fail(IA_ERR_INVALID_ARG,
                    "a per-query-row mask needs a 16-byte aligned base and b, h, q strides");
      if (block_mask_or_null != nullptr)
        return fail(IA_ERR_UNSUPPORTED, "a per-query-row mask cannot be combined with a block mask");
    }
  }
  if (p->q_prologue != nullptr) {
    if (!q_raw)
      return fail(IA_ERR_INVALID_ARG, "params.q_prologue applies to ia_attention_fwd_quant_q only");
    ia_status ps = check_prologue(p->q_prologue, p->D, p->Sq, 0, false);
    if (ps != IA_OK) return ps;
  }
  float sm = p->sm_scale;
  if (std::isnan(sm)) sm = 1.0f / std::sqrt(static_cast<float>(p->D));
  if (!std::isfinite(sm) || sm <= 0.f) return fail(IA_ERR_INVALID_ARG, "sm_scale must be positive");
  int sms = 0;
  ia_status s = check_device(&sms);
  if (s != IA_OK) return s;
  ia::AttnLaunch a{};
  a.q = q;
  a.q_raw = q_raw ? 1 : 0;
  a.k = k_i8;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v = v;
  if (bias_or_null != nullptr) {
    a.bias = bias_or_null;
    a.bias_dtype = IA_MASK_F32;
  } else if (p->mask != nullptr && !row_mask) {
    a.bias = p->mask;
    a.bias_dtype = p->mask_dtype;
    a.bias_sb = p->mask_strides[0];
    a.bias_sh = p->mask_strides[1];
  }
  a.row_mask = row_mask ? 1 : 0;
  a.mask = block_mask_or_null;
  a.out = out;
  a.lse = lse_or_null;
  a.p = *p;
  a.sm_scale = sm;
  a.workspace = p->kv_splits > 1 ? p->workspace : nullptr;
  const char* msg = "";
  s = ia::launch_attention(a, sms, static_cast<cudaStream_t>(stream), &msg);
  if (s != IA_OK) return fail(s, "attention: %s", msg);
  return ok();
}

// Checks and launches of ia_quantize_qk and ia_quantize_qk_prologue.
ia_status quantize(const void* q, const void* k, ia_dtype in_dtype, int B, int H, int Sq, int Sk,
                   int D, const int64_t q_strides[3], const int64_t k_strides[3],
                   ia_granularity granularity, int center_k, const int32_t* kv_valid,
                   const float* k_mean_in, int8_t* q_i8, int8_t* k_i8, float* q_scale,
                   float* k_scale, float* k_mean_out, const ia_qk_prologue* pro, void* stream) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return fail(IA_ERR_INVALID_ARG, "negative shape");
  if (D != 64 && D != 128) return fail(IA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
  if (in_dtype != IA_BF16 && in_dtype != IA_FP16) return fail(IA_ERR_INVALID_ARG, "in_dtype");
  if (granularity != IA_PER_TOKEN && granularity != IA_PER_BLOCK64)
    return fail(IA_ERR_INVALID_ARG, "granularity");
  if (q == nullptr && k == nullptr) return fail(IA_ERR_INVALID_ARG, "q and k are both NULL");
  if (q != nullptr) {
    if (q_i8 == nullptr || q_scale == nullptr || q_strides == nullptr)
      return fail(IA_ERR_INVALID_ARG, "q given without q_i8/q_scale/q_strides");
    if (!aligned16(q) || !strides_ok(q_strides, 3, 2) || !aligned16(q_i8))
      return fail(IA_ERR_INVALID_ARG, "q rows must be 16-byte aligned (base and b,h,s strides)");
  }
  if (k != nullptr) {
    if (k_i8 == nullptr || k_scale == nullptr || k_strides == nullptr)
      return fail(IA_ERR_INVALID_ARG, "k given without k_i8/k_scale/k_strides");
    if (!aligned16(k) || !strides_ok(k_strides, 3, 2) || !aligned16(k_i8))
      return fail(IA_ERR_INVALID_ARG, "k rows must be 16-byte aligned (base and b,h,s strides)");
  }
  if (kv_valid != nullptr && (Sk % 64) != 0)
    return fail(IA_ERR_INVALID_ARG, "kv_valid requires Sk to be a multiple of 64 (Sk=%d)", Sk);
  if (H > 65535 || B > 65535)  // grid (chunks, H, B)
    return fail(IA_ERR_UNSUPPORTED, "H (%d) and B (%d) must be at most 65535", H, B);
  ia_status ps = check_prologue(pro, D, q != nullptr ? Sq : 0, k != nullptr ? Sk : 0, true);
  if (ps != IA_OK) return ps;
  int sms = 0;
  ia_status s = check_device(&sms);
  if (s != IA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ia::QuantArgs aq{}, ak{};
  if (q != nullptr) {
    ia::QuantArgs& a = aq;
    a.x = q;
    a.sb = q_strides[0];
    a.sh = q_strides[1];
    a.ss = q_strides[2];
    a.B = B;
    a.H = H;
    a.S = Sq;
    a.D = D;
    a.dtype = in_dtype;
    a.gran_block = granularity == IA_PER_BLOCK64;
    a.center = 0;
    a.valid = (kv_valid != nullptr && Sq == Sk) ? kv_valid : nullptr;
    a.codes = q_i8;
    a.scales = q_scale;
    set_prologue(&a, pro, true);
  }
  if (k != nullptr) {
    ia::QuantArgs& a = ak;
    a.x = k;
    a.sb = k_strides[0];
    a.sh = k_strides[1];
    a.ss = k_strides[2];
    a.B = B;
    a.H = H;
    a.S = Sk;
    a.D = D;
    a.dtype = in_dtype;
    a.gran_block = granularity == IA_PER_BLOCK64;
    a.center = center_k ? 1 : 0;
    a.valid = kv_valid;
    a.mean_in = center_k ? k_mean_in : nullptr;
    a.mean_out = center_k ? k_mean_out : nullptr;
    a.codes = k_i8;
    a.scales = k_scale;
    set_prologue(&a, pro, false);
  }
  cudaError_t e = cudaSuccess;
  if (q != nullptr && k != nullptr) e = ia::launch_quantize_qk(aq, ak, sms, st);
  else e = ia::launch_quantize(q != nullptr ? aq : ak, sms, st);
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "quantize: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

IA_API const char* ia_status_string(ia_status s) {
  switch (s) {
    case IA_OK: return "ok";
    case IA_ERR_INVALID_ARG: return "invalid argument";
    case IA_ERR_UNSUPPORTED: return "unsupported";
    case IA_ERR_CUDA: return "CUDA error";
    case IA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

IA_API ia_status ia_get_last_error(void) { return t_last; }
IA_API const char* ia_last_error_message(void) { return t_msg; }
IA_API const char* ia_version(void) { return "0.1.0"; }

IA_API void ia_attn_params_init(ia_attn_params* p, int B, int H, int Sq, int Sk, int D,
                                ia_granularity granularity, ia_dtype v_dtype) {
  if (p == nullptr) return;
  std::memset(p, 0, sizeof(*p));
  p->B = B;
  p->H = H;
  p->Sq = Sq;
  p->Sk = Sk;
  p->D = D;
  p->sm_scale = NAN;
  p->granularity = granularity;
  p->v_dtype = v_dtype;
  const int64_t hd = static_cast<int64_t>(D);
  p->q_strides[0] = static_cast<int64_t>(H) * Sq * hd;
  p->q_strides[1] = static_cast<int64_t>(Sq) * hd;
  p->q_strides[2] = hd;
  p->k_strides[0] = static_cast<int64_t>(H) * Sk * hd;
  p->k_strides[1] = static_cast<int64_t>(Sk) * hd;
  p->k_strides[2] = hd;
  const int64_t nq = granularity == IA_PER_BLOCK64 ? (Sq + 63) / 64 : Sq;
  const int64_t nk = granularity == IA_PER_BLOCK64 ? (Sk + 63) / 64 : Sk;
  p->qs_strides[0] = static_cast<int64_t>(H) * nq;
  p->qs_strides[1] = nq;
  p->ks_strides[0] = static_cast<int64_t>(H) * nk;
  p->ks_strides[1] = nk;
  for (int i = 0; i < 3; ++i) p->v_strides[i] = p->k_strides[i];
  for (int i = 0; i < 3; ++i) p->o_strides[i] = p->q_strides[i];
  p->lse_strides[0] = static_cast<int64_t>(H) * Sq;
  p->lse_strides[1] = Sq;
}

IA_API ia_status ia_quantize_qk(const void* q, const void* k, ia_dtype in_dtype, int B, int H,
                                int Sq, int Sk, int D, const int64_t q_strides[3],
                                const int64_t k_strides[3], ia_granularity granularity,
                                int center_k, const int32_t* kv_valid, const float* k_mean_in,
                                int8_t* q_i8, int8_t* k_i8, float* q_scale, float* k_scale,
                                float* k_mean_out, void* stream) {
  return quantize(q, k, in_dtype, B, H, Sq, Sk, D, q_strides, k_strides, granularity, center_k,
                  kv_valid, k_mean_in, q_i8, k_i8, q_scale, k_scale, k_mean_out, nullptr, stream);
}

IA_API ia_status ia_quantize_qk_prologue(const void* q, const void* k, ia_dtype in_dtype, int B,
                                         int H, int Sq, int Sk, int D,
                                         const int64_t q_strides[3], const int64_t k_strides[3],
                                         ia_granularity granularity, int center_k,
                                         const int32_t* kv_valid, const float* k_mean_in,
                                         int8_t* q_i8, int8_t* k_i8, float* q_scale,
                                         float* k_scale, float* k_mean_out,
                                         const ia_qk_prologue* prologue, void* stream) {
  return quantize(q, k, in_dtype, B, H, Sq, Sk, D, q_strides, k_strides, granularity, center_k,
                  kv_valid, k_mean_in, q_i8, k_i8, q_scale, k_scale, k_mean_out, prologue, stream);
}

IA_API ia_status ia_attention_fwd(const int8_t* q_i8, const int8_t* k_i8, const float* q_scale,
                                  const float* k_scale, const void* v, const float* bias_or_null,
                                  const uint8_t* block_mask_or_null, void* out,
                                  float* lse_or_null, const ia_attn_params* p, void* stream) {
  return attention(q_i8, false, k_i8, q_scale, k_scale, v, bias_or_null, block_mask_or_null, out,
                   lse_or_null, p, stream);
}

IA_API ia_status ia_attention_fwd_quant_q(const void* q, const int8_t* k_i8, const float* k_scale,
                                          const void* v, const float* bias_or_null,
                                          const uint8_t* block_mask_or_null, void* out,
                                          float* lse_or_null, const ia_attn_params* p,
                                          void* stream) {
  return attention(q, true, k_i8, nullptr, k_scale, v, bias_or_null, block_mask_or_null, out,
                   lse_or_null, p, stream);
}

IA_API ia_status ia_attention_fwd_static_workspace(
    const int8_t* q_i8, const int8_t* k_i8, const float* q_scale, const float* k_scale,
    const void* v, const float* bias_or_null, const uint8_t* block_mask_or_null, void* out,
    float* lse_or_null, const ia_attn_params* p, void* stream) {
  if (p == nullptr) return fail(IA_ERR_INVALID_ARG, "params is NULL");
  ia_attn_params q = *p;
  q.workspace = nullptr;
  q.workspace_bytes = 0;
  if (q.kv_splits > 1) {
    const size_t need = ia_attention_workspace_size(&q);
    if (need > IA_STATIC_WORKSPACE_BYTES)
      return fail(IA_ERR_INVALID_ARG,
                  "kv_splits=%d needs %zu bytes of scratch; the fixed workspace holds %zu "
                  "(use fewer splits, or ia_attention_fwd with a caller workspace)",
                  q.kv_splits, need, static_cast<size_t>(IA_STATIC_WORKSPACE_BYTES));
  }
  void* ws = nullptr;
  ia_status s = static_workspace(&ws);
  if (s != IA_OK) return s;
  if (q.kv_splits > 1) {
    q.workspace = ws;
    q.workspace_bytes = IA_STATIC_WORKSPACE_BYTES;
  }
  return ia_attention_fwd(q_i8, k_i8, q_scale, k_scale, v, bias_or_null, block_mask_or_null, out,
                          lse_or_null, &q, stream);
}

IA_API size_t ia_attention_workspace_size(const ia_attn_params* p) {
  if (p == nullptr || p->kv_splits <= 1 || p->B <= 0 || p->H <= 0 || p->Sq <= 0) return 0;
  return static_cast<size_t>(p->kv_splits) * static_cast<size_t>(p->B) * p->H * p->Sq *
         (static_cast<size_t>(p->D) + 1) * sizeof(float);
}

IA_API int ia_attention_default_splits(const ia_attn_params* p, int block_mask) {
  if (p == nullptr || p->B <= 0 || p->H <= 0 || p->Sq <= 0 || p->Sk <= 0) return 1;
  int sms = 0;
  if (check_device(&sms) != IA_OK) return 1;
  // one dense CTA (256 query rows) per SM; two block-sparse CTAs (128 rows)
  const int64_t rows_per_cta = block_mask ? 128 : 256;
  const int64_t slots = static_cast<int64_t>(sms) * (block_mask ? 2 : 1);
  const int64_t ctas = (static_cast<int64_t>(p->Sq) + rows_per_cta - 1) / rows_per_cta * p->H * p->B;
  // With a block mask the kept tiles per CTA are unknown here and uneven; a
  // grid of a wave or more balances itself.
  if (block_mask && ctas >= slots) return 1;
  // Cost model in units of one CTA's key-tile iteration: a CTA costs a fixed
  // prologue/epilogue (kFixed tiles) plus its share of the key tiles; the
  // grid runs in ceil(ctas*n / slots) rounds; each split adds the write and
  // the merge read of an fp32 partial (B*H*Sq*(D+1)*8 bytes), converted at
  // kBytesPerTile bytes of HBM traffic per tile time.
  constexpr int64_t kFixed = 4;
  constexpr double kBytesPerTile = 14.0e6;
  const int64_t tile = block_mask ? 64 : 128;
  const int64_t tiles = (p->Sk + tile - 1) / tile;
  const double merge_per_split =
      static_cast<double>(p->B) * p->H * p->Sq * (p->D + 1) * 8.0 / kBytesPerTile;
  int64_t best = 1;
  double best_cost = 0.0;
  for (int64_t n = 1; n <= ia::kMaxParts && n <= tiles; ++n) {
    const int64_t rounds = (ctas * n + slots - 1) / slots;
    double cost = static_cast<double>(rounds) * (kFixed + (tiles + n - 1) / n);
    if (n > 1) cost += merge_per_split * static_cast<double>(n);
    if (n == 1 || cost < best_cost * (best == 1 ? 0.95 : 1.0)) {
      best = n;
      best_cost = cost;
    }
  }
  // Dense head dim 64 with at least one query tile per SM: two ranges run as
  // balanced segments (one CTA per SM takes an equal share of the (query
  // tile, key tile) units, in up to three segments, each with its fixed cost).
  if (!block_mask && p->D == 64 && ctas >= slots) {
    const double seg = static_cast<double>(ctas) * tiles / slots + 2.0 * kFixed + merge_per_split * 2.0;
    if (seg < best_cost) best = 2;
  }
  const int64_t n = best;
  return n < 2 ? 1 : static_cast<int>(n);
}

IA_API ia_status ia_merge_lse_n(const void* const* o_parts, const float* const* lse_parts, int n,
                                void* o_out, float* lse_out, int B, int H, int Sq, int D,
                                ia_dtype dtype, void* stream) {
  if (B < 0 || H < 0 || Sq < 0) return fail(IA_ERR_INVALID_ARG, "negative shape");
  if (D != 64 && D != 128) return fail(IA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
  if (dtype != IA_BF16 && dtype != IA_FP16) return fail(IA_ERR_INVALID_ARG, "dtype");
  if (n < 1 || n > ia::kMaxParts) return fail(IA_ERR_INVALID_ARG, "n must be in [1, %d]", ia::kMaxParts);
  if (static_cast<int64_t>(B) * H * Sq == 0) return ok();
  if (o_parts == nullptr || lse_parts == nullptr || o_out == nullptr)
    return fail(IA_ERR_INVALID_ARG, "a required pointer is NULL");
  for (int k = 0; k < n; ++k) {
    if (o_parts[k] == nullptr || lse_parts[k] == nullptr)
      return fail(IA_ERR_INVALID_ARG, "partial %d is NULL", k);
    if (!aligned16(o_parts[k])) return fail(IA_ERR_INVALID_ARG, "partial %d is not 16-byte aligned", k);
  }
  if (!aligned16(o_out)) return fail(IA_ERR_INVALID_ARG, "o_out must be 16-byte aligned");
  int sms = 0;
  ia_status s = check_device(&sms);
  if (s != IA_OK) return s;
  ia::MergeNArgs a{};
  for (int k = 0; k < n; ++k) {
    a.o[k] = o_parts[k];
    a.l[k] = lse_parts[k];
  }
  a.n = n;
  a.in_f32 = 0;
  a.out = o_out;
  a.lse = lse_out;
  a.B = B;
  a.H = H;
  a.Sq = Sq;
  a.D = D;
  a.dtype = dtype;
  a.o_sb = static_cast<int64_t>(H) * Sq * D;
  a.o_sh = static_cast<int64_t>(Sq) * D;
  a.o_ss = D;
  a.l_sb = static_cast<int64_t>(H) * Sq;
  a.l_sh = Sq;
  cudaError_t e = ia::launch_merge_n(a, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "merge_n: %s", cudaGetErrorString(e));
  return ok();
}

IA_API ia_status ia_merge_lse(const void* o1, const float* lse1, const void* o2,
                              const float* lse2, void* o_out, float* lse_out, int B, int H,
                              int Sq, int D, ia_dtype dtype, void* stream) {
  if (B < 0 || H < 0 || Sq < 0) return fail(IA_ERR_INVALID_ARG, "negative shape");
  if (D != 64 && D != 128) return fail(IA_ERR_INVALID_ARG, "D must be 64 or 128 (got %d)", D);
  if (dtype != IA_BF16 && dtype != IA_FP16) return fail(IA_ERR_INVALID_ARG, "dtype");
  if (static_cast<int64_t>(B) * H * Sq == 0) return ok();
  if (o1 == nullptr || o2 == nullptr || lse1 == nullptr || lse2 == nullptr || o_out == nullptr)
    return fail(IA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(o1) || !aligned16(o2) || !aligned16(o_out))
    return fail(IA_ERR_INVALID_ARG, "outputs and inputs must be 16-byte aligned");
  int sms = 0;
  ia_status s = check_device(&sms);
  if (s != IA_OK) return s;
  ia::MergeArgs a{};
  a.o1 = o1;
  a.l1 = lse1;
  a.o2 = o2;
  a.l2 = lse2;
  a.o = o_out;
  a.l = lse_out;
  a.rows = static_cast<int64_t>(B) * H * Sq;
  a.D = D;
  a.dtype = dtype;
  cudaError_t e = ia::launch_merge(a, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "merge: %s", cudaGetErrorString(e));
  return ok();
}

IA_API ia_status ia_device_status(void* stream) {
  unsigned int w = 0;
  cudaError_t e = ia::attention_read_device_error(&w, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(IA_ERR_CUDA, "device status: %s", cudaGetErrorString(e));
  if (w != 0) return fail(IA_ERR_TIMEOUT, "attention kernel status word 0x%x", w);
  return ok();
}

}  // extern "C"
