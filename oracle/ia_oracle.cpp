// Plain, slow CPU oracle of INT8-QK quantised attention. TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline legs load
// this library (through oracle/ia_oracle.py). It shares no code, header,
// table or helper with the CUDA library, and neither uses the other.
//
// Arithmetic: float64 for attention, the softmax and the merge; float32 with
// IEEE rounding (no contraction: built with -ffp-contract=off) for the
// quantiser's decisions and the RMSNorm + RoPE prologue; exact sums where a
// step is defined as a sum (the K mean, the RMSNorm sum of squares).
//
// Sources (page title, then the part of the page):
//  [FastVideo]   "minimax_h3_sparse_int8" (FastVideo API page): the module
//                description (per-token Q/K scales, K centred by its mean as a
//                softmax-invariant shift, one V scale per head and channel
//                applied once at the end, BF16 PV with FP32 accumulation,
//                tile-64 keys with partial key tiles masked) and the source of
//                sparse_sm89_attention (mean = sum over the sequence / number
//                of valid rows; codes int8 [B,H,S,D], scales fp32 [B,H,S];
//                mask [B,H,S/64,S/64]; validity vector per 64-row tile).
//  [Passthrough] "Feature Request: Direct int8 Q/K passthrough between Comfy
//                Kitchen and SageAttention": 2.1 (mean_seq, quant_qk_int8, int8
//                QK with a 16-bit PV), 3.1 (per-block scales), the
//                maintainer's reply (RMSNorm + RoPE on the 16-bit rows).
//  [model-kernels] "[attention-int8] Multiple build issues and numerical
//                accuracy problem": maintainer's point 1 (symmetric [-127, 127]).
//  [comfy-kitchen] "int8_attention: masked path costs ~1.8x unmasked, and a
//                request for optional return_lse": opening paragraph (one
//                additive bias per key), "The measurement" (mask forms),
//                "Question 2" (merging two partial softmaxes through LSEs).
//  [FlyDSL]      "Add optional forward LSE output": Summary (LSE = sm_scale*m +
//                ln l, natural log), Kernel implementation (-inf for fully
//                masked rows; split-K combine).
//
// Every function is pinned by tests/test_oracle_*.py against closed forms,
// brute force, library routines or invariants; none is "parity unpinned".
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kTile = 64;
constexpr double kNegInf = -std::numeric_limits<double>::infinity();

// ------------------------------------------------------------------ threads
int thread_count(int requested) {
  if (requested > 0) return requested;
  const unsigned hc = std::thread::hardware_concurrency();
  return hc == 0 ? 1 : static_cast<int>(hc);
}

// Runs fn(i) for i in [0, n) on `threads` threads; tasks are independent.
void parallel_for(int64_t n, int threads, const std::function<void(int64_t)>& fn) {
  threads = static_cast<int>(std::min<int64_t>(std::max(threads, 1), std::max<int64_t>(n, 1)));
  if (threads <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&] {
      for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
    });
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------- exact sum
// The exact sum of finite doubles, kept as a fixed-point integer in units of
// 2^-1074 (the smallest double), with positive and negative terms in two
// accumulators of 32-bit digits held in 64-bit words (carries are settled at
// the end). `rounded(p, qmin)` rounds the exact value once, to nearest with
// ties to even, to p significant bits with no bit below 2^qmin: (53, -1074)
// is binary64, (24, -149) binary32.
struct ExactSum {
  static constexpr int kDigits = 68;  // 2176 bits: 2^-1074 .. 2^1024, plus 2^78 terms of growth
  uint64_t pos[kDigits];
  uint64_t neg[kDigits];
  double nonfinite = 0.0;  // running IEEE sum of inf / nan terms
  bool any_nonfinite = false;

  ExactSum() { clear(); }
  void clear() {
    std::memset(pos, 0, sizeof(pos));
    std::memset(neg, 0, sizeof(neg));
    nonfinite = 0.0;
    any_nonfinite = false;
  }

  void add(double x) {
    if (x == 0.0) return;
    if (!std::isfinite(x)) {
      nonfinite += x;
      any_nonfinite = true;
      return;
    }
    int e = 0;
    const double f = std::frexp(std::fabs(x), &e);     // |x| = f * 2^e, f in [0.5, 1)
    uint64_t m = static_cast<uint64_t>(std::ldexp(f, 53));  // |x| = m * 2^(e - 53), exactly
    int sh = e - 53 + 1074;
    if (sh < 0) {  // a subnormal: m carries -sh zero bits at the bottom
      m >>= -sh;
      sh = 0;
    }
    uint64_t* acc = x > 0 ? pos : neg;
    const int d = sh >> 5;
    const unsigned __int128 v = static_cast<unsigned __int128>(m) << (sh & 31);
    acc[d] += static_cast<uint64_t>(v & 0xffffffffu);
    acc[d + 1] += static_cast<uint64_t>((v >> 32) & 0xffffffffu);
    acc[d + 2] += static_cast<uint64_t>(v >> 64);
  }

  static void settle(const uint64_t* in, uint32_t* out) {
    uint64_t carry = 0;
    for (int i = 0; i < kDigits; ++i) {
      const uint64_t t = in[i] + carry;
      out[i] = static_cast<uint32_t>(t & 0xffffffffu);
      carry = t >> 32;
    }
  }

  static int cmp(const uint32_t* a, const uint32_t* b) {
    for (int i = kDigits - 1; i >= 0; --i)
      if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
    return 0;
  }

  static bool bit(const uint32_t* a, int64_t i) {
    return i >= 0 && ((a[i >> 5] >> (i & 31)) & 1u) != 0;
  }

  double rounded(int p, int qmin) const {
    if (any_nonfinite) return nonfinite;
    uint32_t a[kDigits], b[kDigits], d[kDigits];
    settle(pos, a);
    settle(neg, b);
    const int c = cmp(a, b);
    if (c == 0) return 0.0;
    const uint32_t* hi = c > 0 ? a : b;
    const uint32_t* lo = c > 0 ? b : a;
    int64_t borrow = 0;
    for (int i = 0; i < kDigits; ++i) {
      int64_t t = static_cast<int64_t>(hi[i]) - lo[i] - borrow;
      borrow = t < 0 ? 1 : 0;
      if (t < 0) t += (int64_t{1} << 32);
      d[i] = static_cast<uint32_t>(t);
    }
    int64_t top = -1;  // index of the highest set bit of |sum|
    for (int i = kDigits - 1; i >= 0 && top < 0; --i)
      if (d[i] != 0) top = int64_t{i} * 32 + 31 - __builtin_clz(d[i]);
    const int64_t low = std::max<int64_t>(top - p + 1, qmin + 1074);  // lowest bit kept
    uint64_t r = 0;
    for (int64_t i = top; i >= std::max<int64_t>(low, 0); --i) r = (r << 1) | (bit(d, i) ? 1u : 0u);
    if (low > 0) {
      const bool guard = bit(d, low - 1);
      bool sticky = false;
      for (int64_t i = low - 2; i >= 0 && !sticky; --i) sticky = bit(d, i);
      if (guard && (sticky || (r & 1u))) ++r;
    }
    const double mag = std::ldexp(static_cast<double>(r), static_cast<int>(std::max<int64_t>(low, 0) - 1074));
    return c > 0 ? mag : -mag;
  }
};

// ---------------------------------------------------------------- validity
// Row s of a sequence with a validity vector is data iff s % 64 < vbs[s / 64]
// ([FastVideo] sparse_sm89_attention: valid rows per 64-row tile).
inline bool row_valid(const int32_t* vbs, int64_t s) {
  return vbs == nullptr || (s % kTile) < vbs[s / kTile];
}

// --------------------------------------------------------- 16-bit rounding
// float32 -> bf16 -> float32, round to nearest even: add half of the dropped
// 16 bits (plus the kept lsb, for ties to even) and truncate; NaN stays NaN.
float round_bf16(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) {
    u |= 0x00400000u;
  } else {
    u += 0x7fffu + ((u >> 16) & 1u);
  }
  u &= 0xffff0000u;
  float y;
  std::memcpy(&y, &u, 4);
  return y;
}

// float32 -> IEEE binary16 -> float32, round to nearest even (the compiler's
// _Float16 conversion, an IEEE conversion operation).
float round_fp16(float x) { return static_cast<float>(static_cast<_Float16>(x)); }

}  // namespace

extern "C" {

// The K mean ([FastVideo] sparse_sm89_attention; [Passthrough] 2.1 mean_seq):
// mu[b,h,d] = (sum over the valid rows s of k[b,h,s,d]) / n_valid. Reading:
// the page sums in fp32 in an unspecified order; here the sum is exact,
// rounded once to float64, divided by n in float64 and rounded once to
// float32. k: float32 [B,H,S,D] holding exact 16-bit values; mu: [B,H,D].
void or_k_mean(const float* k, int B, int H, int S, int D, const int32_t* kv_valid, float* mu,
               int threads) {
  int64_t n = 0;
  for (int64_t s = 0; s < S; ++s) n += row_valid(kv_valid, s) ? 1 : 0;
  parallel_for(int64_t{B} * H, thread_count(threads), [&](int64_t bh) {
    std::vector<ExactSum> acc(static_cast<size_t>(D));
    const float* base = k + bh * S * D;
    for (int64_t s = 0; s < S; ++s) {
      if (!row_valid(kv_valid, s)) continue;
      for (int d = 0; d < D; ++d) acc[d].add(static_cast<double>(base[s * D + d]));
    }
    for (int d = 0; d < D; ++d) {
      const double total = acc[d].rounded(53, -1074);
      mu[bh * D + d] = static_cast<float>(total / static_cast<double>(std::max<int64_t>(n, 1)));
    }
  });
}

// Symmetric INT8 quantisation of Q or K, per row (granularity 0) or per
// 64-row block (1). Steps, for each row or block:
//   x' = fp32(x - mu) when mu is given (K only; [FastVideo] K centring);
//   amax = max |x'| over the row or block (exact);
//   scale = fp32(amax / 127); inv = fp32(127 / amax);
//   code = round-half-even(fp32(x' * inv)), clamped to [-127, 127]
//   ([model-kernels] point 1: symmetric range; [FastVideo] per-token scales;
//   [Passthrough] 3.1 per-block scales).
// amax == 0 gives codes 0 and scale 0. Rows past the validity vector are not
// data: codes 0, they do not enter a block's amax, a per-row scale is 0.
// Reading: the pages fix neither the rounding mode nor divide versus
// reciprocal; this uses ties-to-even on the product with fp32(127 / amax).
// x: float32 [B,H,S,D]; mu: [B,H,D] or null; codes: [B,H,S,D];
// scales: [B,H,S] or [B,H,ceil(S/64)].
void or_quantize(const float* x, int B, int H, int S, int D, const float* mu, int granularity,
                 const int32_t* kv_valid, int8_t* codes, float* scales, int threads) {
  const int64_t nb = (S + kTile - 1) / kTile;
  parallel_for(int64_t{B} * H, thread_count(threads), [&](int64_t bh) {
    const float* xb = x + bh * S * D;
    const float* m = mu == nullptr ? nullptr : mu + bh * D;
    std::vector<float> xc(static_cast<size_t>(S) * D);
    for (int64_t s = 0; s < S; ++s) {
      const bool ok = row_valid(kv_valid, s);
      for (int d = 0; d < D; ++d) {
        const float v = m == nullptr ? xb[s * D + d] : xb[s * D + d] - m[d];
        xc[s * D + d] = ok ? v : 0.0f;
      }
    }
    auto amax_of = [&](int64_t s0, int64_t s1) {
      float a = 0.0f;
      for (int64_t s = s0; s < s1; ++s)
        for (int d = 0; d < D; ++d) a = std::max(a, std::fabs(xc[s * D + d]));
      return a;
    };
    auto encode = [&](int64_t s0, int64_t s1, float amax) {
      const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
      for (int64_t s = s0; s < s1; ++s)
        for (int d = 0; d < D; ++d) {
          float c = 0.0f;
          if (amax > 0.0f) {
            const float prod = xc[s * D + d] * inv;
            c = std::min(127.0f, std::max(-127.0f, std::nearbyint(prod)));
          }
          codes[bh * S * D + s * D + d] = static_cast<int8_t>(c);
        }
      return amax > 0.0f ? amax / 127.0f : 0.0f;
    };
    if (granularity == 0) {
      for (int64_t s = 0; s < S; ++s) scales[bh * S + s] = encode(s, s + 1, amax_of(s, s + 1));
    } else {
      for (int64_t t = 0; t < nb; ++t) {
        const int64_t s0 = t * kTile, s1 = std::min<int64_t>(S, s0 + kTile);
        scales[bh * nb + t] = encode(s0, s1, amax_of(s0, s1));
      }
    }
  });
}

// RMSNorm then rotary embedding of each row, rounded to the 16-bit type: the
// activations the unfused path hands to attention ([Passthrough],
// maintainer's reply: rms_rope / apply_rope / rms_rope_split_half run on the
// 16-bit rows; the page gives names, not formulas). Reading, per row x:
//  1. RMSNorm (norm_w given): ss = the exact sum of x_d^2, rounded once to
//     fp32; ms = fp32(ss / D); r = fp32(1 / fp32(sqrt(fp32(ms + eps))));
//     y_d = fp32(fp32(x_d * r) * w_d).
//  2. RoPE (rope 1 = interleaved pairs (2i, 2i+1), 2 = split-half pairs
//     (i, i + D/2)); with c = cos[p, i], s = sin[p, i] at the row's position
//     p = pos0 + row: a' = fp32(fp32(a c) - fp32(b s)), b' = fp32(fp32(a s) +
//     fp32(b c)), the rotation of (a, b) by the tabulated angle.
//  3. one rounding to the 16-bit type (dtype 0 = bf16, 1 = fp16).
// x, y: float32 [B,H,S,D]; cos, sin: float32 [P, D/2].
void or_qk_prologue(const float* x, int B, int H, int S, int D, int dtype, const float* norm_w,
                    float eps, int rope, const float* cos_t, const float* sin_t, int pos0,
                    float* y, int threads) {
  const int half = D / 2;
  parallel_for(int64_t{B} * H * S, thread_count(threads), [&](int64_t row) {
    const int64_t s = row % S;
    const float* xr = x + row * D;
    float* yr = y + row * D;
    std::vector<float> t(xr, xr + D);
    if (norm_w != nullptr) {
      ExactSum ss;
      for (int d = 0; d < D; ++d) ss.add(static_cast<double>(t[d]) * static_cast<double>(t[d]));
      const float ssf = static_cast<float>(ss.rounded(24, -149));
      const float ms = ssf / static_cast<float>(D);
      const float r = 1.0f / std::sqrt(ms + eps);
      for (int d = 0; d < D; ++d) t[d] = (t[d] * r) * norm_w[d];
    }
    if (rope == 1 || rope == 2) {
      const float* c = cos_t + (pos0 + s) * half;
      const float* sn = sin_t + (pos0 + s) * half;
      for (int i = 0; i < half; ++i) {
        const int ia = rope == 1 ? 2 * i : i;
        const int ib = rope == 1 ? 2 * i + 1 : i + half;
        const float a = t[ia], b = t[ib];
        const float ac = a * c[i], bs = b * sn[i], as = a * sn[i], bc = b * c[i];
        t[ia] = ac - bs;
        t[ib] = as + bc;
      }
    }
    for (int d = 0; d < D; ++d) yr[d] = dtype == 0 ? round_bf16(t[d]) : round_fp16(t[d]);
  });
}

// Softmax attention in float64 over the rows `rows` of every (b, h):
//   q_kind / k_kind 0: q_hat = code * scale and k_hat likewise (the
//     same-quantisation reference; [Passthrough] 2.1 int8 QK);
//   kinds 1 / 2 (float32 / float64 values): q, k as given (textbook attention
//     on the unquantised inputs, the yardstick of [model-kernels] section 5);
//   s_ij = sm_scale * <q_hat_i, k_hat_j> + bias_j + mask_ij, or -inf where the
//     tile-64 block mask drops key tile j/64 for query tile i/64, key row j
//     lies past the validity vector, or a bool mask is false;
//   O_i = v_scale (*) sum_j softmax_j(s_i.) v_j; LSE_i = m_i + ln sum_j
//     e^(s_ij - m_i) ([FastVideo] module description; [comfy-kitchen] bias;
//     [FlyDSL] Summary: natural log, softmax scale included).
// A row whose logits are all -inf gives O = 0 and LSE = -inf ([FlyDSL]
// Kernel implementation). With pad_query, query rows past the validity
// vector give O = 0 and LSE = -inf (the pages leave them undefined).
// Reading: the bias and the mask are added after the softmax scale, as
// SDPA's additive attn_mask, which [comfy-kitchen] compares against.
// mask_kind: 0 none, 1 additive float64, 2 bool (uint8, keep where nonzero),
// read at mask[b*ms0 + h*ms1 + i*ms2 + j*ms3] (a zero stride broadcasts).
// Layouts: q/k int8 codes, float32 or float64 [B,H,S,D]; scales fp32 [B,H,S]
// or [B,H,ceil(S/64)] (granularity 1); v float32 or float64 (v_kind 1 / 2)
// [B,H,Sk,D]; bias float64 [Sk];
// block_mask uint8 [B,H,ceil(Sq/64),ceil(Sk/64)]; v_scale float64 [H,D];
// out float64 [B,H,n_rows,D]; lse float64 [B,H,n_rows].
void or_attention(int B, int H, int Sq, int Sk, int D, const void* q, int q_kind,
                  const float* q_scale, const void* k, int k_kind, const float* k_scale,
                  int granularity, const void* v, int v_kind, double sm_scale,
                  const double* bias, const void* mask,
                  int mask_kind, const int64_t* mask_strides, const uint8_t* block_mask,
                  const int32_t* kv_valid, const double* v_scale, int pad_query,
                  const int64_t* rows, int64_t n_rows, double* out, double* lse, int threads) {
  const int64_t Tq = (Sq + kTile - 1) / kTile, Tk = (Sk + kTile - 1) / kTile;
  const int64_t nsq = granularity == 1 ? Tq : Sq, nsk = granularity == 1 ? Tk : Sk;
  const int nthreads = thread_count(threads);
  // element `at` of an operand as float64: an int8 code times its row's (or
  // block's) scale (kind 0), or a float32 (1) or float64 (2) value
  auto value = [&](const void* a, int kind, const float* sc, int64_t ns, int64_t bh, int64_t row,
                   int64_t at) -> double {
    if (kind == 0)
      return static_cast<double>(static_cast<const int8_t*>(a)[at]) *
             static_cast<double>(sc[bh * ns + (granularity == 1 ? row / kTile : row)]);
    if (kind == 1) return static_cast<double>(static_cast<const float*>(a)[at]);
    return static_cast<const double*>(a)[at];
  };
  for (int64_t bh = 0; bh < int64_t{B} * H; ++bh) {
    const int64_t b = bh / H, h = bh % H;
    // this head's keys and values in float64
    std::vector<double> kh(static_cast<size_t>(Sk) * D), vh(static_cast<size_t>(Sk) * D);
    parallel_for(Sk, nthreads, [&](int64_t j) {
      for (int d = 0; d < D; ++d) {
        const int64_t at = (bh * Sk + j) * D + d;
        kh[j * D + d] = value(k, k_kind, k_scale, nsk, bh, j, at);
        vh[j * D + d] = value(v, v_kind, nullptr, 0, bh, j, at);
      }
    });
    parallel_for(n_rows, nthreads, [&](int64_t ri) {
      const int64_t i = rows[ri];
      double* o = out + (bh * n_rows + ri) * D;
      double* l_out = lse + bh * n_rows + ri;
      std::vector<double> qh(static_cast<size_t>(D)), s(static_cast<size_t>(Sk)), acc(static_cast<size_t>(D), 0.0);
      for (int d = 0; d < D; ++d) qh[d] = value(q, q_kind, q_scale, nsq, bh, i, (bh * Sq + i) * D + d);
      double m = kNegInf;
      for (int64_t j = 0; j < Sk; ++j) {
        bool vis = row_valid(kv_valid, j);
        if (block_mask != nullptr)
          vis = vis && block_mask[((bh * Tq) + i / kTile) * Tk + j / kTile] != 0;
        double sj = kNegInf;
        if (vis) {
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += qh[d] * kh[j * D + d];
          sj = sm_scale * dot;
          if (bias != nullptr) sj += bias[j];
          if (mask_kind != 0) {
            const int64_t at = b * mask_strides[0] + h * mask_strides[1] + i * mask_strides[2] +
                               j * mask_strides[3];
            if (mask_kind == 1) sj += static_cast<const double*>(mask)[at];
            else if (static_cast<const uint8_t*>(mask)[at] == 0) sj = kNegInf;
          }
        }
        s[j] = sj;
        m = std::max(m, sj);
      }
      const bool pad = pad_query && kv_valid != nullptr && !row_valid(kv_valid, i);
      if (m == kNegInf || pad) {  // fully masked (or padding) row
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *l_out = kNegInf;
        return;
      }
      double l = 0.0;
      for (int64_t j = 0; j < Sk; ++j) {
        if (s[j] == kNegInf) continue;
        const double p = std::exp(s[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) acc[d] += p * vh[j * D + d];
      }
      for (int d = 0; d < D; ++d) {
        double od = acc[d] / l;
        if (v_scale != nullptr) od *= v_scale[h * D + d];
        o[d] = od;
      }
      *l_out = m + std::log(l);
    });
  }
}

// Exact merge of two partial softmax attentions over disjoint key sets
// ([comfy-kitchen] Question 2; [FlyDSL] Kernel implementation, split-K
// combine): M = max(L1, L2); w_k = e^(L_k - M) (0 for an empty partial);
// L = M + ln(w1 + w2); O = (w1 O1 + w2 O2) / (w1 + w2); both empty gives
// O = 0, L = -inf. float64, n rows of D.
void or_merge(const double* o1, const double* l1, const double* o2, const double* l2, int64_t n,
              int D, double* o, double* l) {
  for (int64_t r = 0; r < n; ++r) {
    const double m = std::max(l1[r], l2[r]);
    if (m == kNegInf) {
      for (int d = 0; d < D; ++d) o[r * D + d] = 0.0;
      l[r] = kNegInf;
      continue;
    }
    const double w1 = l1[r] == kNegInf ? 0.0 : std::exp(l1[r] - m);
    const double w2 = l2[r] == kNegInf ? 0.0 : std::exp(l2[r] - m);
    const double den = w1 + w2;
    for (int d = 0; d < D; ++d) o[r * D + d] = (w1 * o1[r * D + d] + w2 * o2[r * D + d]) / den;
    l[r] = m + std::log(den);
  }
}

// The exact sum of n doubles rounded once to p bits (53 or 24): exposed so
// that the tests can pin the summation on its own.
double or_exact_sum(const double* x, int64_t n, int p) {
  ExactSum acc;
  for (int64_t i = 0; i < n; ++i) acc.add(x[i]);
  return p == 24 ? acc.rounded(24, -149) : acc.rounded(53, -1074);
}

int or_hardware_threads(void) { return thread_count(0); }

}  // extern "C"
