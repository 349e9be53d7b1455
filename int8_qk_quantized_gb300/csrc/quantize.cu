// K mean and symmetric INT8 quantisation of Q and K.
//
// "minimax_h3_sparse_int8" (FastVideo API page): per-token scales, K centred by
// its mean over the sequence (sum divided by the number of valid rows), codes
// int8 [B,H,S,D], scales fp32 [B,H,S]. "Feature Request: Direct int8 Q/K
// passthrough between Comfy Kitchen and SageAttention", 3.1: per-block
// scales. "[attention-int8] Multiple build issues and numerical accuracy
// problem", maintainer's point 1: symmetric range [-127, 127].
//
// One kernel handles a head's rows in chunks. For K with centring, the CTAs
// of one head form a thread-block cluster: each CTA sums its chunk's columns
// with error-free two-sum transformations in FP32 (a hi/lo pair per column,
// exact whenever the float64 sum is), the partials are combined in FP64 in a
// fixed order through distributed shared memory, and every CTA of the cluster
// then quantises its own chunk with the same mean. No scratch memory is used.
// The quantiser itself uses correctly rounded FP32 division, multiplication
// and round-half-even, so codes and scales are reproducible bit for bit.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace ia {
namespace {

constexpr int kThreads = 512;
constexpr int kTile = 64;
// Largest centred K (bytes) that takes the one-pass cluster form: all heads are
// read at once, and the code pass finds its chunk still in L2.
constexpr int64_t kOnePassMaxBytes = int64_t{64} << 20;

template <int DT>
__device__ __forceinline__ void unpack8(const uint4 w, float (&v)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == IA_BF16) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
      const float2 f = __half22float2(h);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
}

template <int DT>
__device__ __forceinline__ void load8(const void* p, float (&v)[8]) {
  unpack8<DT>(__ldg(reinterpret_cast<const uint4*>(p)), v);
}

__device__ __forceinline__ bool row_valid(const int32_t* valid, int r) {
  return valid == nullptr || (r % kTile) < __ldg(valid + r / kTile);
}

// Error-free accumulation of two columns at once: (hi, lo) += x lane by lane,
// with hi + lo exact whenever it fits (Knuth's two-sum in packed f32x2 form).
__device__ __forceinline__ void two_sum_acc2(uint64_t& hi, uint64_t& lo, uint64_t x) {
  const uint64_t s = fadd2(hi, x);
  const uint64_t bp = fsub2(s, hi);
  const uint64_t err = fadd2(fsub2(hi, fsub2(s, bp)), fsub2(x, bp));
  hi = s;
  lo = fadd2(lo, err);
}

// code = round-half-even(fl(x * inv)) for 8 values, stored as 8 int8. Adding
// 1.5 * 2^23 to the rounded fp32 product leaves no fraction bits, so the IEEE
// addition rounds it to the nearest integer (ties to even, 1.5 * 2^23 being
// even) and the low byte of the sum's bit pattern is the code in two's
// complement. The multiply and the add are the scalar IEEE intrinsics, which
// are never contracted into a fused multiply-add: a fused form would round
// x * inv + 1.5 * 2^23 once and break exact ties such as 63.5 (the packed
// f32x2 forms were contracted). No clamp is needed: |x| <= amax gives
// x * fl(127 / amax) <= 127 (1 + 2^-24), which rounds to at most 127 + 2^-17
// and then to the integer 127.
__device__ __forceinline__ void store_codes(int8_t* dst, const float (&x)[8], float inv) {
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = __float_as_uint(__fadd_rn(__fmul_rn(x[i], inv), 12582912.0f));
  const uint32_t w0 = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  const uint32_t w1 = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
  *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
}

template <int DT>
__device__ __forceinline__ float round16(float x) {
  if constexpr (DT == IA_BF16) return __bfloat162float(__float2bfloat16_rn(x));
  else return __half2float(__float2half_rn(x));
}

// RMSNorm + RoPE prologue ("Feature Request: Direct int8 Q/K passthrough
// between Comfy Kitchen and SageAttention", maintainer's reply: rms_rope,
// apply_rope, rms_rope_split_half run on the 16-bit rows before attention)
// on this thread's 8 values of row rr; the row's TPR threads are adjacent
// lanes of one warp and every lane of the warp calls this.
//   ss = sum of squares in a fixed fp32 order: this thread's 8 squares in
//        index order, then the TPR partial sums added pairwise, t with
//        t + n/2 (a butterfly of symmetric adds: every lane ends with the
//        same value),
//   r = 1 / sqrt(ss / D + eps), y = (x * r) * w   (IEEE fp32 steps),
//   pair (a, b) with cos c and sin s of position pos0 + rr:
//        a' = a c - b s, b' = a s + b c,
// then one rounding to the 16-bit type. Rows that are not data (ok false)
// come out as 0 and read no table entry.
template <int D, int DT>
__device__ __forceinline__ void prologue8(float (&v)[8], bool ok, int rr, int tc,
                                          const QuantArgs& a) {
  constexpr int TPR = D / 8;
  if (a.norm_w != nullptr) {
    float ss = __fmul_rn(v[0], v[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(v[i], v[i]));
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    const float r = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), a.eps)));
    const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.norm_w + tc * 8));
    const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.norm_w + tc * 8 + 4));
    const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), w[i]);
  }
  if (a.rope == IA_ROPE_INTERLEAVED) {
    float c[4] = {1.f, 1.f, 1.f, 1.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      const int64_t o = static_cast<int64_t>(a.pos0 + rr) * a.rstride + tc * 4;
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.rcos + o));
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(a.rsin + o));
      c[0] = c4.x, c[1] = c4.y, c[2] = c4.z, c[3] = c4.w;
      sn[0] = s4.x, sn[1] = s4.y, sn[2] = s4.z, sn[3] = s4.w;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x0 = v[2 * j], x1 = v[2 * j + 1];
      v[2 * j] = __fsub_rn(__fmul_rn(x0, c[j]), __fmul_rn(x1, sn[j]));
      v[2 * j + 1] = __fadd_rn(__fmul_rn(x0, sn[j]), __fmul_rn(x1, c[j]));
    }
  } else if (a.rope == IA_ROPE_SPLIT_HALF) {
    float pv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pv[i] = __shfl_xor_sync(0xffffffffu, v[i], TPR / 2);
    const bool first = tc < TPR / 2;  // holds the a of its pairs, the partner the b
    float c[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = 1.f, sn[i] = 0.f;
    if (ok) {
      const int64_t o = static_cast<int64_t>(a.pos0 + rr) * a.rstride + (tc % (TPR / 2)) * 8;
      const float4 c0 = __ldg(reinterpret_cast<const float4*>(a.rcos + o));
      const float4 c1 = __ldg(reinterpret_cast<const float4*>(a.rcos + o + 4));
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(a.rsin + o));
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(a.rsin + o + 4));
      c[0] = c0.x, c[1] = c0.y, c[2] = c0.z, c[3] = c0.w, c[4] = c1.x, c[5] = c1.y, c[6] = c1.z, c[7] = c1.w;
      sn[0] = s0.x, sn[1] = s0.y, sn[2] = s0.z, sn[3] = s0.w, sn[4] = s1.x, sn[5] = s1.y, sn[6] = s1.z, sn[7] = s1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x0 = first ? v[i] : pv[i], x1 = first ? pv[i] : v[i];
      v[i] = first ? __fsub_rn(__fmul_rn(x0, c[i]), __fmul_rn(x1, sn[i]))
                   : __fadd_rn(__fmul_rn(x0, sn[i]), __fmul_rn(x1, c[i]));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ok ? round16<DT>(v[i]) : 0.f;
}

// Per-token codes and scales of rows [r_lo, r_hi) of one head, the mean (if
// centring) in s_mu (16-byte aligned shared memory), walked from the last
// row. Four adjacent lanes own a row: lane t of the four loads the row's
// 16-byte chunks t, t+4, t+8, ... (the four read 64 contiguous bytes per
// load), so a warp covers 8 rows, the row maximum takes two shuffles and one
// pair of IEEE divisions serves 8 rows per warp. The raw 16-bit chunks stay
// in registers; the centred values are formed twice (for the maximum, then
// for the codes) with the same IEEE subtraction.
template <int D, int DT, int NT>
__device__ __forceinline__ void lean_codes(const QuantArgs& a, const char* xb, int8_t* cb, float* sc,
                                           int r_lo, int r_hi, const float* s_mu, int tid) {
  constexpr int CPT = D / 32;  // 16-byte chunks per lane
  constexpr int RPP = NT / 4;  // rows per pass
  const int g = tid >> 2, tc = tid & 3;
  // the trip count is uniform over the block: every lane reaches the shuffles
  for (int base = r_hi - RPP; base > r_lo - RPP; base -= RPP) {
    const int rr = base + g;
    const bool in = rr >= r_lo && rr < r_hi;
    const bool ok = in && row_valid(a.valid, rr);
    uint4 w[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j)
      w[j] = ok ? __ldg(reinterpret_cast<const uint4*>(xb + (static_cast<int64_t>(rr) * a.ss + (tc + 4 * j) * 8) * 2))
                : make_uint4(0u, 0u, 0u, 0u);
    auto centred = [&](int j, float (&v)[8]) {
      unpack8<DT>(w[j], v);
      if (a.center && ok) {
        const float4 m0 = *reinterpret_cast<const float4*>(s_mu + (tc + 4 * j) * 8);
        const float4 m1 = *reinterpret_cast<const float4*>(s_mu + (tc + 4 * j) * 8 + 4);
        unpack2(fsub2(pack2(v[0], v[1]), pack2(m0.x, m0.y)), v[0], v[1]);
        unpack2(fsub2(pack2(v[2], v[3]), pack2(m0.z, m0.w)), v[2], v[3]);
        unpack2(fsub2(pack2(v[4], v[5]), pack2(m1.x, m1.y)), v[4], v[5]);
        unpack2(fsub2(pack2(v[6], v[7]), pack2(m1.z, m1.w)), v[6], v[7]);
      }
    };
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      float v[8];
      centred(j, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) m = fmax3(m, fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    if (!in) continue;
    const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      float v[8];
      centred(j, v);
      store_codes(cb + static_cast<int64_t>(rr) * D + (tc + 4 * j) * 8, v, inv);
    }
    if (tc == 0) sc[rr] = (ok && m > 0.f) ? __fdiv_rn(m, 127.f) : 0.f;
  }
}

// Shared memory of one quantize CTA.
template <int D, bool CLUSTER_MEAN>
struct QuantSmem {
  static constexpr int RPP = kThreads / (D / 8);
  __align__(16) float mu[D];
  double red[CLUSTER_MEAN ? RPP : 1][CLUSTER_MEAN ? D : 1];
  double part[CLUSTER_MEAN ? D : 1];
  float wmax[kThreads / 32];
  int count;
};

// Chunk cx of head (b, h): rows [cx*chunk, min(S, (cx+1)*chunk)). With
// CLUSTER_MEAN and a.center the chunks of the head are one cluster (cx its
// rank) and compute the mean; MEAN_ONLY then stops once the mean is written to
// a.mean_out (codes_kernel writes the codes in a second pass).
template <int D, int DT, bool CLUSTER_MEAN, bool PRO, bool MEAN_ONLY>
__device__ __forceinline__ void quantize_chunk(const QuantArgs& a, int chunk, int b, int h, int cx,
                                               QuantSmem<D, CLUSTER_MEAN>& sm) {
  constexpr int TPR = D / 8;            // threads per row, 8 elements each
  constexpr int RPP = kThreads / TPR;   // rows per pass
  static_assert(RPP * TPR == kThreads, "layout");
  float* s_mu = sm.mu;
  auto& s_red = sm.red;
  double* s_part = sm.part;
  float* s_wmax = sm.wmax;
  int& s_count = sm.count;

  const int tid = threadIdx.x;
  const int tr = tid / TPR;
  const int tc = tid % TPR;
  const int r0 = cx * chunk;
  const int r1 = min(a.S, r0 + chunk);
  const char* xb = static_cast<const char*>(a.x) + (static_cast<int64_t>(b) * a.sb +
                                                    static_cast<int64_t>(h) * a.sh) * 2;
  const int64_t bh = static_cast<int64_t>(b) * a.H + h;

  // ---------------------------------------------------------------- mean
  if (a.center) {
    if (CLUSTER_MEAN) {
      uint64_t hi[4], lo[4];  // column pairs (2i, 2i+1)
#pragma unroll
      for (int i = 0; i < 4; ++i) hi[i] = lo[i] = pack2(0.f, 0.f);
      // 8 rows of 16-byte loads in flight per thread, kept packed until used
      constexpr int U1 = PRO ? 4 : 6;  // within 64 registers (the prologue needs its own)
      for (int base = r0; base < r1; base += U1 * RPP) {
        uint4 w[U1];
#pragma unroll
        for (int u = 0; u < U1; ++u) {
          const int rr = base + u * RPP + tr;
          w[u] = (rr < r1 && row_valid(a.valid, rr))
                     ? __ldg(reinterpret_cast<const uint4*>(xb + (static_cast<int64_t>(rr) * a.ss + tc * 8) * 2))
                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U1; ++u) {
          float v[8];
          unpack8<DT>(w[u], v);
          if constexpr (PRO) {
            const int rr = base + u * RPP + tr;
            prologue8<D, DT>(v, rr < r1 && row_valid(a.valid, rr), rr, tc, a);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) two_sum_acc2(hi[i], lo[i], pack2(v[2 * i], v[2 * i + 1]));
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float h0, h1, l0, l1;
        unpack2(hi[i], h0, h1);
        unpack2(lo[i], l0, l1);
        s_red[tr][tc * 8 + 2 * i] = static_cast<double>(h0) + static_cast<double>(l0);
        s_red[tr][tc * 8 + 2 * i + 1] = static_cast<double>(h1) + static_cast<double>(l1);
      }
      if (tid == 0) {
        int n = a.S;
        if (a.valid) {
          n = 0;
          for (int t = 0; t < a.S / kTile; ++t) n += __ldg(a.valid + t);
        }
        s_count = n;
      }
      __syncthreads();
      if (tid < D) {
        double s = 0.0;
        for (int j = 0; j < RPP; ++j) s += s_red[j][tid];
        s_part[tid] = s;
      }
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();
      if (tid < D) {
        double tot = 0.0;
        const int nr = static_cast<int>(cluster.num_blocks());
        // the partials in rank order; eight remote loads in flight at a time
        for (int r0 = 0; r0 < nr; r0 += 8) {
          double pv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) pv[j] = r0 + j < nr ? *cluster.map_shared_rank(&s_part[tid], r0 + j) : 0.0;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (r0 + j < nr) tot += pv[j];
        }
        const int n = s_count > 0 ? s_count : 1;
        s_mu[tid] = static_cast<float>(tot / static_cast<double>(n));
        if (a.mean_out && cluster.block_rank() == 0) a.mean_out[bh * D + tid] = s_mu[tid];
      }
      cluster.sync();  // no CTA leaves while another still reads its partials
      if constexpr (MEAN_ONLY) return;
    } else {
      if (tid < D) {
        s_mu[tid] = __ldg(a.mean_in + bh * D + tid);
        if (a.mean_out && cx == 0) a.mean_out[bh * D + tid] = s_mu[tid];
      }
      __syncthreads();
    }
  }
  float mu[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mu[i] = a.center ? s_mu[tc * 8 + i] : 0.f;

  int8_t* cb = a.codes + bh * static_cast<int64_t>(a.S) * D;
  // ------------------------------------------------------ per-token codes
  if (!PRO && !a.gran_block) {
    lean_codes<D, DT, kThreads>(a, xb, cb, a.scales + bh * a.S, r0, r1, s_mu, tid);
    return;
  }
  if (!a.gran_block) {
    float* sc = a.scales + bh * a.S;
    // The loop bound is uniform across the CTA: every lane reaches the shuffles.
    // The chunk is walked from its end, so rows the mean pass read last are
    // read again first, while they may still sit in L2.
    constexpr int U2 = PRO ? 4 : 8;  // rows of 16-byte loads in flight per thread
    const int nbase = (r1 - r0 + U2 * RPP - 1) / (U2 * RPP);
    for (int ib = nbase - 1; ib >= 0; --ib) {
      const int base = r0 + ib * U2 * RPP;
      uint4 w[U2];
      bool ok[U2];
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const int rr = base + u * RPP + tr;
        ok[u] = rr < r1 && row_valid(a.valid, rr);
        w[u] = ok[u] ? __ldg(reinterpret_cast<const uint4*>(xb + (static_cast<int64_t>(rr) * a.ss + tc * 8) * 2))
                     : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const int rr = base + u * RPP + tr;
        float v[8];
        unpack8<DT>(w[u], v);
        if constexpr (PRO) prologue8<D, DT>(v, ok[u], rr, tc, a);
        if (a.center && ok[u]) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            unpack2(fsub2(pack2(v[2 * i], v[2 * i + 1]), pack2(mu[2 * i], mu[2 * i + 1])), v[2 * i],
                    v[2 * i + 1]);
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) m = fmax3(m, fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1)
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (rr < r1) {
          const float scale = m > 0.f ? __fdiv_rn(m, 127.f) : 0.f;
          const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
          store_codes(cb + static_cast<int64_t>(rr) * D + tc * 8, v, inv);
          if (tc == 0) sc[rr] = ok[u] ? scale : 0.f;
        }
      }
    }
    return;
  }
  // ---------------------------------------------------- per-64-block codes
  constexpr int PPB = kTile / RPP;  // passes per block
  float* sc = a.scales + bh * ((a.S + kTile - 1) / kTile);
  for (int blk0 = r0; blk0 < r1; blk0 += kTile) {
    float v[PPB][8];
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < PPB; ++p) {
      const int rr = blk0 + p * RPP + tr;
      if (rr < r1 && row_valid(a.valid, rr)) {
        load8<DT>(xb + (static_cast<int64_t>(rr) * a.ss + tc * 8) * 2, v[p]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[p][i] = 0.f;
      }
      if constexpr (PRO) prologue8<D, DT>(v[p], rr < r1 && row_valid(a.valid, rr), rr, tc, a);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (a.center && rr < r1 && row_valid(a.valid, rr)) v[p][i] = __fsub_rn(v[p][i], mu[i]);
        m = fmaxf(m, fabsf(v[p][i]));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) s_wmax[tid / 32] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) m = fmaxf(m, s_wmax[w]);
    __syncthreads();
    const float scale = m > 0.f ? __fdiv_rn(m, 127.f) : 0.f;
    const float inv = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;
#pragma unroll
    for (int p = 0; p < PPB; ++p) {
      const int rr = blk0 + p * RPP + tr;
      if (rr < r1) store_codes(cb + static_cast<int64_t>(rr) * D + tc * 8, v[p], inv);
    }
    if (tid == 0) sc[blk0 / kTile] = scale;
  }
}

// grid: (chunks, H, B); with CLUSTER_MEAN the chunks of a head are one cluster.
template <int D, int DT, bool CLUSTER_MEAN, bool PRO, bool MEAN_ONLY = false>
__global__ void __launch_bounds__(kThreads, 2) quantize_kernel(const QuantArgs a, int chunk) {
  __shared__ QuantSmem<D, CLUSTER_MEAN> sm;
  quantize_chunk<D, DT, CLUSTER_MEAN, PRO, MEAN_ONLY>(a, chunk, blockIdx.z, blockIdx.y, blockIdx.x, sm);
}

// Q and a centred K in one launch (a K small enough for the one-pass form):
// grid (chunks, H, 2B) in clusters of `chunks` CTAs along x; z < B are K's
// heads (cluster mean, then codes), z >= B are Q's (codes only, chunk_q rows
// per CTA; the cluster is not used).
template <int D, int DT, bool PRO>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_qk_kernel(const QuantArgs aq, const QuantArgs ak, int chunk_q, int chunk_k) {
  __shared__ QuantSmem<D, true> sm;
  const int z = blockIdx.z;
  if (z < ak.B)
    quantize_chunk<D, DT, true, PRO, false>(ak, chunk_k, z, blockIdx.y, blockIdx.x, sm);
  else
    quantize_chunk<D, DT, true, PRO, false>(aq, chunk_q, z - ak.B, blockIdx.y, blockIdx.x, sm);
}

// Per-token codes without the prologue, the mean (if any) read from
// a.mean_in. grid: (ceil(S / rows), H, B); block x covers rows
// [S - (x+1) rows, S - x rows) clamped at 0, so the first blocks take the
// head's last rows.
constexpr int kCodeThreads = 256;
constexpr int kCodeRows = 512;  // rows per block: 8 passes of 64
template <int D, int DT>
__global__ void __launch_bounds__(kCodeThreads) codes_kernel(const QuantArgs a) {
  __shared__ __align__(16) float s_mu[D];
  const int tid = threadIdx.x;
  const int b = blockIdx.z, h = blockIdx.y;
  const int r_hi = a.S - blockIdx.x * kCodeRows;
  const int r_lo = max(0, r_hi - kCodeRows);
  const int64_t bh = static_cast<int64_t>(b) * a.H + h;
  const char* xb = static_cast<const char*>(a.x) + (static_cast<int64_t>(b) * a.sb +
                                                    static_cast<int64_t>(h) * a.sh) * 2;
  if (tid < D) s_mu[tid] = a.center ? __ldg(a.mean_in + bh * D + tid) : 0.f;
  __syncthreads();
  lean_codes<D, DT, kCodeThreads>(a, xb, a.codes + bh * static_cast<int64_t>(a.S) * D, a.scales + bh * a.S,
                                  r_lo, r_hi, s_mu, tid);
}

// Codes and scales with the mean (if any) already known (a.mean_in).
template <int D, int DT, bool PRO>
cudaError_t launch_codes(const QuantArgs& a, cudaStream_t st) {
  if (!PRO && !a.gran_block) {
    if (a.center && a.mean_out != nullptr && a.mean_out != a.mean_in) {  // the mean that was used
      const cudaError_t e = cudaMemcpyAsync(a.mean_out, a.mean_in, static_cast<size_t>(a.B) * a.H * D * sizeof(float),
                                            cudaMemcpyDeviceToDevice, st);
      if (e != cudaSuccess) return e;
    }
    dim3 grid((a.S + kCodeRows - 1) / kCodeRows, a.H, a.B);
    codes_kernel<D, DT><<<grid, kCodeThreads, 0, st>>>(a);
    return cudaGetLastError();
  }
  // Rows split into chunks of 256 (a multiple of 64); no cluster.
  const int chunk = 256;
  dim3 grid((a.S + chunk - 1) / chunk, a.H, a.B);
  quantize_kernel<D, DT, false, PRO><<<grid, kThreads, 0, st>>>(a, chunk);
  return cudaGetLastError();
}

template <int D, int DT, bool PRO>
cudaError_t launch_typed(const QuantArgs& a, int num_sms, cudaStream_t st) {
  const int BH = a.B * a.H;
  if (a.center && a.mean_in == nullptr) {
    // One cluster per head, sized so that the grid fills two CTAs per SM in
    // one wave where the heads allow (up to the largest cluster the device
    // can place; 16 needs the non-portable cluster size attribute).
    // A K above kOnePassMaxBytes (about half of L2) is not there any more when
    // the fused pass reads it the second time: then, with somewhere to put the mean, two
    // passes (the clusters only sum K and write the mean, the code kernel
    // reads it), which keeps the code pass off the cluster barrier. A
    // smaller K stays in L2 and one fused pass saves a launch.
    const bool two_pass = a.mean_out != nullptr &&
                          static_cast<int64_t>(BH) * a.S * D * 2 > kOnePassMaxBytes;
    auto fused = quantize_kernel<D, DT, true, PRO, false>;
    auto mean_only = quantize_kernel<D, DT, true, PRO, true>;
    auto kern = two_pass ? mean_only : fused;
    static int max_cl = 0;  // the two kernels have the same resources
    if (max_cl == 0) {
      max_cl = 8;
      if (cudaFuncSetAttribute(fused, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
          cudaFuncSetAttribute(mean_only, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(16, 1, 1);
        q.blockDim = dim3(kThreads);
        int n = 0;
        if (cudaOccupancyMaxPotentialClusterSize(&n, kern, &q) == cudaSuccess && n >= 8)
          max_cl = n > 16 ? 16 : n;
      }
      cudaGetLastError();
    }
    int cl = (2 * num_sms) / BH;
    cl = cl < 1 ? 1 : (cl > max_cl ? max_cl : cl);
    const int max_chunks = (a.S + kTile - 1) / kTile;
    if (cl > max_chunks) cl = max_chunks;
    int chunk = (a.S + cl - 1) / cl;
    chunk = (chunk + kTile - 1) / kTile * kTile;
    cl = (a.S + chunk - 1) / chunk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl, a.H, a.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, chunk);
    if (e != cudaSuccess || !two_pass) return e;
    QuantArgs c = a;
    c.mean_in = a.mean_out;
    c.mean_out = nullptr;
    return launch_codes<D, DT, PRO>(c, st);
  }
  return launch_codes<D, DT, PRO>(a, st);
}

// Q and K in one launch: K's clusters as in the one-pass form, sized so that the
// two halves of the grid together fill two CTAs per SM in one wave where the
// heads allow; Q's CTAs take the same number of chunks per head.
template <int D, int DT, bool PRO>
cudaError_t launch_qk_typed(const QuantArgs& aq, const QuantArgs& ak, int num_sms, cudaStream_t st) {
  auto kern = quantize_qk_kernel<D, DT, PRO>;
  static int max_cl = 0;
  if (max_cl == 0) {
    max_cl = 8;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(16, 1, 1);
      q.blockDim = dim3(kThreads);
      int n = 0;
      if (cudaOccupancyMaxPotentialClusterSize(&n, kern, &q) == cudaSuccess && n >= 8)
        max_cl = n > 16 ? 16 : n;
    }
    cudaGetLastError();
  }
  const int BH = ak.B * ak.H;
  int cl = num_sms / BH;
  cl = cl < 1 ? 1 : (cl > max_cl ? max_cl : cl);
  const int max_chunks = (ak.S + kTile - 1) / kTile;
  if (cl > max_chunks) cl = max_chunks;
  int chunk_k = (ak.S + cl - 1) / cl;
  chunk_k = (chunk_k + kTile - 1) / kTile * kTile;
  cl = (ak.S + chunk_k - 1) / chunk_k;
  int chunk_q = (aq.S + cl - 1) / cl;
  chunk_q = (chunk_q + kTile - 1) / kTile * kTile;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl, ak.H, 2 * ak.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, aq, ak, chunk_q, chunk_k);
}

bool has_prologue(const QuantArgs& a) { return a.norm_w != nullptr || a.rope != IA_ROPE_NONE; }

}  // namespace

cudaError_t launch_quantize_qk(const QuantArgs& aq, const QuantArgs& ak, int num_sms, cudaStream_t st) {
  // (Q's CTAs take as many chunks per head as K's cluster: a Q much longer
  // than K is better served by its own code kernel)
  const bool one = ak.center && ak.mean_in == nullptr && has_prologue(aq) == has_prologue(ak) &&
                   aq.S > 0 && ak.S > 0 && aq.S <= 2 * static_cast<int64_t>(ak.S) && ak.B > 0 && ak.H > 0 &&
                   2 * static_cast<int64_t>(ak.B) <= 65535 &&
                   static_cast<int64_t>(ak.B) * ak.H * ak.S * ak.D * 2 <= kOnePassMaxBytes;
  if (!one) {
    const cudaError_t e = launch_quantize(aq, num_sms, st);
    return e != cudaSuccess ? e : launch_quantize(ak, num_sms, st);
  }
  const bool pro = has_prologue(ak);
  if (ak.D == 128) {
    if (pro)
      return ak.dtype == IA_BF16 ? launch_qk_typed<128, IA_BF16, true>(aq, ak, num_sms, st)
                                 : launch_qk_typed<128, IA_FP16, true>(aq, ak, num_sms, st);
    return ak.dtype == IA_BF16 ? launch_qk_typed<128, IA_BF16, false>(aq, ak, num_sms, st)
                               : launch_qk_typed<128, IA_FP16, false>(aq, ak, num_sms, st);
  }
  if (pro)
    return ak.dtype == IA_BF16 ? launch_qk_typed<64, IA_BF16, true>(aq, ak, num_sms, st)
                               : launch_qk_typed<64, IA_FP16, true>(aq, ak, num_sms, st);
  return ak.dtype == IA_BF16 ? launch_qk_typed<64, IA_BF16, false>(aq, ak, num_sms, st)
                             : launch_qk_typed<64, IA_FP16, false>(aq, ak, num_sms, st);
}

cudaError_t launch_quantize(const QuantArgs& a, int num_sms, cudaStream_t st) {
  if (a.S == 0 || a.B == 0 || a.H == 0) return cudaSuccess;
  const bool pro = a.norm_w != nullptr || a.rope != IA_ROPE_NONE;
  if (pro) {
    if (a.D == 128)
      return a.dtype == IA_BF16 ? launch_typed<128, IA_BF16, true>(a, num_sms, st)
                                : launch_typed<128, IA_FP16, true>(a, num_sms, st);
    return a.dtype == IA_BF16 ? launch_typed<64, IA_BF16, true>(a, num_sms, st)
                              : launch_typed<64, IA_FP16, true>(a, num_sms, st);
  }
  if (a.D == 128) {
    return a.dtype == IA_BF16 ? launch_typed<128, IA_BF16, false>(a, num_sms, st)
                              : launch_typed<128, IA_FP16, false>(a, num_sms, st);
  }
  return a.dtype == IA_BF16 ? launch_typed<64, IA_BF16, false>(a, num_sms, st)
                            : launch_typed<64, IA_FP16, false>(a, num_sms, st);
}

}  // namespace ia
