// Exact merge of two partial attentions over disjoint key sets through their
// log-sum-exps: "int8_attention: masked path costs ~1.8x unmasked, and a
// request for optional return_lse", Question 2 (core + skirt calls merged
// exactly), and "Add optional forward LSE output", Kernel implementation
// (the split-K combine's LSE comes from the combined maximum and denominator).
//
//   M = max(L1, L2); w_k = exp(L_k - M); L = M + ln(w1 + w2)
//   O = (w1*O1 + w2*O2) / (w1 + w2);   M = -inf gives O = 0, L = -inf.
//
// A streaming kernel: each row is D/8 threads holding 8 elements (16 bytes) of
// O1, O2 and O, with FP32 arithmetic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"

namespace ia {
namespace {

constexpr int kThreads = 256;

template <int DT>
__device__ __forceinline__ void unpack8(const uint4 w, float (&v)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == IA_BF16) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == IA_BF16) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// Each iteration handles two rows per thread group (this CTA's slot in two
// consecutive grid strides), so a thread has four 16-byte loads in flight.
template <int D, int DT>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeArgs a) {
  constexpr int TPR = D / 8;
  constexpr int RPP = kThreads / TPR;
  constexpr int U = 2;
  const int tc = threadIdx.x % TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * RPP;
  // Uniform trip count per CTA, so the warp barrier below is reached by all lanes.
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * RPP; base < a.rows; base += U * stride) {
    int64_t r[U];
    bool live[U];
    float l1[U], l2[U];
    uint4 w1[U], w2[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      r[u] = base + u * stride + threadIdx.x / TPR;
      live[u] = r[u] < a.rows;
      const int64_t rr = live[u] ? r[u] : 0;
      l1[u] = a.l1[rr];
      l2[u] = a.l2[rr];
      const int64_t off = rr * D + tc * 8;
      w1[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.o1) + off * 2);
      w2[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.o2) + off * 2);
    }
    // Every lane of a row has read its inputs before any lane writes (outputs may alias).
    __syncwarp();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!live[u]) continue;
      const float m = fmaxf(l1[u], l2[u]);
      float o[8];
      float lse;
      if (m == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = 0.f;
        lse = -INFINITY;
      } else {
        const float e1 = expf(l1[u] - m);  // exp(-inf) = 0 for an empty partial
        const float e2 = expf(l2[u] - m);
        const float den = e1 + e2;
        const float c1 = e1 / den, c2 = e2 / den;
        float x1[8], x2[8];
        unpack8<DT>(w1[u], x1);
        unpack8<DT>(w2[u], x2);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = c1 * x1[i] + c2 * x2[i];
        lse = m + logf(den);
      }
      const int64_t off = r[u] * D + tc * 8;
      *reinterpret_cast<uint4*>(static_cast<char*>(a.o) + off * 2) = pack8<DT>(o);
      if (a.l && tc == 0) a.l[r[u]] = lse;
    }
  }
}

template <int D>
cudaError_t launch_d(const MergeArgs& a, int num_sms, cudaStream_t st) {
  constexpr int RPP = kThreads / (D / 8);
  int64_t blocks = (a.rows + RPP - 1) / RPP;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (a.dtype == IA_BF16)
    merge_kernel<D, IA_BF16><<<static_cast<int>(blocks), kThreads, 0, st>>>(a);
  else
    merge_kernel<D, IA_FP16><<<static_cast<int>(blocks), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

// n-way merge: a row is D/8 threads holding 8 output elements each.
template <int D, int DT, bool IN_F32>
__global__ void __launch_bounds__(kThreads) merge_n_kernel(const MergeNArgs a) {
  constexpr int TPR = D / 8;
  constexpr int RPP = kThreads / TPR;
  const int tc = threadIdx.x % TPR;
  const int64_t rows = static_cast<int64_t>(a.B) * a.H * a.Sq;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * RPP;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * RPP; base < rows; base += stride) {
    const int64_t r = base + threadIdx.x / TPR;
    if (r >= rows) continue;
    float m = -INFINITY;
    for (int k = 0; k < a.n; ++k) m = fmaxf(m, a.l[k][r]);
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    float lse = -INFINITY;
    if (m != -INFINITY) {
      float den = 0.f;
      for (int k = 0; k < a.n; ++k) {
        const float w = expf(a.l[k][r] - m);
        if (!(w > 0.f)) continue;  // an empty partial: its O is not read
        den += w;
        float x[8];
        if (IN_F32) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.o[k]) + r * D + tc * 8);
          const float4 x0 = src[0], x1 = src[1];
          x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
          x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
        } else {
          const uint4 w16 = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.o[k]) + (r * D + tc * 8) * 2);
          unpack8<DT>(w16, x);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] += w * x[i];
      }
      const float inv = 1.f / den;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] *= inv;
      lse = m + logf(den);
    }
    const int64_t sidx = r % a.Sq;
    const int64_t bh = r / a.Sq;
    const int64_t hh = bh % a.H, bb = bh / a.H;
    char* dst = static_cast<char*>(a.out) + (bb * a.o_sb + hh * a.o_sh + sidx * a.o_ss + tc * 8) * 2;
    *reinterpret_cast<uint4*>(dst) = pack8<DT>(o);
    if (a.lse && tc == 0) a.lse[bb * a.l_sb + hh * a.l_sh + sidx] = lse;
  }
}

template <int D>
cudaError_t launch_n_d(const MergeNArgs& a, int num_sms, cudaStream_t st) {
  constexpr int RPP = kThreads / (D / 8);
  const int64_t rows = static_cast<int64_t>(a.B) * a.H * a.Sq;
  int64_t blocks = (rows + RPP - 1) / RPP;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const int g = static_cast<int>(blocks);
  if (a.in_f32) {
    if (a.dtype == IA_BF16) merge_n_kernel<D, IA_BF16, true><<<g, kThreads, 0, st>>>(a);
    else merge_n_kernel<D, IA_FP16, true><<<g, kThreads, 0, st>>>(a);
  } else {
    if (a.dtype == IA_BF16) merge_n_kernel<D, IA_BF16, false><<<g, kThreads, 0, st>>>(a);
    else merge_n_kernel<D, IA_FP16, false><<<g, kThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_n(const MergeNArgs& a, int num_sms, cudaStream_t st) {
  if (static_cast<int64_t>(a.B) * a.H * a.Sq == 0) return cudaSuccess;
  return a.D == 128 ? launch_n_d<128>(a, num_sms, st) : launch_n_d<64>(a, num_sms, st);
}

cudaError_t launch_merge(const MergeArgs& a, int num_sms, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  return a.D == 128 ? launch_d<128>(a, num_sms, st) : launch_d<64>(a, num_sms, st);
}

}  // namespace ia
