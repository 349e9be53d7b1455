// The tcgen05 CTA-pair semantics the attention kernel's CTA pairs rely on, checked
// against products computed on the host:
//  * one warp of each CTA of a two-CTA cluster allocates TMEM collectively
//    (cta_group::2) and both receive the same address;
//  * a 256-row MMA issued by the even CTA takes rows 0-127 of A from that CTA
//    and rows 128-255 from its peer (same shared-memory offsets), and N columns
//    0..N/2-1 of B from the even CTA and N/2..N-1 from its peer; each CTA receives
//    its 128 rows of D, all N columns, in its own TMEM;
//  * the same holds with A read from each CTA's TMEM (the P V form);
//  * a multicast commit arrives on the barrier at the same offset in both CTAs.
// SS: D[256 x 128] = A[256 x 64] B[128 x 64]^T; TS: D2 = P[256 x 64] V[64 x 128].
// Integer data, exact in fp32. Every wait is bounded (200 ms); the program prints
// the mismatch counts under both readings of the N split and exits 0.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_fp16.h>
#include "../../int8_qk_quantized_gb300/csrc/ptx.cuh"
using namespace ia;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void alloc2(uint32_t dst, uint32_t n) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(n) : "memory");
}
__device__ __forceinline__ void dealloc2(uint32_t t, uint32_t n) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(n) : "memory");
}
__device__ __forceinline__ void relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void mma_ss2(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_ts2(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
               "r"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void commit2_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(bar), "h"(mask) : "memory");
}

__host__ __device__ inline int fa(int c, int r, int k) { return ((r * 7 + k * 3 + c * 5) % 11) - 5; }
__host__ __device__ inline int fb(int c, int n, int k) { return ((n * 5 + k * 11 + c * 3) % 13) - 6; }
__host__ __device__ inline int fp(int c, int r, int k) { return ((r * 3 + k * 5 + c * 7) % 9) - 4; }
__host__ __device__ inline int fv(int c, int k, int j) { return ((k * 7 + j * 3 + c * 11) % 10) - 5; }

// out1/out2: [2][128][128] floats; info: [2][4]
__global__ void __launch_bounds__(128) probe(float* out1, float* out2, unsigned* info) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t c = cluster_rank();
  const int tid = threadIdx.x, warp = tid >> 5;
  uint8_t* A = sm;            // 128 x 64 f16 K-major SW128
  uint8_t* B = sm + 16384;    // 64 x 64 f16 K-major SW128
  uint8_t* V = sm + 24576;    // 64 keys x 64 n, MN-major SW128
  const uint32_t bar = smem_u32(sm + 32768);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 32800);
  unsigned status = 0;

  if (warp == 0) alloc2(smem_u32(slot), 256);
  for (int i = tid; i < 128 * 64; i += 128) {
    const int r = i / 64, k = i % 64;
    *reinterpret_cast<__half*>(A + r * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2) = __int2half_rn(fa(c, r, k));
  }
  for (int i = tid; i < 64 * 64; i += 128) {
    const int n = i / 64, k = i % 64;
    *reinterpret_cast<__half*>(B + n * 128 + (((k >> 3) ^ (n & 7)) << 4) + (k & 7) * 2) = __int2half_rn(fb(c, n, k));
    const int kk = i / 64, j = i % 64;
    *reinterpret_cast<__half*>(V + kk * 128 + (((j >> 3) ^ (kk & 7)) << 4) + (j & 7) * 2) = __int2half_rn(fv(c, kk, j));
  }
  fence_proxy_async_smem();
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init_cluster(); }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(slot);

  if (c == 0 && tid == 0) {
    const uint32_t id = idesc_f16(256, 128, 0, 0, 0, 0);
    for (int kk = 0; kk < 4; ++kk)
      mma_ss2(tmem, sdesc_sw128(smem_u32(A) + kk * 32, 16, 1024), sdesc_sw128(smem_u32(B) + kk * 32, 16, 1024),
              id, kk > 0);
    commit2_mc(bar, 3);
  }
  auto wait = [&](uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
      if (globaltimer_ns() - t0 > 200000000ull) { status |= 1u << parity; return false; }
    }
    return true;
  };
  const int row = warp * 32 + (tid & 31);
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  if (wait(0)) {
    tc_fence_after();
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + c0, r);
      tmem_wait_ld(r);
      for (int e = 0; e < 32; ++e) out1[(c * 128 + row) * 128 + c0 + e] = __uint_as_float(r[e]);
    }
  }
  // P rows into TMEM columns 128..159 (fp16 pairs)
  {
    uint32_t r[32];
    for (int e = 0; e < 32; ++e) {
      __half2 h = __halves2half2(__int2half_rn(fp(c, row, 2 * e)), __int2half_rn(fp(c, row, 2 * e + 1)));
      r[e] = *reinterpret_cast<uint32_t*>(&h);
    }
    tmem_st32(tmem + lane_off + 128, r);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (c == 0 && tid == 0 && status == 0) {
    const uint32_t id = idesc_f16(256, 128, 0, 0, 0, 1);
    for (int kk = 0; kk < 4; ++kk)
      mma_ts2(tmem, tmem + 128 + kk * 8, sdesc_sw128(smem_u32(V) + kk * 16 * 128, 8192, 1024), id, kk > 0);
    commit2_mc(bar, 3);
  }
  if (status == 0 && wait(1)) {
    tc_fence_after();
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + c0, r);
      tmem_wait_ld(r);
      for (int e = 0; e < 32; ++e) out2[(c * 128 + row) * 128 + c0 + e] = __uint_as_float(r[e]);
    }
  }
  if (status) atomicOr(&info[c * 4 + 1], status);
  if (tid == 0) info[c * 4 + 0] = tmem;
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) { dealloc2(tmem, 256); relinquish2(); }
}

int main() {
  float *d1, *d2; unsigned* di;
  cudaMalloc(&d1, 2 * 128 * 128 * 4); cudaMalloc(&d2, 2 * 128 * 128 * 4); cudaMalloc(&di, 8 * 4);
  cudaMemset(d1, 0xff, 2 * 128 * 128 * 4); cudaMemset(d2, 0xff, 2 * 128 * 128 * 4); cudaMemset(di, 0, 32);
  const int smem = 48 * 1024;
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2); cfg.blockDim = dim3(128); cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  cfg.attrs = at; cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, probe, d1, d2, di);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { printf("cuda error: %s\n", cudaGetErrorString(e)); return 1; }
  std::vector<float> h1(2 * 128 * 128), h2(2 * 128 * 128); unsigned hi[8];
  cudaMemcpy(h1.data(), d1, h1.size() * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h2.data(), d2, h2.size() * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(hi, di, 32, cudaMemcpyDeviceToHost);
  printf("tmem addr cta0 %08x cta1 %08x; status %u %u\n", hi[0], hi[4], hi[1], hi[5]);
  // hypotheses for the N split: h=0 CTA0 holds n<64; h=1 CTA1 holds n<64
  for (int h = 0; h < 2; ++h) {
    long bad1 = 0, bad2 = 0;
    for (int c = 0; c < 2; ++c)
      for (int r = 0; r < 128; ++r)
        for (int n = 0; n < 128; ++n) {
          const int owner = ((n < 64) ? 0 : 1) ^ h, nn = n & 63;
          double s1 = 0, s2 = 0;
          for (int k = 0; k < 64; ++k) {
            s1 += fa(c, r, k) * fb(owner, nn, k);
            s2 += fp(c, r, k) * fv(owner, k, nn);
          }
          bad1 += h1[(c * 128 + r) * 128 + n] != (float)s1;
          bad2 += h2[(c * 128 + r) * 128 + n] != (float)s2;
        }
    printf("hypothesis %d: SS mismatches %ld, TS mismatches %ld of %d\n", h, bad1, bad2, 2 * 128 * 128);
  }
  printf("sample SS c0 r0: %g %g %g | c1 r5: %g %g\n", h1[0], h1[1], h1[64], h1[(128 + 5) * 128 + 0], h1[(128 + 5) * 128 + 100]);
  return 0;
}
