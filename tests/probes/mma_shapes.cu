// Cycles per tcgen05.mma kind::f16 for the shapes the attention kernels choose
// between, on one CTA (cta_group::1, K = 16 per MMA): M = 64 against M = 128
// (one block-sparse query tile per MMA, or two tiles sharing the union of
// their key lists), N = 64 / 128 / 256, with A from shared memory (SS, the QK^T
// form, K-major SW128) and from TMEM (TS, the P V form, B MN-major SW128).
// Each case issues 8000 MMAs back to back from one thread, commits, waits for
// the commit (bounded, 0.5 s) and prints the cycles per MMA (clock64) and
// whether the wait completed. Operand values do not affect the time: shared
// memory holds zeros, the TMEM A operand whatever the allocation held.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include "../../int8_qk_quantized_gb300/csrc/ptx.cuh"
using namespace ia;

__global__ void __launch_bounds__(128) probe(unsigned long long* out, int M, int N, int reps, int ts) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  uint8_t* A = sm;            // 128 rows x 64 K fp16 (16 KB)
  uint8_t* B = sm + 16384;    // 256 rows x 64 K fp16 (32 KB): N up to 256
  const uint32_t bar = smem_u32(sm + 49152);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 49152 + 64);
  for (int i = tid; i < 49152 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) { tmem_alloc(smem_u32(slot), 256); tmem_relinquish(); }
  if (tid == 0) { mbar_init(bar, 1); fence_mbar_init(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(slot);
  if (tid == 0) {
    const uint32_t id = idesc_f16(M, N, 0, 0, 0, 0);
    const uint64_t ad = sdesc_sw128(smem_u32(A), 16, 1024);
    const uint64_t bd = sdesc_sw128(smem_u32(B), 16, 1024);
    // TS: A (M x 16 fp16 per MMA) from TMEM columns 192..223, D in columns 0..N-1
    const uint64_t vd = sdesc_sw128(smem_u32(B), 8192, 1024);  // B MN-major (as V), N <= 64 per block
    const uint32_t idv = idesc_f16(M, N, 0, 0, 0, 1);
    const long long t0 = clock64();
    if (ts) {
      for (int r = 0; r < reps; ++r)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem, tmem + 192 + kk * 8, vd + ((kk * 16 * 128) >> 4), idv, (r | kk) ? 1u : 0u);
    } else {
      for (int r = 0; r < reps; ++r)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, ad + ((kk * 32) >> 4), bd + ((kk * 32) >> 4), id, (r | kk) ? 1u : 0u);
    }
    const long long t1 = clock64();
    mma_commit(bar);
    const uint64_t g0 = globaltimer_ns();
    bool ok = true;
    while (!mbar_try_wait(bar, 0))
      if (globaltimer_ns() - g0 > 500000000ull) { ok = false; break; }
    const long long t2 = clock64();
    out[0] = static_cast<unsigned long long>(t1 - t0);
    out[1] = static_cast<unsigned long long>(t2 - t0);
    out[2] = ok ? 1 : 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

int main() {
  unsigned long long* d;
  cudaMalloc(&d, 64);
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, 52 * 1024);
  const int reps = 2000;
  for (int ts = 0; ts < 2; ++ts)
  for (int M : {64, 128})
    for (int N : {64, 128, 256}) {
      if (ts && N > 128) continue;  // TS: B as one or two 64-column V blocks within the 32 KB buffer
      for (int t = 0; t < 2; ++t) {
        cudaMemset(d, 0, 64);
        probe<<<1, 128, 52 * 1024>>>(d, M, N, reps, ts);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) { printf("cuda error %s\n", cudaGetErrorString(e)); return 1; }
        unsigned long long h[3];
        cudaMemcpy(h, d, 24, cudaMemcpyDeviceToHost);
        const double per = double(h[1]) / (reps * 4);
        const double flop = 2.0 * M * N * 16;
        printf("%s M=%d N=%d K=16: %.1f cycles per MMA (issue %.1f), %.0f flop/cycle, done=%llu\n", ts ? "TS" : "SS", M, N, per,
               double(h[0]) / (reps * 4), flop / per, h[2]);
      }
    }
  return 0;
}
