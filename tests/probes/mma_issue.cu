// What the issuing thread's own instruction stream costs tcgen05.mma
// throughput, on one CTA (cta_group::1, kind::f16, K = 16 per MMA).
//
// Each case issues 2000 groups of MMAs back to back and prints the SM clock
// cycles per group (clock64) and whether the final commit's bounded wait
// (0.5 s) completed. A group is 4 SS MMAs (M = 128, N = 128: the QK^T shape)
// or, for the "mix" cases, 4 SS MMAs and 8 TS MMAs (M = 128, N = 64: the
// head-dim-64 P V shape), each followed by a commit. Between groups a case
// adds nothing, a fence, or a wait on an mbarrier phase that has already
// completed (so the wait returns at once), or a poll of a shared-memory word
// that is already set (an acquire load, or a volatile one). The two-issuer case
// runs the mix with waits from one thread in each of two warps (disjoint
// accumulators) and prints cycles per group of the two together.
//
// Operand values do not affect the time: shared memory holds zeros, the TMEM A
// operand whatever the allocation held. Every wait is bounded.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "../../int8_qk_quantized_gb300/csrc/ptx.cuh"

__device__ __forceinline__ uint32_t ld_acq(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];"
               : "=r"(v)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_vol(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];"
               : "=r"(v)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p)))
               : "memory");
  return v;
}

using namespace ia;

namespace {

constexpr int kGroups = 2000;
constexpr int kSmem = 52 * 1024;

__device__ __forceinline__ void wait_done(uint32_t bar) {
  for (int g = 0; g < 1000 && !mbar_try_wait(bar, 0); ++g) {
  }
}

template <bool ACQ>
__device__ __forceinline__ void poll_flag(const uint32_t* f) {
  for (int g = 0; g < 1000; ++g)
    if ((ACQ ? ld_acq(f) : ld_vol(f)) == 1u) break;
}

// CASE 0: 4 SS; 1: + commit + fence::after_thread_sync; 2: + commit + wait;
// 3: + commit + wait + fence; 4: mix without waits; 5: mix with a wait (and
// fence) after each commit; 6: case 5 on two issuers; 7, 8: case 3 with an
// acquire / volatile poll of a set word instead of the wait; 9, 10: case 5
// likewise.
template <int CASE>
__global__ void __launch_bounds__(128) probe(unsigned long long* out) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* a_tile = sm;           // 128 rows x 64 fp16, SW128 K-major (16 KB)
  uint8_t* b_tile = sm + 16384;   // 128 rows x 64 fp16, or V as 64 keys x 64 columns
  const uint32_t bars = smem_u32(sm + 49152);  // done[2], commit[2], pre
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 49152 + 64);
  for (int i = tid; i < 49152 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(bars + 8 * i, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t pre = bars + 32;
  if (tid == 0) mbar_arrive(pre);  // phase 0 of `pre` completes here
  if (tid == 0) slot[1] = 1u;      // the flag the poll cases read
  __syncthreads();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(slot);
  const int who = (CASE == 6) ? (lane == 0 && warp < 2 ? warp : -1) : (tid == 0 ? 0 : -1);
  if (who >= 0) {
    const uint32_t idq = idesc_f16(128, 128, 0, 0, 0, 0);
    const uint32_t idv = idesc_f16(128, 64, 0, 0, 0, 1);
    const uint64_t ad = sdesc_sw128(smem_u32(a_tile), 16, 1024);
    const uint64_t bd = sdesc_sw128(smem_u32(b_tile), 16, 1024);
    const uint64_t vd = sdesc_sw128(smem_u32(b_tile), 8192, 1024);
    const uint32_t dq = tmem + who * 128, dv = tmem + 256 + who * 64, pa = tmem + 384 + who * 64;
    const uint32_t done = bars + 8 * who, cbar = bars + 16 + 8 * who;
    const int groups = CASE == 6 ? kGroups / 2 : kGroups;
    const long long t0 = clock64();
    for (int r = 0; r < groups; ++r) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(dq, ad + ((kk * 32) >> 4), bd + ((kk * 32) >> 4), idq, (r | kk) ? 1u : 0u);
      if constexpr (CASE >= 1) mma_commit(cbar);
      if constexpr (CASE == 2 || CASE == 3 || (CASE >= 5 && CASE <= 6)) wait_done(pre);
      if constexpr (CASE == 7 || CASE == 9) poll_flag<true>(slot + 1);
      if constexpr (CASE == 8 || CASE == 10) poll_flag<false>(slot + 1);
      if constexpr (CASE == 1 || CASE == 3 || CASE >= 5) tc_fence_after();
      if constexpr (CASE == 4 || CASE == 5 || CASE == 6 || CASE >= 9) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(dv, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), idv, (r | kk) ? 1u : 0u);
        mma_commit(cbar);
        if constexpr (CASE == 5 || CASE == 6) {
          wait_done(pre);
          tc_fence_after();
        }
        if constexpr (CASE >= 9) {
          poll_flag<CASE == 9>(slot + 1);
          tc_fence_after();
        }
      }
    }
    mma_commit(done);
    const uint64_t g0 = globaltimer_ns();
    bool ok = true;
    while (!mbar_try_wait(done, 0))
      if (globaltimer_ns() - g0 > 500000000ull) {
        ok = false;
        break;
      }
    out[2 * who] = static_cast<unsigned long long>(clock64() - t0);
    out[2 * who + 1] = ok ? 1 : 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int CASE>
void run(unsigned long long* d, const char* name) {
  cudaFuncSetAttribute(probe<CASE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  cudaMemset(d, 0, 64);
  probe<CASE><<<1, 128, kSmem>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    printf("cuda error %s\n", cudaGetErrorString(e));
    exit(1);
  }
  unsigned long long h[4];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  const unsigned long long t = CASE == 6 ? (h[0] > h[2] ? h[0] : h[2]) : h[0];
  const bool ok = h[1] == 1 && (CASE != 6 || h[3] == 1);
  printf("case %d %s: %.1f cycles per group, done=%d\n", CASE, name, double(t) / kGroups, ok ? 1 : 0);
}

}  // namespace

int main() {
  unsigned long long* d;
  if (cudaMalloc(&d, 64) != cudaSuccess) return 1;
  run<0>(d, "4SS");
  run<1>(d, "4SS+commit+fence");
  run<2>(d, "4SS+commit+wait");
  run<3>(d, "4SS+commit+wait+fence");
  run<4>(d, "mix");
  run<5>(d, "mix+waits");
  run<6>(d, "mix+waits,two-issuers");
  run<7>(d, "4SS+commit+acquire-poll+fence");
  run<8>(d, "4SS+commit+volatile-poll+fence");
  run<9>(d, "mix+acquire-polls");
  run<10>(d, "mix+volatile-polls");
  return 0;
}
