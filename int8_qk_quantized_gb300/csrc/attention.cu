// Forward attention with INT8 Q/K and a 16-bit P.V on sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes ("minimax_h3_sparse_int8", FastVideo API page, module
// description and sparse_sm89_attention; "int8_attention: masked path costs
// ~1.8x unmasked, and a request for optional return_lse", opening paragraph;
// "Add optional forward LSE output", Summary):
//   s_ij = sm_scale * qs_i * ks_j * <q8_i, k8_j> + bias_j       (or -inf if masked)
//   O_i  = v_scale (*) sum_j softmax_j(s_i.) v_j,   LSE_i = ln sum_j e^{s_ij}
//
// How, on GB300:
//  * INT8 codes in [-127, 127] are exact in FP16, each product is exact in
//    FP32 and every partial sum of a D <= 128 dot product stays below 2^24, so
//    the QK^T MMA runs as tcgen05 kind::f16 on FP16-coded codes and yields the
//    exact integer dot products in its FP32 accumulator (sm_103a has no
//    kind::i8). The int8 tiles travel from HBM by TMA at one byte per element
//    and two converter warps widen them in shared memory into the 128-byte
//    swizzled K-major layout the MMA reads.
//  * A CTA owns QS query stages of 128 rows. One thread issues the MMAs:
//    S_s = Q_s K_j^T into TMEM, then O_s += P_s V_j with P_s read from TMEM.
//    While the softmax warpgroup of one stage works on its S tile, the tensor
//    core runs the other stage's MMAs.
//  * Dense D = 128 runs as CTA pairs (clusters of two): the even CTA issues
//    256-row MMAs (cta_group::2) over both CTAs' query rows; each CTA holds and
//    widens half of every K tile and half of V's columns, which cuts each SM's
//    operand reads from shared memory by a third and its widening by half.
//  * Softmax warpgroups own one query row per thread (TMEM lane = row). They
//    apply k_scale (and bias, masks) to the FP32 logits, keep a running
//    maximum in log2 units, rescale O in TMEM only when the maximum grew by
//    more than 8 (2^8 headroom in P), write P as bf16/f16 into the S columns
//    and keep the row sum in FP32. The epilogue applies 1/l and the
//    per-channel V scale once and writes the LSE in natural log.
//  * The per-key bias and the k scales are loaded once per key tile into
//    shared memory and read by all query rows (the [1,1,1,K] broadcast).
//  * Block-sparse: one 128-row stage (two 64-row query tiles) walks the
//    union of its tiles' kept key tiles (64 keys each); rows whose own query
//    tile dropped a key tile write P = 0 for it without reading S.
//  * Every mbarrier wait is bounded. When one runs out the kernel records it
//    in a device status word, stops issuing work, drains what is in flight,
//    frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdio>
#include <cstring>

#include "launch.h"
#include "ptx.cuh"

namespace ia {

__device__ unsigned int g_attn_status;

// Phase timestamps of CTA (0,0,0), compiled in only with -DIA_TRACE (a
// profiling build; the library never defines it).
#ifdef IA_TRACE
__device__ unsigned long long g_attn_trace[16][64];
#define IA_TRACE_POINT(slot, it)                                                   \
  do {                                                                               \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (it) < 64)          \
      g_attn_trace[slot][it] = clock64();                                            \
  } while (0)
#else
#define IA_TRACE_POINT(slot, it) \
  do {                           \
  } while (0)
#endif

namespace {

constexpr int kM = 128;              // query rows per stage (MMA M)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8

enum : unsigned {
  kErrProducer = 1u,
  kErrConverter = 2u,
  kErrMma = 4u,
  kErrSoftmax = 8u,
  kErrDrain = 16u,
  kErrSmemAlign = 32u,
};

struct Params {
  const float* q_scale;
  const float* k_scale;
  const void* bias;  // per-key offsets: the fp32 bias, or a mask whose query stride is 0
  int bias_dtype;    // ia_mask_dtype
  int64_t bias_sb, bias_sh;  // element strides of the per-(b,h) key rows (0 broadcasts)
  int rm_dtype;      // ROWMASK kernels: ia_mask_dtype of the per-row mask tiles
  int rm_h, rm_b;    //   1 if the mask has that dimension (0: broadcast, coordinate 0)
  const uint8_t* mask;
  const int32_t* kv_valid;
  const float* v_scale;
  void* out;
  float* lse;
  int H, Sq, Sk;
  int n_tiles;   // key tiles (dense); mask width Tk (sparse)
  int Tq, Tk;
  float cq_mult;  // sm_scale * log2(e)
  int gran_block;
  int pad_query;
  int64_t qs_sb, qs_sh, ks_sb, ks_sh;
  int64_t o_sb, o_sh, o_ss;
  int64_t l_sb, l_sh;
  unsigned long long timeout_ns;
  int debug_stall;
  int nsplit;        // key ranges per (query tiles, head); 1 = no split
  int tps;           // dense: key tiles per range
  float* ws_o;       // nsplit >= 2: fp32 partial O [nsplit][B][H][Sq][D]
  float* ws_l;       //              fp32 partial LSE [nsplit][B][H][Sq]
  int64_t seg_units;  // > 0 (nsplit == 2): balanced segments over B*H*seg_nqt*n_tiles units
  int seg_nqt;        // query tiles of kM*QS rows per (b, h)
  int B;
  // QRAW kernels: RMSNorm + RoPE of the Q rows before the in-kernel quantization
  int q_pro;          // 1: apply the fields below
  const float* qp_w;   // fp32 [D] or null
  float qp_eps;
  int qp_rope;         // ia_rope_layout
  const float* qp_cos;
  const float* qp_sin;
  int64_t qp_stride;
  int qp_pos0;
};

template <int D, int QS, int BN, bool SPARSE, bool ROWMASK = false, bool PAIR = false,
          bool KB = false>
struct Layout {
  // Block-sparse, D == 128: the int8 K tile lands (by TMA) in the second
  // 64-column block of its fp16 K buffer and is widened in place, which keeps
  // the CTA small enough for two per SM. Otherwise it has staging buffers.
  static constexpr bool INPLACE = SPARSE && D == 128;
  static constexpr int NKS = 2, NVS = 2, NSC = 2;
  static constexpr int NRS = INPLACE ? 0 : 2;
  // A CTA pair (PAIR) holds half of each key tile's K rows and half of V's
  // columns per CTA; the 256-row MMA reads the other halves from the peer.
  // One query stage (QS == 1): S is double-buffered in TMEM, so the QK^T of
  // key tile j+1 runs while the softmax works on tile j; B_PVT then counts the
  // P V of every tile (the softmax waits on it before rescaling O). B_OF is
  // committed once, after the last P V, in every kernel: the epilogue waits
  // on its single phase.
  static constexpr bool DBS = QS == 1;
  // dense single-CTA head-dim-64 kernels can take a balanced share of the
  // (query tile, key tile) units in segments (Params::seg_units; not with the
  // in-kernel Q quantization, whose registers the segment loop would spill)
  static constexpr bool SEGOK = D == 64 && QS == 2 && !PAIR && !SPARSE && !ROWMASK;
  static constexpr int NSB = DBS ? 2 : QS;  // S buffers in TMEM
  static constexpr int KROWS = PAIR ? BN / 2 : BN;  // keys of a K tile held here
  static constexpr int VCOLS = PAIR ? D / 2 : D;    // V columns held here
  // Dense head dim 64 with per-row K scales (single CTAs): the P V MMA has
  // N = D + 16, its last 16 columns reading a block of ones in shared memory,
  // so that column D of O accumulates the row sum of the 16-bit P the MMA
  // multiplied (the softmax keeps no running sum). A ones block sits at a fixed
  // distance (the descriptor's leading byte offset) from each V buffer. With
  // per-block K scales (KB) the softmax is light and the tensor core sets the
  // pace, so the extra MMA columns would cost more than the sum they save.
  static constexpr bool ONES = D == 64 && QS == 2 && !PAIR && !SPARSE && !ROWMASK && !KB;
  static constexpr int OW = D + (ONES ? 16 : 0);  // O columns per stage in TMEM
  static constexpr int QH = kM * D * 2;      // fp16 Q stage
  static constexpr int KH = KROWS * D * 2;   // fp16 K tile
  static constexpr int VB = BN * VCOLS * 2;  // 16-bit V tile
  static constexpr int KR = KROWS * D;       // int8 K tile
  static constexpr int QR = kM * D;          // int8 Q stage
  // Q staging: the V buffers, or (PAIR, whose V buffers are too small) a
  // region of its own sized for 16-bit rows.
  static constexpr int QST = PAIR ? QS * kM * D * 2 : 0;
  static constexpr int SC = BN * 8 + 16;  // k scales, bias*log2e, flags
  // Per-row mask tile (ROWMASK): kM rows x BN keys as TMA boxes of 128-byte
  // rows with the 128-byte swizzle; 32 fp32, 64 16-bit or 128 bool keys per box.
  // Sized for two fp32 boxes of one stage, or (QS == 2, masks of at most two
  // bytes) one box per stage.
  static constexpr int MB = ROWMASK ? BN * 4 * kM : 0;
  static constexpr int OFF_QH = 0;
  static constexpr int OFF_KH = OFF_QH + QS * QH;
  static constexpr int OFF_V = OFF_KH + NKS * KH;
  static constexpr int OFF_KR = OFF_V + NVS * VB;
  static constexpr int OFF_QST = OFF_KR + NRS * KR;
  static constexpr int OFF_QIN = PAIR ? OFF_QST : OFF_V;  // where Q lands before conversion
  static constexpr int OFF_ONES = OFF_QST + QST;  // ONES: NVS blocks of BN x 64 ones
  static constexpr int OFF_MK = OFF_ONES + (ONES ? NVS * VB : 0);
  static constexpr int OFF_SC = OFF_MK + NSC * MB;
  static constexpr int OFF_VS = OFF_SC + NSC * SC;
  static constexpr int OFF_BAR = (OFF_VS + D * 4 + 7) / 8 * 8;
  // barrier indices
  static constexpr int B_QFULL = 0, B_QCONV = 1, B_KRF = 2, B_KRE = B_KRF + NKS,
                       B_KCF = B_KRE + NRS, B_KCE = B_KCF + NKS, B_VF = B_KCE + NKS,
                       B_VE = B_VF + NVS, B_SCF = B_VE + NVS, B_SCE = B_SCF + NSC,
                       B_SF = B_SCE + NSC, B_PF = B_SF + NSB, B_OF = B_PF + NSB,
                       B_PVT = B_OF + QS, B_DRAIN = B_PVT + 1, B_STALL = B_DRAIN + 1,
                       B_MF = B_STALL + 1, NBAR = B_MF + NSC;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;       // tmem base, abort, count, pad
  static constexpr int OFF_LIST = OFF_MISC + 16 + 32;       // + warp counts for the list scan
  static constexpr int SMEM_FIXED = OFF_LIST;
  static constexpr int TMEM_NEED = NSB * BN + QS * OW;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                   : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int NWARPS = 4 * QS + 4;
  static constexpr int W_PROD = 4 * QS, W_MMA = 4 * QS + 1, W_CONV = 4 * QS + 2;
  static_assert(PAIR || QS * QR <= NVS * VB, "int8 Q is staged in the V buffers");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(OFF_QH % 1024 == 0 && OFF_KH % 1024 == 0 && OFF_V % 1024 == 0 &&
                    OFF_MK % 1024 == 0 && OFF_QST % 1024 == 0 && OFF_ONES % 1024 == 0,
                "swizzle align");
  static_assert(!ONES || (VB == BN * 128 && (OFF_ONES - OFF_V) / 16 < (1 << 14)),
                "one 64-column V block per buffer; the ones within the descriptor's reach");
  static_assert(!ROWMASK || ((QS == 1 || QS == 2) && BN == 64 && !SPARSE), "row-mask shape");
  static_assert(!INPLACE || KR == BN * 128, "the int8 tile fills one 64-column fp16 block");
  // the pair's V half is one 64-column swizzle block; dense tiles only
  static_assert(!PAIR || (D == 128 && QS == 2 && BN == 128 && !SPARSE && !ROWMASK), "pair shape");
};

struct Ctl {
  volatile int* abort;
  unsigned long long timeout;
};

// Bounded wait on an mbarrier phase. Returns false when the wait ran out here
// (the status word and the CTA's abort flag are set) or another thread of
// the CTA has already aborted.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const Ctl& c,
                                           unsigned code) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if ((n & 15u) == 0 && *reinterpret_cast<volatile unsigned*>(&g_attn_status) != 0u) {
      *c.abort = 1;  // another CTA already timed out: stop waiting as well
      return false;
    }
    if ((n & 15u) == 0 && globaltimer_ns() - t0 > c.timeout) {
      *c.abort = 1;
      atomicOr(&g_attn_status, code);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                         unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, c, code);
}

// Bounded wait that ignores the abort flag: used to let copies and MMAs that
// were already issued land before the CTA releases its shared memory and TMEM.
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned long long timeout) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return;
    if ((n & 15u) == 15u && globaltimer_ns() - t0 > timeout) {
      atomicOr(&g_attn_status, kErrDrain);
      return;
    }
  }
}

// int8 tile [ROWS x D] row-major -> fp16 [ROWS x D] in 128-byte-swizzled
// K-major blocks of 64 columns (block stride ROWS*128 bytes), as tcgen05 reads
// with a SWIZZLE_128B descriptor. 64 threads; each row belongs to one warp.
// IN_PLACE: `raw` is the second block of `dst` (D == 128), so every lane reads
// its chunks before any lane of the warp writes a row back.
// A 16-byte access is served in phases of 8 lanes. For D == 128 the 32 lanes
// of a warp take 4 rows, and each 8-lane phase takes half of one row and the
// other half of the next: its int8 reads then cover all 32 banks once, and its
// fp16 writes land in 8 distinct 16-byte slots of the swizzle (a phase holding
// one whole row would write both 64-column blocks to the same slots).
template <int D, int ROWS, bool IN_PLACE>
__device__ __forceinline__ void widen_tile(const uint8_t* raw, uint8_t* dst, int ct) {
  constexpr int CPR = D / 16;              // 16-byte int8 chunks per row
  constexpr int NI = ROWS * CPR / 64;      // chunks per thread
  // Chunks loaded before any is stored. In place, all of them: a warp owns
  // whole rows and a row's fp16 output overwrites only its own int8 row, so one
  // warp barrier after the loads suffices (instead of a load-barrier-store
  // round trip per chunk). From a staging buffer, one at a time; the loop is
  // kept rolled, as unrolling it cost the masked softmax registers (and
  // loading all of a thread's chunks first measured slower in the pairs).
  constexpr int NB = IN_PLACE ? NI : 1;
  static_assert(ROWS * CPR % 64 == 0 && NI % NB == 0, "widen layout");
#pragma unroll 1
  for (int i0 = 0; i0 < NI; i0 += NB) {
    uint4 w[NB];
    int rr[NB], cc[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int idx = ct + 64 * (i0 + j);
      if constexpr (CPR == 8) {
        const int lane = idx & 31, p = lane >> 3, q = lane & 7, hf = q >> 2;
        rr[j] = ((idx & ~31) >> 3) + 2 * (p >> 1) + hf;
        cc[j] = (((p & 1) ^ hf) << 2) | (q & 3);
      } else {
        rr[j] = idx / CPR;
        cc[j] = idx % CPR;
      }
      w[j] = *reinterpret_cast<const uint4*>(raw + rr[j] * D + cc[j] * 16);
    }
    if (IN_PLACE) __syncwarp();
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      uint32_t h[8];
      i8x4_to_f16x4(w[j].x, h[0], h[1]);
      i8x4_to_f16x4(w[j].y, h[2], h[3]);
      i8x4_to_f16x4(w[j].z, h[4], h[5]);
      i8x4_to_f16x4(w[j].w, h[6], h[7]);
      const int blk = cc[j] >> 2;          // 64-column block
      const int k0 = (cc[j] & 3) * 2;      // first 16-byte chunk within the 128-byte row
      uint8_t* rowp = dst + blk * (ROWS * 128) + rr[j] * 128;
      const int sw = rr[j] & 7;
      *reinterpret_cast<uint4*>(rowp + ((k0 ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(rowp + (((k0 + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// max |x| over one row of D 16-bit values in shared memory, as the 16-bit
// pattern of |x| (for non-negative IEEE values the pattern order is the value
// order). Thread r starts at chunk r so that a warp's 32 rows spread over the
// shared-memory banks.
template <int D>
__device__ __forceinline__ uint32_t row_amax_bits(const uint8_t* row, int r) {
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  uint32_t am = 0;
#pragma unroll
  for (int c = 0; c < CPR; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + ((c + r) & (CPR - 1)) * 16);
    am = max_u16x2(am, w.x & 0x7fff7fffu);
    am = max_u16x2(am, w.y & 0x7fff7fffu);
    am = max_u16x2(am, w.z & 0x7fff7fffu);
    am = max_u16x2(am, w.w & 0x7fff7fffu);
  }
  return max(am & 0xffffu, am >> 16);
}

template <bool BF16>
__device__ __forceinline__ float half_bits_to_float(uint32_t b) {
  if constexpr (BF16) return __uint_as_float(b << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

template <bool BF16>
__device__ __forceinline__ float2 unpack_16x2(uint32_t w) {
  if constexpr (BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Round-half-to-even to an integer, for |v| < 2^22: adding 1.5 * 2^23 leaves
// no fraction bits, so the IEEE addition rounds v to the nearest integer
// (ties to even, as 1.5 * 2^23 is even) and the subtraction is exact.
__device__ __forceinline__ float rne_integer(float v) {
  return __fsub_rn(__fadd_rn(v, 12582912.0f), 12582912.0f);
}

// Symmetric INT8 quantization of one Q row inside the kernel ("minimax_h3_
// sparse_int8", FastVideo API page, quant_qk_int8 and the per-token or
// per-64-row-block scale layouts): scale = amax / 127, code =
// rne(x * (127 / amax)), both divisions IEEE-rounded, amax = 0 gives codes 0.
// |code| <= 127 without a clamp: x * fl(127/amax) <= 127 (1 + 2^-24), which
// rounds to at most 127 + 2^-17 and then to the integer 127. The codes go to
// the fp16 Q stage in the 128-byte-swizzled K-major layout the MMA reads;
// returns the scale. `inv` is 0 for rows that are not quantized (padding).
template <int D, bool BF16>
__device__ __forceinline__ void write_q_codes(const uint8_t* row, uint8_t* qh, int r, float inv) {
  constexpr int CPR = D / 8;
#pragma unroll
  for (int c = 0; c < CPR; ++c) {
    const int cc = (c + r) & (CPR - 1);
    const uint4 w = *reinterpret_cast<const uint4*>(row + cc * 16);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_16x2<BF16>(in[e]);
      hv[e] = cvt_f16x2(rne_integer(__fmul_rn(f.x, inv)), rne_integer(__fmul_rn(f.y, inv)));
    }
    const int blk = cc >> 3, k0 = cc & 7;  // 64-column block, 16-byte chunk in the row
    *reinterpret_cast<uint4*>(qh + blk * (kM * 128) + r * 128 + ((k0 ^ (r & 7)) << 4)) =
        make_uint4(hv[0], hv[1], hv[2], hv[3]);
  }
}

// One thread's int8 row of D codes (row r of a kM-row stage) -> fp16 codes in
// the 128-byte-swizzled K-major layout widen_tile writes (64-column blocks
// kM*128 bytes apart). Thread r starts at chunk r so that a warp's rows spread
// over the shared-memory banks.
template <int D>
__device__ __forceinline__ void widen_row(const uint8_t* row, uint8_t* qh, int r) {
  constexpr int CPR = D / 16;  // 16-byte int8 chunks in the row
#pragma unroll
  for (int c = 0; c < CPR; ++c) {
    const int cc = (c + r) & (CPR - 1);
    const uint4 w = *reinterpret_cast<const uint4*>(row + cc * 16);
    uint32_t hv[8];
    i8x4_to_f16x4(w.x, hv[0], hv[1]);
    i8x4_to_f16x4(w.y, hv[2], hv[3]);
    i8x4_to_f16x4(w.z, hv[4], hv[5]);
    i8x4_to_f16x4(w.w, hv[6], hv[7]);
    const int blk = cc >> 2, k0 = (cc & 3) * 2;  // 64-column block, first 16-byte chunk
    uint8_t* rowp = qh + blk * (kM * 128) + r * 128;
    *reinterpret_cast<uint4*>(rowp + ((k0 ^ (r & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(rowp + (((k0 + 1) ^ (r & 7)) << 4)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
  }
}

// One per-key offset of a key row of a general mask, in two steps so that the
// load can be issued early and converted later: the raw bits of element
// `key`, then their value in logit units (float dtypes as they are, bool as
// 0 or -inf).
__device__ __forceinline__ uint32_t key_bias_bits(const void* row, int key, int dt) {
  if (dt == IA_MASK_F32) return __ldg(reinterpret_cast<const unsigned int*>(row) + key);
  if (dt == IA_MASK_BOOL) return __ldg(reinterpret_cast<const unsigned char*>(row) + key);
  return __ldg(reinterpret_cast<const unsigned short*>(row) + key);
}

__device__ __forceinline__ float key_bias_value(uint32_t bits, int dt) {
  if (dt == IA_MASK_F32) return __uint_as_float(bits);
  if (dt == IA_MASK_BF16) return __uint_as_float(bits << 16);
  if (dt == IA_MASK_F16) return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
  return bits ? 0.f : -INFINITY;
}

// Four consecutive keys c..c+3 of row r of a per-row mask tile in shared
// memory (TMA boxes of 128-byte rows, 128-byte swizzle: 16-byte chunk j of
// row r sits at chunk j ^ (r & 7)), as logit offsets.
__device__ __forceinline__ void row_mask4(const uint8_t* buf, int r, int c, int dt, float out[4]) {
  const uint8_t* row = buf + r * 128;
  const int sw = r & 7;
  if (dt == IA_MASK_F32) {
    const int j = (c & 31) >> 2;
    const float4 v = *reinterpret_cast<const float4*>(buf + (c >> 5) * (kM * 128) + r * 128 +
                                                      ((j ^ sw) << 4));
    out[0] = v.x, out[1] = v.y, out[2] = v.z, out[3] = v.w;
  } else if (dt == IA_MASK_BOOL) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + (((c >> 4) ^ sw) << 4) + (c & 15));
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = ((w >> (8 * e)) & 0xffu) ? 0.f : -INFINITY;
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(row + (((c >> 3) ^ sw) << 4) + (c & 7) * 2);
    if (dt == IA_MASK_BF16) {
      out[0] = __uint_as_float(w.x << 16), out[1] = __uint_as_float(w.x & 0xffff0000u);
      out[2] = __uint_as_float(w.y << 16), out[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
      const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
      const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
      out[0] = lo.x, out[1] = lo.y, out[2] = hi.x, out[3] = hi.y;
    }
  }
}

// The mask values of 16 consecutive keys of one row (bool and 16-bit masks),
// held as raw 16-byte chunks: one load per 16 (bool) or 8 (16-bit) keys instead
// of one per 4, and a quarter-warp's eight rows (r & 7 distinct) read eight
// different bank groups of the swizzled rows. fp32 masks read per 4 keys.
struct RowMask16 {
  uint4 w0, w1;
  __device__ __forceinline__ void load(const uint8_t* buf, int r, int c16, int dt) {
    const uint8_t* row = buf + r * 128;
    const int sw = r & 7;
    if (dt == IA_MASK_BOOL) {
      w0 = *reinterpret_cast<const uint4*>(row + (((c16 >> 4) ^ sw) << 4));
    } else if (dt != IA_MASK_F32) {
      w0 = *reinterpret_cast<const uint4*>(row + (((c16 >> 3) ^ sw) << 4));
      w1 = *reinterpret_cast<const uint4*>(row + ((((c16 >> 3) + 1) ^ sw) << 4));
    }
  }
  // keys c .. c+3 (c a multiple of 4, within the 16 loaded last)
  __device__ __forceinline__ void get4(const uint8_t* buf, int r, int c, int dt, float out[4]) const {
    if (dt == IA_MASK_F32) {
      row_mask4(buf, r, c, dt, out);
    } else if (dt == IA_MASK_BOOL) {
      const int q = (c & 15) >> 2;
      const uint32_t w = q == 0 ? w0.x : q == 1 ? w0.y : q == 2 ? w0.z : w0.w;
#pragma unroll
      for (int e = 0; e < 4; ++e) out[e] = ((w >> (8 * e)) & 0xffu) ? 0.f : -INFINITY;
    } else {
      const uint4 v = (c & 8) ? w1 : w0;
      const uint32_t x = (c & 4) ? v.z : v.x, y = (c & 4) ? v.w : v.y;
      if (dt == IA_MASK_BF16) {
        out[0] = __uint_as_float(x << 16), out[1] = __uint_as_float(x & 0xffff0000u);
        out[2] = __uint_as_float(y << 16), out[3] = __uint_as_float(y & 0xffff0000u);
      } else {
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&y));
        out[0] = lo.x, out[1] = lo.y, out[2] = hi.x, out[3] = hi.y;
      }
    }
  }
};

// RMSNorm + RoPE of one raw 16-bit Q row in shared memory, in place, before
// the fused quantization ("Feature Request: Direct int8 Q/K passthrough
// between Comfy Kitchen and SageAttention", maintainer's reply: rms_rope /
// apply_rope / rms_rope_split_half run on the 16-bit rows before attention):
// ss = fp32 sum of squares (each 8-channel chunk in index order, then the D/8
// chunk sums added pairwise, t with t + n/2), r = 1/sqrt(ss/D + eps),
// y = (x r) w, the rotation a' = ac - bs, b' = as + bc of each channel pair
// with the tables at position `pos`, one rounding to the 16-bit type. The same
// fp32 sequence as the quantize kernel's prologue, so the codes agree bit for
// bit with ia_quantize_qk_prologue. Chunks are visited from chunk r on, which
// spreads a warp's 32 rows over the shared-memory banks.
template <int D, bool BF16>
__device__ __noinline__ void q_prologue_row(uint8_t* row, int r, int64_t pos, const Params& a) {
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  const bool split = a.qp_rope == IA_ROPE_SPLIT_HALF;
  float rf = 1.f;
  if (a.qp_w != nullptr) {
    float part[CPR];
    for (int c = 0; c < CPR; ++c) {
      const int cc = (c + r) & (CPR - 1);
      const uint4 w = *reinterpret_cast<const uint4*>(row + cc * 16);
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_16x2<BF16>(in[e]);
        sum = e == 0 ? __fmul_rn(f.x, f.x) : __fadd_rn(sum, __fmul_rn(f.x, f.x));
        sum = __fadd_rn(sum, __fmul_rn(f.y, f.y));
      }
      part[cc] = sum;
    }
#pragma unroll
    for (int n = CPR; n > 1; n >>= 1)
#pragma unroll
      for (int t = 0; t < n / 2; ++t) part[t] = __fadd_rn(part[t], part[t + n / 2]);
    rf = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(part[0], static_cast<float>(D)), a.qp_eps)));
  }
  const float* cs = a.qp_cos + pos * a.qp_stride;
  const float* sn = a.qp_sin + pos * a.qp_stride;
  const int NU = split ? CPR / 2 : CPR;  // a chunk, or a chunk and its partner half
  for (int c = 0; c < NU; ++c) {
    const int u = (c + r) & (NU - 1);
    const int ch[2] = {u, u + CPR / 2};
    float y[2][8];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      if (hlf == 1 && !split) break;
      const uint4 w = *reinterpret_cast<const uint4*>(row + ch[hlf] * 16);
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_16x2<BF16>(in[e]);
        y[hlf][2 * e] = f.x, y[hlf][2 * e + 1] = f.y;
      }
      if (a.qp_w != nullptr) {
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.qp_w + ch[hlf] * 8));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.qp_w + ch[hlf] * 8 + 4));
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) y[hlf][i] = __fmul_rn(__fmul_rn(y[hlf][i], rf), wv[i]);
      }
    }
    if (a.qp_rope == IA_ROPE_INTERLEAVED) {  // pairs (2i, 2i+1): i = 4u .. 4u+3
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(cs + u * 4));
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(sn + u * 4));
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = y[0][2 * j], x1 = y[0][2 * j + 1];
        y[0][2 * j] = __fsub_rn(__fmul_rn(x0, cv[j]), __fmul_rn(x1, sv[j]));
        y[0][2 * j + 1] = __fadd_rn(__fmul_rn(x0, sv[j]), __fmul_rn(x1, cv[j]));
      }
    } else if (split) {  // pairs (i, i + D/2): i = 8u .. 8u+7
      const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs + u * 8));
      const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + u * 8 + 4));
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(sn + u * 8));
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(sn + u * 8 + 4));
      const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x0 = y[0][i], x1 = y[1][i];
        y[0][i] = __fsub_rn(__fmul_rn(x0, cv[i]), __fmul_rn(x1, sv[i]));
        y[1][i] = __fadd_rn(__fmul_rn(x0, sv[i]), __fmul_rn(x1, cv[i]));
      }
    }
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      if (hlf == 1 && !split) break;
      uint32_t hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (BF16) hv[e] = cvt_bf16x2(y[hlf][2 * e], y[hlf][2 * e + 1]);
        else hv[e] = cvt_f16x2(y[hlf][2 * e], y[hlf][2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(row + ch[hlf] * 16) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// PAIR: the grid's CTAs run as clusters of two along x. Each CTA owns its
// QS x 128 query rows; the pair walks the same key tiles, each CTA loading
// and widening half of every K tile and half of V's columns, and the
// even-ranked CTA issues 256-row MMAs over both (cta_group::2).
// KB: per-64-key-block K scales in the dense head-dim-64 kernel, folded into one
// constant per block and row (see the softmax).
// SEGM: the balanced-segment form (Params::seg_units), a separate
// instantiation so that the one-range form keeps its own register allocation.
template <int D, int QS, int BN, bool SPARSE, bool VBF16, bool QRAW, bool ROWMASK, bool PAIR,
          bool KB = false, bool SEGM = false>
__global__ void __launch_bounds__(32 * (4 * QS + 4), SPARSE ? 2 : 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_m, const Params a) {
  using L = Layout<D, QS, BN, SPARSE, ROWMASK, PAIR, KB>;
  constexpr bool SEG = SEGM;
  // dense single-CTA head-dim-64 kernels with int8 Q and per-token K scales: the
  // softmax threads widen their own Q rows (each a row), so the converters start
  // on K at once (with per-block scales the softmax is the lighter side and this
  // measured slower)
  constexpr bool QSOFT = L::SEGOK && !QRAW && !KB;
  static_assert(!SEGM || (L::SEGOK && !QRAW), "segments: dense single-CTA head-dim-64, int8 Q");
  // Where Q lands before it is widened or quantized: the V buffers, or (16-bit Q
  // rows of two stages with a per-row mask, 64 KB at head dim 128) the mask ring,
  // whose first tiles are copied only once Q has been quantized
  constexpr bool Q_IN_MK = QRAW && ROWMASK && QS == 2;
  constexpr int OFF_QIN = Q_IN_MK ? L::OFF_MK : L::OFF_QIN;
  static_assert(PAIR || !QRAW || QS * L::QR * 2 <= (Q_IN_MK ? L::NSC * L::MB : L::NVS * L::VB),
                "16-bit Q fits its staging area");
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if ((smem_u32(smem) & 1023u) != 0) {  // swizzled operands need 1024-byte alignment
    if (tid == 0) atomicOr(&g_attn_status, kErrSmemAlign);
    return;
  }
  if (tid == 0) IA_TRACE_POINT(14, 0);  // events of CTA 0 in slot 14 (profiling build only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const Ctl ctl{abort_flag, a.timeout_ns};
  auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };
  // Pair roles: the leader (even rank) issues the MMAs; the peer's threads
  // arrive on the leader's barriers through these addresses.
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0u;
  auto lbar = [&](int i) -> uint32_t { return mapa_shared(bar(i), crank & ~1u); };
  // arrivals the leader's MMA barriers take from the peer (one per peer warp
  // for K and P; one forwarded arrival for Q and V)
  const uint32_t peer_k = (PAIR && leader) ? 2u : 0u;
  const uint32_t peer_p = (PAIR && leader) ? 4u : 0u;
  const uint32_t peer_f = (PAIR && leader) ? 1u : 0u;

  // Work of this CTA: one query tile and key range, or (a.seg_units > 0, dense
  // single-CTA head-dim-64 kernels) an equal share of all (query tile, key
  // tile) units: the contiguous run [x U / C, (x+1) U / C) of the units ordered
  // by query tile, then key tile, cut into segments at query-tile boundaries.
  // A segment that starts a query tile's keys writes partial 0, one that ends
  // them partial 1 (a share of at least n_tiles units meets each query tile
  // at most twice); one that covers all of them writes partial 0 and marks
  // partial 1 empty. The body below runs once per segment; TMEM stays
  // allocated, the barriers are initialised again.
  // (a trip count of one for the kernels without segments: no loop is left there)
  for (int seg = 0; seg < (SEG ? INT_MAX : 1); ++seg) {
    // segment seg: key tiles [seg_k0, seg_k1) of one query tile
    int seg_b = 0, seg_h = 0, seg_q0 = 0, seg_k0 = 0, seg_k1 = 0;
    if constexpr (SEG) {
      if (a.seg_units > 0) {
        // it starts at this CTA's first unit, then at each following query
        // tile's first key tile (recomputed, not carried across segments)
        const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.seg_units / gridDim.x;
        const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.seg_units / gridDim.x;
        const int64_t us = seg == 0 ? u0 : (u0 / a.n_tiles + seg) * a.n_tiles;
        if (us >= u1) break;
        const int64_t qt = us / a.n_tiles;
        seg_k0 = static_cast<int>(us - qt * a.n_tiles);
        seg_k1 = static_cast<int>(min(static_cast<int64_t>(a.n_tiles), seg_k0 + (u1 - us)));
        const int bh = static_cast<int>(qt / a.seg_nqt);
        seg_q0 = static_cast<int>(qt % a.seg_nqt) * (kM * QS);
        seg_h = bh % a.H;
        seg_b = bh / a.H;
      } else if (seg > 0) {
        break;
      }
    }
    const bool segd = SEG && a.seg_units > 0;
    const int h = segd ? seg_h : static_cast<int>(blockIdx.y);
    const int b = segd ? seg_b : static_cast<int>(blockIdx.z) / a.nsplit;
    const int split = segd ? (seg_k0 == 0 ? 0 : 1) : static_cast<int>(blockIdx.z) % a.nsplit;
    const int q0 = segd ? seg_q0 : static_cast<int>(blockIdx.x) * (kM * QS);
    const bool seg_full = segd && seg_k0 == 0 && seg_k1 == a.n_tiles;
    if (seg > 0) {
      // every role has finished the last segment: its copies landed, its
      // MMAs completed (the issuer's drain), its barriers have no waiter
      tc_fence_before();
      __syncthreads();
      if (*abort_flag) break;
    }
    // The barriers are (invalidated after a segment, then) initialised by five
    // threads in five warps, side by side.
    auto binit = [&](int i, uint32_t n) {
      if (seg > 0) mbar_inval(bar(i));
      mbar_init(bar(i), n);
    };
    if (tid == 0) {
      binit(L::B_QFULL, 1);
      binit(L::B_QCONV, ((QRAW || QSOFT) ? QS * kM : 64) + peer_f);
      binit(L::B_PVT, 1);
      binit(L::B_DRAIN, 1);
      binit(L::B_STALL, 1);  // never signalled: the timeout test hook waits on it
      misc[1] = 0;
    } else if (tid == 32) {
      for (int i = 0; i < L::NKS; ++i) {
        binit(L::B_KRF + i, 1);
        binit(L::B_KCF + i, 64 + peer_k);
        binit(L::B_KCE + i, 1);
      }
      for (int i = 0; i < L::NRS; ++i) binit(L::B_KRE + i, 64);
    } else if (tid == 64) {
      for (int i = 0; i < L::NVS; ++i) {
        binit(L::B_VF + i, 1 + peer_f);
        binit(L::B_VE + i, 1);
      }
      for (int i = 0; i < L::NSC; ++i) binit(L::B_MF + i, 1);
    } else if (tid == 96) {
      for (int i = 0; i < L::NSC; ++i) {
        binit(L::B_SCF + i, 64);
        binit(L::B_SCE + i, 4 * QS);
      }
    } else if (tid == 128) {
      for (int s = 0; s < L::NSB; ++s) {
        binit(L::B_SF + s, 1);
        binit(L::B_PF + s, kM + peer_p);
      }
      for (int s = 0; s < QS; ++s) binit(L::B_OF + s, 1);
    }
    if ((tid & 31) == 0 && tid <= 128) fence_mbar_init();
    if (seg == 0 && warp == L::W_MMA) {  // TMEM stays allocated for every segment
      if constexpr (PAIR) {
        tmem_alloc_pair(smem_u32(misc), L::TMEM_COLS);
        tmem_relinquish_pair();
      } else {
        tmem_alloc(smem_u32(misc), L::TMEM_COLS);
        tmem_relinquish();
      }
    }
    float* vsc = reinterpret_cast<float*>(smem + L::OFF_VS);
    for (int i = tid; i < D; i += blockDim.x) vsc[i] = a.v_scale ? __ldg(a.v_scale + h * D + i) : 1.f;
    if constexpr (L::ONES) {  // the row-sum columns of V: 1.0 in V's type
      const uint32_t one2 = VBF16 ? 0x3F803F80u : 0x3C003C00u;
      uint4* ones = reinterpret_cast<uint4*>(smem + L::OFF_ONES);
      for (int i = tid; i < L::NVS * L::VB / 16; i += blockDim.x) ones[i] = make_uint4(one2, one2, one2, one2);
      fence_proxy_async_smem();
    }

    // Key tiles this CTA visits: all of them (dense) or the union of the kept
    // tiles of its two 64-row query tiles, in ascending order (block-sparse).
    uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::OFF_LIST);
    int n_it, it0;
    const int qt0 = q0 / 64;
    const int qt1 = qt0 + 1;
    if constexpr (SPARSE) {
      const uint8_t* m0 = a.mask + (static_cast<int64_t>(b * a.H + h) * a.Tq + qt0) * a.Tk;
      const uint8_t* m1 = qt1 < a.Tq ? m0 + a.Tk : nullptr;
      int* wcnt = reinterpret_cast<int*>(smem + L::OFF_MISC + 16);
      int total = 0;
      const int nw = blockDim.x >> 5;
      for (int base = 0; base < a.Tk; base += blockDim.x) {
        const int t = base + tid;
        const bool keep = t < a.Tk && (m0[t] != 0 || (m1 != nullptr && m1[t] != 0));
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) wcnt[warp] = __popc(bal);
        __syncthreads();
        int before = total;
        for (int w = 0; w < warp; ++w) before += wcnt[w];
        if (keep) list[before + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(t);
        for (int w = 0; w < nw; ++w) total += wcnt[w];
        __syncthreads();
      }
      // this CTA's share of the kept-tile list
      const int per = (total + a.nsplit - 1) / a.nsplit;
      it0 = split * per;
      n_it = max(0, min(total - it0, per));
    } else if (SEG && a.seg_units > 0) {
      it0 = seg_k0;
      n_it = seg_k1 - seg_k0;
    } else {
      it0 = split * a.tps;
      n_it = max(0, min(a.n_tiles - it0, a.tps));
    }
    tc_fence_before();
    __syncthreads();
    // a pair's barriers take arrivals from both CTAs: both are initialised first
    if constexpr (PAIR) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    if (tid == 0) IA_TRACE_POINT(14, 1);

    const uint32_t sm_qh = smem_u32(smem + L::OFF_QH);
    const uint32_t sm_kh = smem_u32(smem + L::OFF_KH);
    const uint32_t sm_v = smem_u32(smem + L::OFF_V);
    const uint32_t sm_kr = smem_u32(smem + L::OFF_KR);

    if (warp == L::W_PROD) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (ROWMASK) prefetch_tmap(&tm_m);
        int kr_last[L::NKS], v_last[L::NVS], m_last[L::NSC];
        for (int i = 0; i < L::NKS; ++i) kr_last[i] = -1;
        for (int i = 0; i < L::NVS; ++i) v_last[i] = -1;
        for (int i = 0; i < L::NSC; ++i) m_last[i] = -1;
        // per-row mask boxes: 128-byte rows of 32 fp32, 64 16-bit or 128 bool keys
        const int m_kpb = a.rm_dtype == IA_MASK_F32 ? 32 : a.rm_dtype == IA_MASK_BOOL ? 128 : 64;
        const int m_nbox = a.rm_dtype == IA_MASK_F32 ? 2 : 1;
        const int m_h = a.rm_h ? h : 0, m_b = a.rm_b ? b : 0;
        // int8 Q codes, or 16-bit Q rows that the softmax warps quantize; either
        // way they are staged in the V buffers until converted
        constexpr int QB = QRAW ? 2 : 1;
        const uint32_t sm_qin = smem_u32(smem + OFF_QIN);
        mbar_arrive_expect_tx(bar(L::B_QFULL), QS * kM * D * QB);
        IA_TRACE_POINT(14, 2);
        for (int s = 0; s < QS; ++s)
          tma_load_4d(sm_qin + s * L::QR * QB, &tm_q, bar(L::B_QFULL), 0, q0 + s * kM, h, b);
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
          const int kt = SPARSE ? static_cast<int>(list[it0 + it]) : it0 + it;
          // int8 K tile: into its fp16 buffer (in place) or a staging buffer
          const int ks = it % L::NKS;
          uint32_t kdst;
          if constexpr (L::INPLACE) {
            if (it >= L::NKS) ok = wait_bar(bar(L::B_KCE + ks), ((it / L::NKS) - 1) & 1, ctl, kErrProducer);
            kdst = sm_kh + ks * L::KH + BN * 128;
          } else {
            const int rs = it % L::NRS;
            if (it >= L::NRS) ok = wait_bar(bar(L::B_KRE + rs), ((it / L::NRS) - 1) & 1, ctl, kErrProducer);
            kdst = sm_kr + rs * L::KR;
          }
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::B_KRF + ks), L::KROWS * D);
          tma_load_4d(kdst, &tm_k, bar(L::B_KRF + ks), 0, kt * BN + static_cast<int>(crank) * L::KROWS, h, b);
          kr_last[ks] = it;
          const int vs = it % L::NVS;
          // Q sits in V buffer 0, or in all of them (16-bit Q, or int8 Q of two
          // stages larger than one V buffer) until it has been widened
          constexpr bool Q_ALL_V = QRAW || QS * L::QR > L::VB;
          if (!PAIR && !Q_IN_MK && (it == 0 || (Q_ALL_V && it < L::NVS)))
            ok = wait_bar(bar(L::B_QCONV), 0, ctl, kErrProducer);
          else if (it >= L::NVS)
            ok = wait_bar(bar(L::B_VE + vs), ((it / L::NVS) - 1) & 1, ctl, kErrProducer);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::B_VF + vs), BN * L::VCOLS * 2);
  #pragma unroll
          for (int c = 0; c < L::VCOLS / 64; ++c)
            tma_load_4d(sm_v + vs * L::VB + c * BN * 128, &tm_v, bar(L::B_VF + vs),
                        static_cast<int>(crank) * L::VCOLS + c * 64, kt * BN, h, b);
          v_last[vs] = it;
          if constexpr (ROWMASK) {  // the tile's mask rows, released with the tile's k scales
            // boxes of stage s at (s * m_nbox + x) * kM * 128 (two stages: one box each)
            const int ms = it % L::NSC;
            if (Q_IN_MK && it < L::NSC)  // the ring still holds the 16-bit Q rows
              ok = wait_bar(bar(L::B_QCONV), 0, ctl, kErrProducer);
            else if (it >= L::NSC)
              ok = wait_bar(bar(L::B_SCE + ms), ((it / L::NSC) - 1) & 1, ctl, kErrProducer);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(L::B_MF + ms), QS * m_nbox * kM * 128);
            for (int s = 0; s < QS; ++s)
              for (int x = 0; x < m_nbox; ++x)
                tma_load_4d(smem_u32(smem + L::OFF_MK + ms * L::MB + (s * m_nbox + x) * kM * 128), &tm_m,
                            bar(L::B_MF + ms), kt * BN + x * m_kpb, q0 + s * kM, m_h, m_b);
            m_last[ms] = it;
          }
        }
        if (((PAIR && !leader) || SEG) && ok) {
          // The last V-empty commits (in a pair, the leader's, which arrive here
          // too) have no other waiter: take them before this CTA may exit or
          // its barriers are initialised for the next segment.
          for (int t = max(0, n_it - L::NVS); t < n_it - 1; ++t)
            drain_bar(bar(L::B_VE + t % L::NVS), (t / L::NVS) & 1, a.timeout_ns);
        }
        if (!ok) {  // let issued copies land before the CTA's shared memory goes away
          drain_bar(bar(L::B_QFULL), 0, a.timeout_ns);
          for (int i = 0; i < L::NKS; ++i)
            if (kr_last[i] >= 0) drain_bar(bar(L::B_KRF + i), (kr_last[i] / L::NKS) & 1, a.timeout_ns);
          for (int i = 0; i < L::NVS; ++i)
            if (v_last[i] >= 0) drain_bar(bar(L::B_VF + i), (v_last[i] / L::NVS) & 1, a.timeout_ns);
          for (int i = 0; i < L::NSC; ++i)
            if (m_last[i] >= 0) drain_bar(bar(L::B_MF + i), (m_last[i] / L::NSC) & 1, a.timeout_ns);
        }
      }
    } else if (warp == L::W_MMA) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && PAIR && !leader) {
        // The peer issues no MMA: its lane forwards the completion of its Q
        // conversion and of each V tile's copy to the leader's barriers.
        bool ok = wait_bar(bar(L::B_QCONV), 0, ctl, kErrMma);
        if (ok) mbar_arrive_remote(lbar(L::B_QCONV));
        for (int it = 0; it < n_it && ok; ++it) {
          const int vs = it % L::NVS;
          ok = wait_bar(bar(L::B_VF + vs), (it / L::NVS) & 1, ctl, kErrMma);
          if (ok) mbar_arrive_remote(lbar(L::B_VF + vs));
        }
        // The leader's last commit reaches this CTA too, after every earlier
        // one (and after all of the pair's MMAs, which read this CTA's shared
        // memory and TMEM): wait for it before this CTA may leave, on the
        // normal path and after an abort alike.
        drain_bar(bar(L::B_DRAIN), 0, a.timeout_ns);
      } else if (lane == 0) {
        constexpr int MM = PAIR ? 2 * kM : kM;  // rows of one MMA
        constexpr uint32_t idq = idesc_f16(MM, BN, 0, 0, 0, 0);                  // f16 x f16, K-major
        constexpr uint32_t idv = idesc_f16(MM, L::OW, VBF16 ? 1 : 0, VBF16 ? 1 : 0, 0, 1);  // V MN-major
        // Descriptors are built once; a k-step or buffer offset is added to the
        // 14-bit start-address field (16-byte units), which cannot overflow for
        // addresses inside the CTA's shared memory. This keeps the issuing
        // thread to a few instructions per MMA.
        const uint64_t qdesc = sdesc_sw128(sm_qh, 16, 1024);
        const uint64_t kdesc = sdesc_sw128(sm_kh, 16, 1024);
        // V's 64-column blocks are BN*128 bytes apart; the ones block sits at the
        // same distance from every V buffer
        const uint64_t vdesc = sdesc_sw128(sm_v, L::ONES ? L::OFF_ONES - L::OFF_V : BN * 128, 1024);
        // a barrier that also counts the peer's arrivals
        auto wait_in = [&](int i, uint32_t parity) { return wait_bar(bar(i), parity, ctl, kErrMma); };
        auto commit = [&](int i) {
          if constexpr (PAIR) mma_commit_pair(bar(i), 3);
          else mma_commit(bar(i));
        };
        // S buffer sb <- Q_s K^T (K from stage kst)
        auto issue_qk = [&](int s, int kst, int sb) {
          const uint64_t qa = qdesc + static_cast<uint64_t>((s * L::QH) >> 4);
          const uint64_t kb = kdesc + static_cast<uint64_t>((kst * L::KH) >> 4);
          const uint32_t dt = tmem + sb * BN;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = qa + static_cast<uint64_t>(((kk >> 2) * (kM * 128) + (kk & 3) * 32) >> 4);
            const uint64_t bd = kb + static_cast<uint64_t>(((kk >> 2) * (L::KROWS * 128) + (kk & 3) * 32) >> 4);
            if constexpr (PAIR) mma_ss_pair(dt, ad, bd, idq, kk > 0 ? 1u : 0u);
            else mma_ss(dt, ad, bd, idq, kk > 0 ? 1u : 0u);
          }
        };
        // O_s += P V (P from S buffer sb, V from stage vs)
        auto issue_pv = [&](int s, int vs, bool first, int sb) {
          const uint64_t vb = vdesc + static_cast<uint64_t>((vs * L::VB) >> 4);
          const uint32_t dt = tmem + L::NSB * BN + s * L::OW;
          const uint32_t pt = tmem + sb * BN;
  #pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = vb + static_cast<uint64_t>((kk * 16 * 128) >> 4);
            if constexpr (PAIR) mma_ts_pair(dt, pt + kk * 8, bd, idv, (first && kk == 0) ? 0u : 1u);
            else mma_ts(dt, pt + kk * 8, bd, idv, (first && kk == 0) ? 0u : 1u);
          }
        };
        bool ok = wait_in(L::B_QCONV, 0);
        IA_TRACE_POINT(14, 5);
        if (ok && a.debug_stall) ok = wait_bar(bar(L::B_STALL), 0, ctl, kErrMma);
        tc_fence_after();
        if constexpr (L::DBS) {
          // QK^T of tiles 0 and 1, then per tile j: P_j V_j, and the QK^T of
          // tile j+2 into the S buffer that P_j V_j has just read
          auto qk_step = [&](int j) -> bool {
            const int kst = j % L::NKS;
            if (!wait_in(L::B_KCF + kst, (j / L::NKS) & 1)) return false;
            tc_fence_after();
            issue_qk(0, kst, j & 1);
            commit(L::B_SF + (j & 1));
            commit(L::B_KCE + kst);
            return true;
          };
          for (int j = 0; j < 2 && j < n_it && ok; ++j) ok = qk_step(j);
          for (int it = 0; it < n_it && ok; ++it) {
            const int vs = it % L::NVS;
            ok = wait_in(L::B_VF + vs, (it / L::NVS) & 1);
            if (ok) ok = wait_bar(bar(L::B_PF + (it & 1)), (it >> 1) & 1, ctl, kErrMma);
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, vs, it == 0, it & 1);
            commit(L::B_PVT);  // one phase per tile
            commit(L::B_VE + vs);
            if (it + 2 < n_it) ok = qk_step(it + 2);
          }
          if (ok && n_it > 0) commit(L::B_OF);  // after the last P V: the epilogue's one phase
        }
        for (int it = 0; it < n_it && ok && !L::DBS; ++it) {
          const int kst = it % L::NKS;
          IA_TRACE_POINT(8, it);
          ok = wait_in(L::B_KCF + kst, (it / L::NKS) & 1);
          if (!ok) break;
          IA_TRACE_POINT(9, it);
          tc_fence_after();
          const int pvs = (it + L::NVS - 1) % L::NVS;
          if (it > 0) {
            ok = wait_in(L::B_VF + pvs, ((it - 1) / L::NVS) & 1);
            if (!ok) break;
            tc_fence_after();
          }
          for (int s = 0; s < QS && ok; ++s) {
            if (it > 0) {
              ok = wait_bar(bar(L::B_PF + s), (it - 1) & 1, ctl, kErrMma);
              if (!ok) break;
              tc_fence_after();
              issue_pv(s, pvs, it == 1, s);
            }
            issue_qk(s, kst, s);
            commit(L::B_SF + s);
            IA_TRACE_POINT(10 + s, it);
          }
          if (!ok) break;
          commit(L::B_KCE + kst);
          if (it > 0) commit(L::B_VE + pvs);
        }
        if (ok && n_it > 0 && !L::DBS) {
          const int pvs = (n_it - 1) % L::NVS;
          ok = wait_in(L::B_VF + pvs, ((n_it - 1) / L::NVS) & 1);
          if (ok) tc_fence_after();
          for (int s = 0; s < QS && ok; ++s) {
            ok = wait_bar(bar(L::B_PF + s), (n_it - 1) & 1, ctl, kErrMma);
            if (!ok) break;
            tc_fence_after();
            issue_pv(s, pvs, n_it == 1, s);
            commit(L::B_OF + s);
          }
        }
        // every MMA issued above has completed once this arrives (in both CTAs
        // of a pair: the peer waits for it before it exits)
        IA_TRACE_POINT(14, 7);
        if constexpr (PAIR) mma_commit_pair(bar(L::B_DRAIN), 3);
        else mma_commit(bar(L::B_DRAIN));
        drain_bar(bar(L::B_DRAIN), 0, a.timeout_ns);
      }
    } else if (warp >= L::W_CONV) {
      // ---------------------------------------------- int8 -> fp16 converters
      const int ct = tid - L::W_CONV * 32;
      bool ok = (QRAW || QSOFT) ? true : wait_bar(bar(L::B_QFULL), 0, ctl, kErrConverter);
      if constexpr (PAIR) ok = __all_sync(0xffffffffu, ok);
      if (ct == 0) IA_TRACE_POINT(14, 3);
      if (ok && !QRAW && !QSOFT) {
        for (int s = 0; s < QS; ++s)
          widen_tile<D, kM, false>(smem + OFF_QIN + s * L::QR, smem + L::OFF_QH + s * L::QH, ct);
        fence_proxy_async_smem();
        mbar_arrive(bar(L::B_QCONV));
        if (ct == 0) IA_TRACE_POINT(14, 4);
      }
      const uint8_t* mrow0 = nullptr;
      const uint8_t* mrow1 = nullptr;
      if (SPARSE) {
        mrow0 = a.mask + (static_cast<int64_t>(b * a.H + h) * a.Tq + qt0) * a.Tk;
        mrow1 = qt1 < a.Tq ? mrow0 + a.Tk : nullptr;
      }
      const float* ksb = a.k_scale + b * a.ks_sb + h * a.ks_sh;
      const void* brow = nullptr;  // this (b, h)'s row of per-key offsets
      if (a.bias != nullptr) {
        const int es = a.bias_dtype == IA_MASK_F32 ? 4 : a.bias_dtype == IA_MASK_BOOL ? 1 : 2;
        brow = static_cast<const char*>(a.bias) + (b * a.bias_sb + h * a.bias_sh) * es;
      }
      for (int it = 0; it < n_it && ok; ++it) {
        const int kt = SPARSE ? static_cast<int>(list[it0 + it]) : it0 + it;
        // Per-key constants of this tile: the global loads are issued first and
        // land while the K tile is widened.
        constexpr int KPT = (BN + 63) / 64;  // keys per converter thread
        float kv[KPT];
        uint32_t braw[KPT];
        bool kval[KPT];
  #pragma unroll
        for (int e = 0; e < KPT; ++e) {
          const int key = kt * BN + ct + 64 * e;
          kval[e] = key < a.Sk && (a.kv_valid == nullptr || (key & 63) < __ldg(a.kv_valid + (key >> 6)));
          kv[e] = kval[e] ? __ldg(ksb + (a.gran_block ? (key >> 6) : key)) : 0.f;
          braw[e] = (kval[e] && brow != nullptr) ? key_bias_bits(brow, key, a.bias_dtype) : 0u;
        }
        // K tile: int8 -> fp16 codes in the swizzled layout the MMA reads
        const int kst = it % L::NKS;
        ok = wait_bar(bar(L::B_KRF + kst), (it / L::NKS) & 1, ctl, kErrConverter);
        if constexpr (PAIR) ok = __all_sync(0xffffffffu, ok);  // warps stay converged
        if (!ok) break;
        if (ct == 0) IA_TRACE_POINT(12, it);
        if constexpr (L::INPLACE) {
          uint8_t* kh = smem + L::OFF_KH + kst * L::KH;
          widen_tile<D, BN, true>(kh + BN * 128, kh, ct);
        } else {
          const int rs = it % L::NRS;
          if (it >= L::NKS) ok = wait_bar(bar(L::B_KCE + kst), ((it / L::NKS) - 1) & 1, ctl, kErrConverter);
          if constexpr (PAIR) ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          widen_tile<D, L::KROWS, false>(smem + L::OFF_KR + rs * L::KR, smem + L::OFF_KH + kst * L::KH, ct);
          mbar_arrive(bar(L::B_KRE + rs));
        }
        if (ct == 0) IA_TRACE_POINT(13, it);
        fence_proxy_async_smem();
        if (PAIR && !leader) {  // the leader's MMA reads this half: one arrival per warp
          __syncwarp();
          if ((ct & 31) == 0) mbar_arrive_remote(lbar(L::B_KCF + kst));
        } else {
          mbar_arrive(bar(L::B_KCF + kst));
        }
        // k scales, bias * log2(e) (-inf past the valid keys) and tile flags
        const int ss = it % L::NSC;
        if (it >= L::NSC) ok = wait_bar(bar(L::B_SCE + ss), ((it / L::NSC) - 1) & 1, ctl, kErrConverter);
        if constexpr (PAIR) ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        float* ksm = reinterpret_cast<float*>(smem + L::OFF_SC + ss * L::SC);
        float* b2m = ksm + BN;
        uint32_t* flg = reinterpret_cast<uint32_t*>(b2m + BN);
        bool nonzero = false;  // a valid key of this thread has a nonzero offset
  #pragma unroll
        for (int e = 0; e < KPT; ++e) {
          if (ct + 64 * e < BN) {
            const float off =
                kval[e] ? (brow ? key_bias_value(braw[e], a.bias_dtype) * kLog2e : 0.f) : -INFINITY;
            ksm[ct + 64 * e] = kv[e];
            b2m[ct + 64 * e] = off;
            nonzero |= kval[e] && off != 0.f;
          }
        }
        // Each converter warp records whether its keys carry any offset: a tile
        // whose offsets are all zero (e.g. the core of a window's bias) keeps the
        // softmax's fast path. Separate words, so the warps need no barrier.
        {
          const bool any_nz = __any_sync(__activemask(), nonzero);
          if ((ct & 31) == 0) flg[1 + (ct >> 5)] = any_nz ? 1u : 0u;
        }
        if (ct == 0) {
          bool partial = kt * BN + BN > a.Sk;
          if (a.kv_valid)
            for (int t = (kt * BN) >> 6; t < ((kt + 1) * BN) >> 6 && t * 64 < a.Sk; ++t)
              partial |= __ldg(a.kv_valid + t) < 64;
          uint32_t f = (ROWMASK || partial) ? 1u : 0u;
          if (SPARSE) {
            const uint32_t k0 = mrow0[kt] ? 1u : 0u;
            const uint32_t k1 = (mrow1 != nullptr && mrow1[kt]) ? 1u : 0u;
            f |= (k0 << 1) | (k1 << 2);
          } else {
            f |= 6u;
          }
          *flg = f;
        }
        mbar_arrive(bar(L::B_SCF + ss));
      }
      if (((PAIR && !leader) || SEG) && ok) {
        // the last K-empty commits (in a pair, the leader's) have no other
        // waiter: take them before exit or the next segment's initialisation
        for (int t = max(0, n_it - L::NKS); t < n_it; ++t)
          drain_bar(bar(L::B_KCE + t % L::NKS), (t / L::NKS) & 1, a.timeout_ns);
      }
    } else {
      // ------------------------------------------------------------- softmax
      const int s = warp >> 2;
      const int r = tid & (kM - 1);
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tS0 = tmem + s * BN + lane_off;
      const uint32_t tO = tmem + L::NSB * BN + s * L::OW + lane_off;
      const int row = q0 + s * kM + r;
      const bool row_ok = row < a.Sq;
      float cq = 0.f;
      bool ok = true;
      if constexpr (QRAW) {
        // This thread quantizes its own row (per 64-row block: each of the
        // block's two warps also scans the other warp's rows; without the
        // prologue those rows are not modified, so no barrier is needed).
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_QFULL), 0, ctl, kErrSoftmax));
        uint8_t* raw = smem + OFF_QIN + static_cast<size_t>(s * kM) * D * 2;
        auto quantized = [&](int rr) {  // row rr of this stage: real and not padding
          const int gr = q0 + s * kM + rr;
          return gr < a.Sq && !(a.pad_query && (gr & 63) >= __ldg(a.kv_valid + (gr >> 6)));
        };
        if (a.q_pro) {  // RMSNorm + RoPE of the thread's own row, in place
          if (ok && quantized(r))
            q_prologue_row<D, VBF16>(raw + r * D * 2, r, static_cast<int64_t>(a.qp_pos0) + q0 + s * kM + r, a);
          // a 64-row block's two warps read each other's rows below: both warps
          // always reach this barrier (its condition is uniform over the CTA)
          if (a.gran_block) named_bar_sync(1 + (warp >> 1), 64);
        }
        if (ok) {
          const bool keep = quantized(r);
          uint32_t am = keep ? row_amax_bits<D>(raw + r * D * 2, r) : 0u;
          if (a.gran_block) {
            const int rp = r ^ 32;
            if (quantized(rp)) am = max(am, row_amax_bits<D>(raw + rp * D * 2, r));
            am = __reduce_max_sync(0xffffffffu, am);
          }
          const float amax = half_bits_to_float<VBF16>(am);
          const float scale = __fdiv_rn(amax, 127.0f);
          const float inv = (keep && amax > 0.f) ? __fdiv_rn(127.0f, amax) : 0.f;
          write_q_codes<D, VBF16>(raw + r * D * 2, smem + L::OFF_QH + s * L::QH, r, inv);
          cq = scale * a.cq_mult;
          fence_proxy_async_smem();
          mbar_arrive(bar(L::B_QCONV));
        }
      } else {
        if constexpr (QSOFT) {  // this thread widens its own Q row
          ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_QFULL), 0, ctl, kErrSoftmax));
          if (ok) {
            widen_row<D>(smem + OFF_QIN + s * L::QR + r * D, smem + L::OFF_QH + s * L::QH, r);
            fence_proxy_async_smem();
            mbar_arrive(bar(L::B_QCONV));
          }
        }
        if (row_ok)
          cq = __ldg(a.q_scale + b * a.qs_sb + h * a.qs_sh + (a.gran_block ? (row >> 6) : row)) * a.cq_mult;
      }
      const int half = (r >= 64) ? 1 : 0;
      // O *= alpha over all of this stage's O columns (with ONES, the row sum too)
      auto rescale_o = [&](float alpha) {
  #pragma unroll 1
        for (int c0 = 0; c0 + 32 <= L::OW; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tO + c0, rr);
          tmem_wait_ld(rr);
  #pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tO + c0, rr);
        }
        if constexpr (L::OW % 32 != 0) {
          uint32_t rr[16];
          tmem_ld16(tO + (L::OW & ~31), rr);
          tmem_wait_ld(rr);
  #pragma unroll
          for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st16(tO + (L::OW & ~31), rr);
        }
      };
      // p = 2^t for two logits, packed to the 16-bit type of V. Without ONES the
      // fp32 p are also added to the row sum `acc`; with ONES the MMA sums the
      // 16-bit P it multiplies.
      auto p_pack = [&](float t0, float t1, uint64_t& acc) -> uint32_t {
        const float p0 = ex2(t0), p1 = ex2(t1);
        if constexpr (!L::ONES) acc = fadd2(acc, pack2(p0, p1));
        return VBF16 ? cvt_bf16x2(p0, p1) : cvt_f16x2(p0, p1);
      };
      float m = -INFINITY;  // reference maximum (log2 units) that P is relative to
      float m_pend = -INFINITY;  // one-pass tiles: the reference the next tile takes
      float l = 0.f;
      // One query stage: O is rescaled only once the previous tile's P V has
      // completed (B_PVT, one phase per tile). That wait cannot alias: when this
      // tile's S is ready, the P V two tiles back has completed, so B_PVT is at
      // most one phase behind the phase waited for. The epilogue instead waits
      // on B_OF, committed once after the last P V: a parity wait on B_PVT there
      // could find the barrier two phases behind (the last two P Vs in flight)
      // and pass before O is complete. A wait that runs out (voted across the
      // warp) clears `ok`, which ends the loop after this tile.
      for (int it = 0; it < n_it && ok; ++it) {
        const int ss = it % L::NSC;
        if (r == 0) IA_TRACE_POINT(4 * s, it);
        // this tile's S buffer (alternating with one query stage)
        const int sb = L::DBS ? (it & 1) : s;
        const uint32_t tS = L::DBS ? tS0 + sb * BN : tS0;
        bool w = wait_bar(bar(L::B_SF + sb), L::DBS ? (it >> 1) & 1 : it & 1, ctl, kErrSoftmax);
        w = w && wait_bar(bar(L::B_SCF + ss), (it / L::NSC) & 1, ctl, kErrSoftmax);
        if (ROWMASK) w = w && wait_bar(bar(L::B_MF + ss), (it / L::NSC) & 1, ctl, kErrSoftmax);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (r == 0) IA_TRACE_POINT(1 + 4 * s, it);
        const float* ksm = reinterpret_cast<const float*>(smem + L::OFF_SC + ss * L::SC);
        const float* b2m = ksm + BN;
        const volatile uint32_t* fw = reinterpret_cast<const volatile uint32_t*>(b2m + BN);
        const uint32_t flags = fw[0];
        // the masked path is needed for a partial tile, a per-row mask or a
        // nonzero per-key offset in either converter warp's keys
        const bool fast = ((flags & 1u) | fw[1] | fw[2]) == 0;
        const bool keep = SPARSE ? ((flags >> (1 + half)) & 1u) != 0 : true;
        const uint64_t cq2 = pack2(cq, cq);
        // KB: each 64-key half of the tile has one k scale; s * k * cq becomes
        // s * (k * cq), one constant per half and row, so the logits take one
        // packed FMA and no per-key scale loads.
        float cb0 = 0.f, cb1 = 0.f;
        if constexpr (KB) {
          cb0 = ksm[0] * cq;
          cb1 = ksm[64] * cq;
        }
        if (SPARSE && !keep) {
          // This row's query tile dropped the key tile: P = 0, the row's maximum
          // and sum stay as they are, and S need not be read.
          uint32_t z[BN / 2];
  #pragma unroll
          for (int e = 0; e < BN / 2; ++e) z[e] = 0u;
          if constexpr (BN == 128) {
            tmem_st64(tS, z);
          } else {
            tmem_st32(tS, z);
          }
        } else {
          // The whole S row of this thread in one TMEM round trip.
          uint32_t sv[BN];
          if constexpr (BN == 128) {
            tmem_ld128(tS, sv);
          } else {
            tmem_ld64(tS, sv);
          }
          tmem_wait_ld(sv);
          if (r == 0) IA_TRACE_POINT(2 + 4 * s, it);
          uint64_t lsum[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
          RowMask16 rmk;  // ROWMASK: the current 16 keys' mask words
          // One pass (two query stages, a reference already set): P is taken
          // relative to the reference the previous tiles set (P may exceed 1: up to
          // 2^64 in bf16, 2^15 in fp16), the tile's maximum is taken in the same
          // pass, and a reference that grew by more than 2^8 is applied at the
          // start of the next tile (O and l rescaled there, before this stage's
          // next P V; that stage's previous P V has completed by then). This
          // saves the separate pass over the row for its maximum. A row whose
          // maximum exceeds the reference by more than that bound redoes the tile
          // in two passes from S, still in TMEM.
          constexpr bool OP = !L::DBS;
          // fp16 P holds values below 2^16, bf16 P those below 2^128
          constexpr float kRedo = VBF16 ? 64.f : 15.f;
          bool one = false;
          if constexpr (OP) {
            if (__any_sync(0xffffffffu, m_pend > m)) {  // the reference grew on the last tile
              const float alpha = m_pend > m ? ex2(m - m_pend) : 1.f;
              rescale_o(alpha);
              l *= alpha;
              m = fmaxf(m, m_pend);
            }
            one = __all_sync(0xffffffffu, m > -INFINITY);
            if (one) {
              const uint64_t cq2o = pack2(cq, cq);
              const uint64_t nmo = pack2(-m, -m);
              float mo[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
              if (!fast) {  // t = acc k cq + offset (log2 units; -inf for invalid keys)
    #pragma unroll
                for (int c = 0; c < BN; c += 4) {
                  const float4 b4 = *reinterpret_cast<const float4*>(b2m + c);
                  float t[4];
                  if constexpr (KB) {
                    const uint64_t c2 = c < 64 ? pack2(cb0, cb0) : pack2(cb1, cb1);
                    unpack2(ffma2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), c2,
                                  pack2(b4.x, b4.y)), t[0], t[1]);
                    unpack2(ffma2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), c2,
                                  pack2(b4.z, b4.w)), t[2], t[3]);
                  } else {
                    const float4 k4 = *reinterpret_cast<const float4*>(ksm + c);
                    unpack2(ffma2(fmul2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), pack2(k4.x, k4.y)),
                                  cq2o, pack2(b4.x, b4.y)), t[0], t[1]);
                    unpack2(ffma2(fmul2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), pack2(k4.z, k4.w)),
                                  cq2o, pack2(b4.z, b4.w)), t[2], t[3]);
                  }
                  if constexpr (ROWMASK) {  // this row's mask values (log2 units)
                    const uint8_t* mb = smem + L::OFF_MK + ss * L::MB + s * (kM * 128);
                    if ((c & 15) == 0) rmk.load(mb, r, c, a.rm_dtype);
                    float mk[4];
                    rmk.get4(mb, r, c, a.rm_dtype, mk);
    #pragma unroll
                    for (int e = 0; e < 4; ++e) t[e] = fmaf(mk[e], kLog2e, t[e]);
                  }
                  const int q = (c >> 2) & 3;
                  mo[q] = fmax3(mo[q], fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
    #pragma unroll
                  for (int h2 = 0; h2 < 2; ++h2) {
                    float t0, t1;
                    unpack2(fadd2(pack2(t[2 * h2], t[2 * h2 + 1]), nmo), t0, t1);
                    sv[(c >> 1) + h2] = p_pack(t0, t1, lsum[h2]);
                  }
                }
              } else if constexpr (KB) {
                // raw maxima per 64-key half (mo[0..1] and mo[2..3]), scaled below
    #pragma unroll
                for (int c = 0; c < BN; c += 8) {
                  const uint64_t c2 = c < 64 ? pack2(cb0, cb0) : pack2(cb1, cb1);
    #pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    const float s0 = __uint_as_float(sv[c + 2 * q]), s1 = __uint_as_float(sv[c + 2 * q + 1]);
                    const int i = (c < 64 ? 0 : 2) + (q & 1);
                    mo[i] = fmax3(mo[i], s0, s1);
                    float t0, t1;
                    unpack2(ffma2(pack2(s0, s1), c2, nmo), t0, t1);
                    sv[(c >> 1) + q] = p_pack(t0, t1, lsum[q & 1]);
                  }
                }
              } else {
    #pragma unroll
              for (int c = 0; c < BN; c += 8) {
                const float4 ka = *reinterpret_cast<const float4*>(ksm + c);
                const float4 kb = *reinterpret_cast<const float4*>(ksm + c + 4);
                float u[8];
                unpack2(fmul2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), pack2(ka.x, ka.y)), u[0], u[1]);
                unpack2(fmul2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), pack2(ka.z, ka.w)), u[2], u[3]);
                unpack2(fmul2(pack2(__uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5])), pack2(kb.x, kb.y)), u[4], u[5]);
                unpack2(fmul2(pack2(__uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7])), pack2(kb.z, kb.w)), u[6], u[7]);
    #pragma unroll
                for (int q = 0; q < 4; ++q) {
                  mo[q] = fmax3(mo[q], u[2 * q], u[2 * q + 1]);
                  float t0, t1;
                  unpack2(ffma2(pack2(u[2 * q], u[2 * q + 1]), cq2o, nmo), t0, t1);
                  sv[(c >> 1) + q] = p_pack(t0, t1, lsum[q & 1]);
                }
              }
              }
              const float rmo = fmaxf(fmaxf(mo[0], mo[1]), fmaxf(mo[2], mo[3]));
              float tmx = fast ? cq * rmo : rmo;
              if (KB && fast) tmx = fmaxf(fmaxf(mo[0], mo[1]) * cb0, fmaxf(mo[2], mo[3]) * cb1);
              if (__any_sync(0xffffffffu, tmx > m + kRedo)) {
                one = false;  // redo exactly: S is still in TMEM
                if constexpr (BN == 128) tmem_ld128(tS, sv);
                else tmem_ld64(tS, sv);
                tmem_wait_ld(sv);
                lsum[0] = lsum[1] = pack2(0.f, 0.f);
              } else {
                m_pend = tmx > m + kRescaleLog2 ? tmx : m;
              }
            }
          }
          if (!one) {  // ---- two passes: the row maximum, then P
          // u = acc * k_scale (fast tiles) or t = u * cq + bias*log2e / -inf
          // (masked tiles), in place, and the row maximum.
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (KB && fast) {  // raw S stays; maxima per 64-key half
    #pragma unroll
            for (int c = 0; c < BN; c += 8)
    #pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int i = (c < 64 ? 0 : 2) + (q & 1);
                mx[i] = fmax3(mx[i], __uint_as_float(sv[c + 2 * q]), __uint_as_float(sv[c + 2 * q + 1]));
              }
          } else if (fast) {
    #pragma unroll
            for (int c = 0; c < BN; c += 8) {
              const float4 ka = *reinterpret_cast<const float4*>(ksm + c);
              const float4 kb = *reinterpret_cast<const float4*>(ksm + c + 4);
              float f[8];
              unpack2(fmul2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), pack2(ka.x, ka.y)), f[0], f[1]);
              unpack2(fmul2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), pack2(ka.z, ka.w)), f[2], f[3]);
              unpack2(fmul2(pack2(__uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5])), pack2(kb.x, kb.y)), f[4], f[5]);
              unpack2(fmul2(pack2(__uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7])), pack2(kb.z, kb.w)), f[6], f[7]);
    #pragma unroll
              for (int q = 0; q < 4; ++q) mx[q] = fmax3(mx[q], f[2 * q], f[2 * q + 1]);
    #pragma unroll
              for (int q = 0; q < 8; ++q) sv[c + q] = __float_as_uint(f[q]);
            }
          } else {
    #pragma unroll
            for (int c = 0; c < BN; c += 4) {
              const float4 b4 = *reinterpret_cast<const float4*>(b2m + c);
              float f[4];
              if constexpr (KB) {
                const uint64_t c2 = c < 64 ? pack2(cb0, cb0) : pack2(cb1, cb1);
                unpack2(ffma2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), c2,
                              pack2(b4.x, b4.y)), f[0], f[1]);
                unpack2(ffma2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), c2,
                              pack2(b4.z, b4.w)), f[2], f[3]);
              } else {
                const float4 k4 = *reinterpret_cast<const float4*>(ksm + c);
                unpack2(ffma2(fmul2(pack2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), pack2(k4.x, k4.y)),
                              cq2, pack2(b4.x, b4.y)), f[0], f[1]);
                unpack2(ffma2(fmul2(pack2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), pack2(k4.z, k4.w)),
                              cq2, pack2(b4.z, b4.w)), f[2], f[3]);
              }
              if constexpr (ROWMASK) {
                const uint8_t* mb = smem + L::OFF_MK + ss * L::MB + s * (kM * 128);
                if ((c & 15) == 0) rmk.load(mb, r, c, a.rm_dtype);
                float mk[4];
                rmk.get4(mb, r, c, a.rm_dtype, mk);
    #pragma unroll
                for (int e = 0; e < 4; ++e) f[e] = fmaf(mk[e], kLog2e, f[e]);
              }
              const int q = (c >> 2) & 3;
              mx[q] = fmax3(mx[q], fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
    #pragma unroll
              for (int e = 0; e < 4; ++e) sv[c + e] = __float_as_uint(f[e]);
            }
          }
          const float rmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          float tmax = fast ? cq * rmax : rmax;
          if (KB && fast) tmax = fmaxf(fmaxf(mx[0], mx[1]) * cb0, fmaxf(mx[2], mx[3]) * cb1);
          const float m_new = fmaxf(m, tmax);
          const bool need = m_new > m + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2(m - m_new) : 1.f;
            if (L::DBS && it > 0) {  // the previous tile's P V may still be adding into O
              ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_PVT), (it - 1) & 1, ctl, kErrSoftmax));
              if (!ok) break;
              tc_fence_after();
            }
            if (it > 0) rescale_o(alpha);
            l *= alpha;
            if (need) m = m_new;
          }
          const float mref = (m == -INFINITY) ? 0.f : m;
          const float k1 = fast ? cq : 1.f;
          const uint64_t k1v = pack2(k1, k1);
          const uint64_t nm = pack2(-mref, -mref);
          // p = 2^(t - m) with the row sum in fp32; P packed to 16 bits in place
          // (pair i lands in word i, whose value is already consumed) and written
          // to the first BN/2 columns of S in one store.
    #pragma unroll
          for (int e = 0; e < BN / 2; ++e) {
            uint64_t kv2 = k1v;
            if (KB && fast) kv2 = 2 * e < 64 ? pack2(cb0, cb0) : pack2(cb1, cb1);
            float t0, t1;
            unpack2(ffma2(pack2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), kv2, nm), t0, t1);
            sv[e] = p_pack(t0, t1, lsum[e & 1]);
          }
          if (OP) m_pend = m;
          }  // ---- two passes
          if constexpr (BN == 128) {
            tmem_st64(tS, *reinterpret_cast<uint32_t(*)[64]>(sv));
          } else {
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(sv));
          }
          float la, lb, lc, ld;
          unpack2(lsum[0], la, lb);
          unpack2(lsum[1], lc, ld);
          l += (la + lb) + (lc + ld);
        }
        tmem_wait_st();
        tc_fence_before();
        if (PAIR && !leader) {
          // The leader's MMA reads this P from this CTA's TMEM: one arrival per
          // warp, ordered by the tcgen05 wait and fence above.
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(lbar(L::B_PF + sb));
        } else {
          mbar_arrive(bar(L::B_PF + sb));
        }
        if (r == 0) IA_TRACE_POINT(3 + 4 * s, it);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_SCE + ss));
      }
      // ------------------------------------------------------------ epilogue
      if (ok && n_it > 0)
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_OF + s), 0, ctl, kErrSoftmax));
      if (ok) {
        tc_fence_after();
        if (r == 0 && s == 0) IA_TRACE_POINT(14, 8);
        if constexpr (L::ONES) {  // the row sum the MMA accumulated in column D
          if (n_it > 0) {
            uint32_t lr[16];
            tmem_ld16(tO + D, lr);
            tmem_wait_ld(lr);
            l = __uint_as_float(lr[0]);
          }
        }
        bool pad = false;
        if (a.pad_query && row_ok) pad = (row & 63) >= __ldg(a.kv_valid + (row >> 6));
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        char* orow = static_cast<char*>(a.out) +
                     (b * a.o_sb + h * a.o_sh + static_cast<int64_t>(row) * a.o_ss) * 2;
        // Head dim 64: an fp32 partial goes out through shared memory (the K
        // buffers for stage 0, the V buffers for stage 1, idle once this
        // stage's last P V has completed), each warp storing its 32 rows as 512
        // contiguous bytes per instruction instead of 32 scattered 16-byte
        // pieces. 16-byte chunk j of lane l's row sits at slot j ^ (l & 15).
        constexpr bool STAGE = L::SEGOK;
        const bool staged = STAGE && a.ws_o != nullptr;
        uint8_t* stg = smem + (s == 0 ? L::OFF_KH : L::OFF_V) + (warp & 3) * (32 * D * 4);
        if (staged) fence_proxy_async_smem();
  #pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          if (n_it > 0) {
            tmem_ld32(tO + c0, rr);
            tmem_wait_ld(rr);
          } else {
  #pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
          uint32_t pk[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i) {
            float o0 = __uint_as_float(rr[2 * i]) * inv_l * vsc[c0 + 2 * i];
            float o1 = __uint_as_float(rr[2 * i + 1]) * inv_l * vsc[c0 + 2 * i + 1];
            if (pad) o0 = o1 = 0.f;
            pk[i] = VBF16 ? cvt_bf16x2(o0, o1) : cvt_f16x2(o0, o1);
          }
          if (staged) {
  #pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              float f[4];
  #pragma unroll
              for (int e = 0; e < 4; ++e)
                f[e] = pad ? 0.f : __uint_as_float(rr[4 * v4 + e]) * inv_l * vsc[c0 + 4 * v4 + e];
              const int j = c0 / 4 + v4;
              *reinterpret_cast<float4*>(stg + lane * (D * 4) + ((j ^ (lane & 15)) << 4)) =
                  make_float4(f[0], f[1], f[2], f[3]);
            }
          } else if (row_ok && a.ws_o != nullptr) {  // fp32 partial of this key range
            float4* dst = reinterpret_cast<float4*>(
                a.ws_o + ((static_cast<int64_t>(split * a.B + b) * a.H + h) * a.Sq + row) * D + c0);
  #pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              float f[4];
  #pragma unroll
              for (int e = 0; e < 4; ++e)
                f[e] = pad ? 0.f : __uint_as_float(rr[4 * v4 + e]) * inv_l * vsc[c0 + 4 * v4 + e];
              dst[v4] = make_float4(f[0], f[1], f[2], f[3]);
            }
          } else if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 2);
  #pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if constexpr (STAGE) {
          if (staged) {
            static_assert(D == 64 && L::NKS * L::KH >= 4 * 32 * D * 4 && L::NVS * L::VB >= 4 * 32 * D * 4,
                          "staging: 256-byte rows, 32 KB per stage");
            __syncwarp();
            float* wsb = a.ws_o + (static_cast<int64_t>(split * a.B + b) * a.H + h) * a.Sq * D;
            const int rbase = q0 + s * kM + (warp & 3) * 32;
  #pragma unroll 4
            for (int i = 0; i < 16; ++i) {  // rows 2i and 2i+1, one per half-warp
              const int rw = 2 * i + (lane >> 4), j = lane & 15;
              const float4 v = *reinterpret_cast<const float4*>(stg + rw * (D * 4) + ((j ^ (rw & 15)) << 4));
              if (rbase + rw < a.Sq)
                *reinterpret_cast<float4*>(wsb + static_cast<int64_t>(rbase + rw) * D + j * 4) = v;
            }
            fence_proxy_async_smem();  // before the next segment's copies into these buffers
          }
        }
        if (row_ok && (a.lse != nullptr || a.ws_l != nullptr)) {
          const float lse = (pad || !(l > 0.f)) ? -INFINITY : (m + log2f(l)) * kLn2;
          if (a.ws_l != nullptr) {
            a.ws_l[(static_cast<int64_t>(split * a.B + b) * a.H + h) * a.Sq + row] = lse;
            if (seg_full)  // the query tile's second partial is empty (its O is not read)
              a.ws_l[(static_cast<int64_t>(a.B + b) * a.H + h) * a.Sq + row] = -INFINITY;
          } else {
            a.lse[b * a.l_sb + h * a.l_sh + row] = lse;
          }
        }
      }
    }

  }  // segments

  // ------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0) IA_TRACE_POINT(14, 9);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) IA_TRACE_POINT(14, 10);
  // Neither CTA of a pair leaves while the leader's MMAs may still read the
  // peer's shared memory or TMEM, or the peer's arrivals reach the leader.
  if constexpr (PAIR) cluster_sync();
  if (warp == L::W_MMA) {
    tc_fence_after();
    const uint32_t tmem = misc[0];
    if constexpr (PAIR) tmem_dealloc_pair(tmem, L::TMEM_COLS);
    else tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 4-D map over [B][H][S][D] (innermost first), strides in bytes.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int esize, int D, int S,
              int H, int B, int64_t ss, int64_t sh, int64_t sb, int box0, int box1,
              CUtensorMapSwizzle sw) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const int64_t es = esize;
  int64_t s1 = ss * es, s2 = sh * es, s3 = sb * es;
  if (H <= 1) s2 = s1 * (S > 0 ? S : 1);
  if (B <= 1) s3 = s2 * (H > 0 ? H : 1);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S > 0 ? S : 1),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s1), static_cast<cuuint64_t>(s2),
                           static_cast<cuuint64_t>(s3)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1), 1, 1};
  cuuint32_t est[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, est,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int QS, int BN, bool SPARSE, bool VBF16, bool QRAW, bool ROWMASK, bool PAIR = false,
          bool KB = false>
ia_status run(const AttnLaunch& A, int num_sms, cudaStream_t st, const char** msg) {
  using L = Layout<D, QS, BN, SPARSE, ROWMASK, PAIR, KB>;
  const ia_attn_params& p = A.p;
  CUtensorMap tq, tk, tv, tm;
  std::memset(&tm, 0, sizeof(tm));
  if constexpr (ROWMASK) {  // per-row mask tiles: [B][H][Sq][Sk], broadcast dims of size 1
    const int dt = p.mask_dtype;
    const int es = dt == IA_MASK_F32 ? 4 : dt == IA_MASK_BOOL ? 1 : 2;
    const CUtensorMapDataType mdt = dt == IA_MASK_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : dt == IA_MASK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : dt == IA_MASK_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int Hm = p.mask_strides[1] != 0 ? p.H : 1, Bm = p.mask_strides[0] != 0 ? p.B : 1;
    if (!make_map(&tm, mdt, p.mask, es, p.Sk, p.Sq, Hm, Bm, p.mask_strides[2], p.mask_strides[1],
                  p.mask_strides[0], 128 / es, kM, CU_TENSOR_MAP_SWIZZLE_128B)) {
      *msg = "cuTensorMapEncodeTiled rejected the mask layout (alignment or stride)";
      return IA_ERR_INVALID_ARG;
    }
  }
  const CUtensorMapDataType qdt = !QRAW ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : VBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const bool okq = make_map(&tq, qdt, A.q, QRAW ? 2 : 1, D, p.Sq, p.H, p.B, p.q_strides[2],
                            p.q_strides[1], p.q_strides[0], D, kM, CU_TENSOR_MAP_SWIZZLE_NONE);
  const bool okk = make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, A.k, 1, D, p.Sk, p.H, p.B,
                            p.k_strides[2], p.k_strides[1], p.k_strides[0], D, L::KROWS,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
  const bool okv = make_map(&tv, VBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                            A.v, 2, D, p.Sk, p.H, p.B, p.v_strides[2], p.v_strides[1],
                            p.v_strides[0], 64, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!(okq && okk && okv)) {
    *msg = "cuTensorMapEncodeTiled rejected a Q/K/V layout (alignment or stride)";
    return IA_ERR_INVALID_ARG;
  }
  Params a{};
  if (QRAW && p.q_prologue != nullptr) {
    const ia_qk_prologue& pr = *p.q_prologue;
    a.q_pro = (pr.q_norm_weight != nullptr || pr.rope != IA_ROPE_NONE) ? 1 : 0;
    a.qp_w = pr.q_norm_weight;
    a.qp_eps = pr.eps;
    a.qp_rope = pr.rope;
    a.qp_cos = pr.rope_cos;
    a.qp_sin = pr.rope_sin;
    a.qp_stride = pr.rope_stride;
    a.qp_pos0 = pr.q_pos0;
  }
  a.q_scale = A.q_scale;
  a.k_scale = A.k_scale;
  a.bias = A.bias;
  a.bias_dtype = A.bias_dtype;
  a.bias_sb = A.bias_sb;
  a.bias_sh = A.bias_sh;
  a.rm_dtype = p.mask_dtype;
  a.rm_h = p.mask_strides[1] != 0 ? 1 : 0;
  a.rm_b = p.mask_strides[0] != 0 ? 1 : 0;
  a.mask = A.mask;
  a.kv_valid = p.kv_valid;
  a.v_scale = p.v_scale;
  a.out = A.out;
  a.lse = A.lse;
  a.H = p.H;
  a.Sq = p.Sq;
  a.Sk = p.Sk;
  a.Tq = (p.Sq + 63) / 64;
  a.Tk = (p.Sk + 63) / 64;
  a.n_tiles = SPARSE ? a.Tk : (p.Sk + BN - 1) / BN;
  a.cq_mult = A.sm_scale * kLog2e;
  a.gran_block = p.granularity == IA_PER_BLOCK64 ? 1 : 0;
  a.pad_query = (p.kv_valid != nullptr && p.Sq == p.Sk) ? 1 : 0;
  a.qs_sb = p.qs_strides[0];
  a.qs_sh = p.qs_strides[1];
  a.ks_sb = p.ks_strides[0];
  a.ks_sh = p.ks_strides[1];
  a.o_sb = p.o_strides[0];
  a.o_sh = p.o_strides[1];
  a.o_ss = p.o_strides[2];
  a.l_sb = p.lse_strides[0];
  a.l_sh = p.lse_strides[1];
  a.timeout_ns = p.wait_timeout_ns ? p.wait_timeout_ns : 2000000000ull;
  a.debug_stall = p.debug_stall;
  a.B = p.B;
  const int nsplit = p.kv_splits > 1 ? p.kv_splits : 1;
  a.nsplit = nsplit;
  a.tps = (a.n_tiles + nsplit - 1) / nsplit;
  a.ws_o = nullptr;
  a.ws_l = nullptr;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
  if (nsplit > 1) {
    a.ws_o = static_cast<float*>(A.workspace);
    a.ws_l = a.ws_o + static_cast<int64_t>(nsplit) * rows * D;
  }
  const size_t smem = L::SMEM_FIXED + (SPARSE ? static_cast<size_t>(a.Tk) * 2 : 0);
  // Two key ranges on the dense head-dim-64 kernel with at least one query tile
  // per SM: one CTA per SM, each taking an equal share of the (query tile, key
  // tile) units, instead of a grid whose last round runs part-empty.
  int gx = (p.Sq + kM * QS - 1) / (kM * QS);
  if (PAIR) gx = (gx + 1) & ~1;  // whole pairs; a surplus CTA's rows are all past Sq
  dim3 grid(gx, p.H, p.B * nsplit);
  a.seg_units = 0;
  a.seg_nqt = gx;
  auto kern = attn_fwd_kernel<D, QS, BN, SPARSE, VBF16, QRAW, ROWMASK, PAIR, KB>;
  if constexpr (L::SEGOK && !QRAW) {
    const int64_t n_qt = static_cast<int64_t>(p.B) * p.H * gx;
    if (nsplit == 2 && n_qt >= num_sms && n_qt * a.n_tiles < (int64_t{1} << 40)) {
      a.seg_units = n_qt * a.n_tiles;
      grid = dim3(num_sms, 1, 1);
      kern = attn_fwd_kernel<D, QS, BN, SPARSE, VBF16, QRAW, ROWMASK, PAIR, KB, true>;
    }
  }
  if (smem > 232448) {
    *msg = "key-tile list does not fit in shared memory (too many key tiles)";
    return IA_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return IA_ERR_CUDA;
  }

  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(L::NWARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tm, a);
    if (e != cudaSuccess) {
      *msg = cudaGetErrorString(e);
      return IA_ERR_CUDA;
    }
  } else {
    kern<<<grid, L::NWARPS * 32, smem, st>>>(tq, tk, tv, tm, a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return IA_ERR_CUDA;
  }
  if (nsplit > 1) {  // exact merge of the key ranges
    MergeNArgs m{};
    for (int k = 0; k < nsplit; ++k) {
      m.o[k] = a.ws_o + static_cast<int64_t>(k) * rows * D;
      m.l[k] = a.ws_l + static_cast<int64_t>(k) * rows;
    }
    m.n = nsplit;
    m.in_f32 = 1;
    m.out = A.out;
    m.lse = A.lse;
    m.B = p.B;
    m.H = p.H;
    m.Sq = p.Sq;
    m.D = D;
    m.dtype = VBF16 ? IA_BF16 : IA_FP16;
    m.o_sb = p.o_strides[0];
    m.o_sh = p.o_strides[1];
    m.o_ss = p.o_strides[2];
    m.l_sb = p.lse_strides[0];
    m.l_sh = p.lse_strides[1];
    e = launch_merge_n(m, num_sms, st);
    if (e != cudaSuccess) {
      *msg = cudaGetErrorString(e);
      return IA_ERR_CUDA;
    }
  }
  return IA_OK;
}

template <bool QRAW>
ia_status dispatch(const AttnLaunch& A, int num_sms, cudaStream_t st, const char** msg) {
  const ia_attn_params& p = A.p;
  const bool bf = p.v_dtype == IA_BF16;
  if (A.row_mask) {  // 64-key tiles, mask tiles by TMA
    // masks of at most two bytes per key: two 128-row stages, whose mask rows
    // fit the ring (16-bit Q rows are staged in that ring until quantized);
    // fp32 masks take one stage
    if (p.mask_dtype != IA_MASK_F32) {
      if (p.D == 128)
        return bf ? run<128, 2, 64, false, true, QRAW, true>(A, num_sms, st, msg)
                  : run<128, 2, 64, false, false, QRAW, true>(A, num_sms, st, msg);
      return bf ? run<64, 2, 64, false, true, QRAW, true>(A, num_sms, st, msg)
                : run<64, 2, 64, false, false, QRAW, true>(A, num_sms, st, msg);
    }
    if (p.D == 128)
      return bf ? run<128, 1, 64, false, true, QRAW, true>(A, num_sms, st, msg)
                : run<128, 1, 64, false, false, QRAW, true>(A, num_sms, st, msg);
    return bf ? run<64, 1, 64, false, true, QRAW, true>(A, num_sms, st, msg)
              : run<64, 1, 64, false, false, QRAW, true>(A, num_sms, st, msg);
  }
  if (A.mask != nullptr) {
    if (p.D == 128)
      return bf ? run<128, 1, 64, true, true, QRAW, false>(A, num_sms, st, msg)
                : run<128, 1, 64, true, false, QRAW, false>(A, num_sms, st, msg);
    return bf ? run<64, 1, 64, true, true, QRAW, false>(A, num_sms, st, msg)
              : run<64, 1, 64, true, false, QRAW, false>(A, num_sms, st, msg);
  }
  if (p.D == 128)  // CTA pairs with 256-row MMAs
    return bf ? run<128, 2, 128, false, true, QRAW, false, true>(A, num_sms, st, msg)
              : run<128, 2, 128, false, false, QRAW, false, true>(A, num_sms, st, msg);
  if (p.granularity == IA_PER_BLOCK64)  // per-block K scales folded into the softmax constants
    return bf ? run<64, 2, 128, false, true, QRAW, false, false, true>(A, num_sms, st, msg)
              : run<64, 2, 128, false, false, QRAW, false, false, true>(A, num_sms, st, msg);
  return bf ? run<64, 2, 128, false, true, QRAW, false>(A, num_sms, st, msg)
            : run<64, 2, 128, false, false, QRAW, false>(A, num_sms, st, msg);
}

}  // namespace

ia_status launch_attention(const AttnLaunch& A, int num_sms, cudaStream_t st, const char** msg) {
  const ia_attn_params& p = A.p;
  if (p.B == 0 || p.H == 0 || p.Sq == 0) return IA_OK;
  return A.q_raw ? dispatch<true>(A, num_sms, st, msg) : dispatch<false>(A, num_sms, st, msg);
}

cudaError_t attention_read_device_error(unsigned int* out, cudaStream_t st) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_attn_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(unsigned int));
}

}  // namespace ia

#ifdef IA_TRACE
extern "C" __attribute__((visibility("default"))) int ia_trace_read(unsigned long long* out) {
  cudaDeviceSynchronize();
  return static_cast<int>(cudaMemcpyFromSymbol(out, ia::g_attn_trace, sizeof(ia::g_attn_trace)));
}
#endif
