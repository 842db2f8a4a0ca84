// mx9.cu -- MX9 pack / unpack for sm_103a.
//
// Method: AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
// pack/unpack" (Summary, "Key design choices", review thread): blocks of 16
// elements along the last axis; shared E8M0 exponent E = the block's largest
// element exponent from the native bits; one prime bit per pair of elements
// (set when the pair's exponent is below E); scale exponent
// k = max(E - 6 - prime, -126); q = clamp(round_half_even(x / 2^k), -127, 127).
//
// pack: persistent and warp-specialized like the dual-axis kernel.  One
// producer warp streams contiguous runs of blocks into a shared-memory
// ring with 1-D bulk copies (TMA); each consumer thread then owns whole
// 16-element blocks (one per stage for fp32, two for bf16), so exponents and
// prime bits need no shuffles, and writes their 16 q bytes, exponent byte and
// prime byte with coalesced stores.  Finite blocks round with one FMA against
// 1.5 * 2^23 and clamp two elements at once as int16 pairs; bf16 blocks take
// their exponent maximum on the packed words and feed the bf16 halves to a
// mixed-precision FMA, which keeps the integer pipe (the limit for bf16) light.
// unpack: a streaming kernel, one wave of resident blocks; each lane writes 16
// output bytes (4 fp32 or 8 bf16 elements), exact q * 2^k built without
// conversion instructions.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxq.h"
#include "mxq_device.cuh"
#include "mxq_host.h"

namespace {

using namespace mxq;

// Launch shape.  The defaults are the measured best on GB300; the macros only
// exist so that other shapes can be built for measurement.
#ifndef MXQ_MX9_PACK_F32_WARPS
#define MXQ_MX9_PACK_F32_WARPS 8
#endif
#ifndef MXQ_MX9_PACK_F32_RING_KB
#define MXQ_MX9_PACK_F32_RING_KB 64
#endif
#ifndef MXQ_MX9_PACK_BF16_WARPS
#define MXQ_MX9_PACK_BF16_WARPS 8
#endif
#ifndef MXQ_MX9_PACK_BF16_RING_KB
#define MXQ_MX9_PACK_BF16_RING_KB 48
#endif
#ifndef MXQ_MX9_PACK_CTAS_PER_SM
#define MXQ_MX9_PACK_CTAS_PER_SM 2
#endif
#ifndef MXQ_MX9_PACK_FMA_ROUND
#define MXQ_MX9_PACK_FMA_ROUND 1
#endif
#ifndef MXQ_MX9_PACK_BF16_PER_THREAD
#define MXQ_MX9_PACK_BF16_PER_THREAD 2
#endif
#ifndef MXQ_MX9_PACK_F32_PER_THREAD
#define MXQ_MX9_PACK_F32_PER_THREAD 1
#endif
#ifndef MXQ_MX9_PACK_MIXED_FMA
#define MXQ_MX9_PACK_MIXED_FMA 1
#endif
#ifndef MXQ_MX9_UNPACK_PRMT_F32
#define MXQ_MX9_UNPACK_PRMT_F32 0
#endif
#ifndef MXQ_MX9_UNPACK_PRMT_BF16
#define MXQ_MX9_UNPACK_PRMT_BF16 1
#endif
#ifndef MXQ_MX9_UNPACK_UNROLL_F32
#define MXQ_MX9_UNPACK_UNROLL_F32 2
#endif
#ifndef MXQ_MX9_UNPACK_UNROLL_BF16
#define MXQ_MX9_UNPACK_UNROLL_BF16 4
#endif

constexpr int kUnpackBlock = 256;

// Sticky status word of this file's kernels (MXQ_DEV_* bits).
__device__ unsigned int g_mx9_status = 0;

// Pack kernel shape per input type: consumer warps (kPerThread 16-element
// blocks per consumer thread and stage), one producer warp, a ring of stages.
// Rings deeper than these measured slower.
template <bool kBF16>
struct PackShape {
  static constexpr int kWarps = kBF16 ? MXQ_MX9_PACK_BF16_WARPS : MXQ_MX9_PACK_F32_WARPS;
  static constexpr int kPerThread = kBF16 ? MXQ_MX9_PACK_BF16_PER_THREAD : MXQ_MX9_PACK_F32_PER_THREAD;
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kBlocksPerStage = kConsumers * kPerThread;
  static constexpr uint32_t kBlockBytes = kBF16 ? 32u : 64u;  // 16 elements
  static constexpr uint32_t kStageBytes = kBlocksPerStage * kBlockBytes;
  static constexpr uint32_t kRingBytes =
      (kBF16 ? MXQ_MX9_PACK_BF16_RING_KB : MXQ_MX9_PACK_F32_RING_KB) * 1024u;
  static constexpr int kStages = static_cast<int>(kRingBytes / kStageBytes);
  static constexpr uint32_t kOffBar = kStages * kStageBytes;
  static constexpr uint32_t kOffFlag = kOffBar + 16u * kStages;
  static constexpr uint32_t kSmemBytes = kOffFlag + 16u + 128u;  // + alignment slack
  static_assert(kStages >= 2, "ring too small");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory budget");
};

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Multiplier 2^-k of a pair from the block's exponent field eb8 (E = eb8 - 127)
// and the pair's prime bit t: k = max(E - 6 - t, -126), 127 - k = min(260 - eb8 + t, 253).
__device__ __forceinline__ float pair_multiplier(uint32_t eb8, uint32_t t) {
  return __uint_as_float(min(260u - eb8 + t, 253u) << 23);
}

// x * 2^-k (exact multiply, no flush) rounded half-to-even to an integer and
// clamped to [-127, 127]; cvt.rni gives 0 for NaN and saturates +-Inf.
__device__ __forceinline__ uint32_t q_byte(float x, float mult) {
  const int r = __float2int_rn(fmul_rn_noftz(x, mult));
  return static_cast<uint32_t>(max(-127, min(127, r))) & 0xFFu;
}

__device__ __forceinline__ float fma_rn_noftz(float a, float b, float c) {
  float r;
  asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two elements of a finite block: round_half_even(x * mult) clamped to
// [-127, 127], as two int16 in one word.  For |x * mult| < 2^22 the FMA
// 1.5 * 2^23 + x * mult rounds once, half to even, to an integer whose
// two's-complement value sits in the low 16 bits of the result; a finite
// block gives |x * mult| < 2^8.
__device__ __forceinline__ uint32_t q_pair_s16x2(uint32_t a, uint32_t b, float mult) {
  const float ra = fma_rn_noftz(__uint_as_float(a), mult, 12582912.0f);
  const float rb = fma_rn_noftz(__uint_as_float(b), mult, 12582912.0f);
  uint32_t h = __byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x5410);
  asm("max.s16x2 %0, %0, %1;" : "+r"(h) : "r"(0xFF81FF81u));
  asm("min.s16x2 %0, %0, %1;" : "+r"(h) : "r"(0x007F007Fu));
  return h;
}

// q_pair_s16x2 on the two bf16 halves of w without widening them: the
// mixed-precision FMA takes bf16 factors and an fp32 addend and rounds once.
// mult_bits: the fp32 power-of-two multiplier, exact as bf16 (its high half).
__device__ __forceinline__ uint32_t q_pair_s16x2_bf16(uint32_t w, uint32_t mult_bits) {
  float ra, rb;
  asm("{\n\t.reg .b16 xl, xh, ml, mh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "mov.b32 {ml, mh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, mh, %4;\n\t"
      "fma.rn.f32.bf16 %1, xh, mh, %4;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "r"(w), "r"(mult_bits), "f"(12582912.0f));
  uint32_t h = __byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x5410);
  asm("max.s16x2 %0, %0, %1;" : "+r"(h) : "r"(0xFF81FF81u));
  asm("min.s16x2 %0, %0, %1;" : "+r"(h) : "r"(0x007F007Fu));
  return h;
}

// One block of 16 elements given as 16 fp32 bit patterns.
__device__ __forceinline__ void pack_block(const uint32_t* f, uint4* q, uint32_t* eb_out,
                                           uint32_t* prime_out) {
  uint32_t pe[8];
  uint32_t eb = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    pe[p] = max(f[2 * p] & 0x7F800000u, f[2 * p + 1] & 0x7F800000u);
    eb = max(eb, pe[p]);
  }
  const uint32_t eb8 = eb >> 23;
  if (MXQ_MX9_PACK_FMA_ROUND && eb8 != 255u) {
    // finite block (no Inf or NaN): rounding by FMA, clamping on int16 pairs
    const float m0 = pair_multiplier(eb8, 0u), m1 = pair_multiplier(eb8, 1u);
    uint32_t bits = 0, h[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t t = pe[p] < eb;
      bits |= t << p;
      h[p] = q_pair_s16x2(f[2 * p], f[2 * p + 1], t ? m1 : m0);
    }
    *q = make_uint4(__byte_perm(h[0], h[1], 0x6420), __byte_perm(h[2], h[3], 0x6420),
                    __byte_perm(h[4], h[5], 0x6420), __byte_perm(h[6], h[7], 0x6420));
    *eb_out = eb8;
    *prime_out = bits;
    return;
  }
  uint32_t bits = 0, word[4] = {0, 0, 0, 0};
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t t = pe[p] < eb;
    bits |= t << p;
    const float m = pair_multiplier(eb8, t);
    const uint32_t two = q_byte(__uint_as_float(f[2 * p]), m) |
                         (q_byte(__uint_as_float(f[2 * p + 1]), m) << 8);
    word[p >> 1] |= two << (16 * (p & 1));
  }
  *q = make_uint4(word[0], word[1], word[2], word[3]);
  *eb_out = eb8;
  *prime_out = bits;
}

__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One block of 16 bf16 elements given as 8 words, word p = pair p (element 2p
// in the low half).  Exponent fields are compared in place, two per word; a
// pair is demoted when both of its fields are below the block's: with
// e16 = block field << 7, the low half of (w & 0x7F80) + 0x8000 - e16 reaches
// bit 15 exactly when the element's field is >= the block's, and likewise for
// the high half at bit 31 (the low half cannot carry).
__device__ __forceinline__ void pack_block_bf16(const uint32_t* w, uint4* q, uint32_t* eb_out,
                                                uint32_t* prime_out) {
  uint32_t m[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) m[p] = w[p] & 0x7F807F80u;
  const uint32_t mx = vmax_u16x2(vmax_u16x2(vmax_u16x2(m[0], m[1]), vmax_u16x2(m[2], m[3])),
                                 vmax_u16x2(vmax_u16x2(m[4], m[5]), vmax_u16x2(m[6], m[7])));
  const uint32_t e16 = max(mx & 0xFFFFu, mx >> 16);
  const uint32_t eb8 = e16 >> 7;
  if (!MXQ_MX9_PACK_FMA_ROUND || eb8 == 255u) {
    uint32_t f[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      f[2 * k] = w[k] << 16;                 // exact widening of each bf16
      f[2 * k + 1] = w[k] & 0xFFFF0000u;
    }
    pack_block(f, q, eb_out, prime_out);
    return;
  }
  const uint32_t d2 = (0x8000u - e16) * 0x10001u;
  const float m0 = pair_multiplier(eb8, 0u), m1 = pair_multiplier(eb8, 1u);
  uint32_t bits = 0, h[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t t = ((m[p] + d2) & 0x80008000u) == 0u;
    bits |= t << p;
    if (MXQ_MX9_PACK_MIXED_FMA)
      h[p] = q_pair_s16x2_bf16(w[p], __float_as_uint(t ? m1 : m0));
    else
      h[p] = q_pair_s16x2(w[p] << 16, w[p] & 0xFFFF0000u, t ? m1 : m0);
  }
  *q = make_uint4(__byte_perm(h[0], h[1], 0x6420), __byte_perm(h[2], h[3], 0x6420),
                  __byte_perm(h[4], h[5], 0x6420), __byte_perm(h[6], h[7], 0x6420));
  *eb_out = eb8;
  *prime_out = bits;
}

template <bool kBF16>
__global__ void __launch_bounds__(PackShape<kBF16>::kThreads, MXQ_MX9_PACK_CTAS_PER_SM)
    mx9_pack_kernel(const uint8_t* __restrict__ x, int64_t nb, uint4* __restrict__ q,
                    uint8_t* __restrict__ max_exp, uint8_t* __restrict__ prime) {
  using S = PackShape<kBF16>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + S::kOffFlag);
  auto full = [&](int s) { return base + S::kOffBar + 8u * s; };
  auto empty = [&](int s) { return base + S::kOffBar + 8u * (S::kStages + s); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nchunks = (nb + S::kBlocksPerStage - 1) / S::kBlocksPerStage;
  const int64_t my =
      static_cast<int64_t>(blockIdx.x) < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), S::kWarps);
    }
    *abort_flag = 0u;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == S::kWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int64_t issued = 0;
    for (int64_t i = 0; i < my; ++i) {
      const int s = static_cast<int>(i % S::kStages);
      if (i >= S::kStages &&
          !mbar_wait_bounded(empty(s), static_cast<uint32_t>(((i / S::kStages) - 1) & 1),
                             abort_flag, &g_mx9_status, MXQ_DEV_TIMEOUT))
        break;
      const int64_t b0 = (blockIdx.x + i * static_cast<int64_t>(gridDim.x)) * S::kBlocksPerStage;
      const int64_t nblk = nb - b0 < S::kBlocksPerStage ? nb - b0 : S::kBlocksPerStage;
      const uint32_t bytes = static_cast<uint32_t>(nblk) * S::kBlockBytes;
      mbar_arrive_expect_tx(full(s), bytes);
      bulk_load_1d(base + static_cast<uint32_t>(s) * S::kStageBytes, x + b0 * S::kBlockBytes,
                   bytes, full(s));
      issued = i + 1;
    }
    // drain (a no-op after a normal run: consumers waited for every stage)
    for (int64_t i = issued > S::kStages ? issued - S::kStages : 0; i < issued; ++i)
      mbar_wait_drain(full(static_cast<int>(i % S::kStages)),
                      static_cast<uint32_t>((i / S::kStages) & 1));
    return;
  }

  // -------------------------------------------------------------- consumers
  for (int64_t i = 0; i < my; ++i) {
    const int s = static_cast<int>(i % S::kStages);
    const bool ok = mbar_wait_bounded(full(s), static_cast<uint32_t>((i / S::kStages) & 1),
                                      abort_flag, &g_mx9_status, MXQ_DEV_TIMEOUT);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    const int64_t blk0 = (blockIdx.x + i * static_cast<int64_t>(gridDim.x)) * S::kBlocksPerStage;
#pragma unroll
    for (int j = 0; j < S::kPerThread; ++j) {
      const int local = j * S::kConsumers + tid;
      const int64_t blk = blk0 + local;
      if (blk >= nb) break;
      const uint32_t src = base + static_cast<uint32_t>(s) * S::kStageBytes + local * S::kBlockBytes;
      uint4 qv;
      uint32_t eb8, bits;
      if (kBF16) {
        const uint4 a = lds128(src), b = lds128(src + 16);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        pack_block_bf16(w, &qv, &eb8, &bits);
      } else {
        uint32_t f[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 a = lds128(src + 16u * k);
          f[4 * k] = a.x;
          f[4 * k + 1] = a.y;
          f[4 * k + 2] = a.z;
          f[4 * k + 3] = a.w;
        }
        pack_block(f, &qv, &eb8, &bits);
      }
      __stcs(q + blk, qv);
      max_exp[blk] = static_cast<uint8_t>(eb8);
      prime[blk] = static_cast<uint8_t>(bits);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }
}

// ---------------------------------------------------------------------------
// unpack
// ---------------------------------------------------------------------------

// 2^e as fp32 for e in the normal range [-126, 127].
__device__ __forceinline__ float exp2_normal(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

__device__ __forceinline__ float fadd_rn_noftz(float a, float b) {
  float r;
  asm("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Exact float of a small integer q (|q| < 2^22) without a conversion
// instruction: the bits of 1.5 * 2^23 + q, minus 1.5 * 2^23.
__device__ __forceinline__ float small_int_to_float(int32_t q) {
  return fadd_rn_noftz(__int_as_float(0x4B400000 + q), -12582912.0f);
}

// A lane writes 16 output bytes: 4 fp32 or 8 bf16 elements, so 4 (fp32) or
// 2 (bf16) lanes share a block.  q * 2^k is exact (|q| <= 127, k >= -126)
// except for overflow in max_exp 255 blocks; a bf16 result has at most 7
// significant bits, so the top half of the fp32 is the exact bf16.
template <bool kBF16>
struct UnpackLane {
  static constexpr int kElems = kBF16 ? 8 : 4;
  static constexpr int kLanesPerBlock = 16 / kElems;
  static constexpr int kUnroll = kBF16 ? MXQ_MX9_UNPACK_UNROLL_BF16 : MXQ_MX9_UNPACK_UNROLL_F32;
};

__device__ __forceinline__ void unpack4(uint32_t w, float s0, float s1, float* y) {
  const int32_t v = static_cast<int32_t>(w);
  y[0] = fmul_rn_noftz(small_int_to_float((v << 24) >> 24), s0);
  y[1] = fmul_rn_noftz(small_int_to_float((v << 16) >> 24), s0);
  y[2] = fmul_rn_noftz(small_int_to_float((v << 8) >> 24), s1);
  y[3] = fmul_rn_noftz(small_int_to_float(v >> 24), s1);
}

// The same four values from vx = w ^ 0x80808080 (each byte then holds q + 128):
// a byte permute puts byte k under the exponent of 2^23, giving the float
// 2^23 + 128 + q, and one exact subtraction leaves q.  Fewer integer
// instructions than the shifts of unpack4; measured faster for bf16 output
// (+5%) and slower for fp32 (-2%), so each output type keeps its better form.
__device__ __forceinline__ void unpack4_biased(uint32_t vx, float s0, float s1, float* y) {
  constexpr float kBias = 8388736.0f;  // 2^23 + 128
  y[0] = fmul_rn_noftz(fadd_rn_noftz(__uint_as_float(__byte_perm(vx, 0x4B000000u, 0x7650)), -kBias), s0);
  y[1] = fmul_rn_noftz(fadd_rn_noftz(__uint_as_float(__byte_perm(vx, 0x4B000000u, 0x7651)), -kBias), s0);
  y[2] = fmul_rn_noftz(fadd_rn_noftz(__uint_as_float(__byte_perm(vx, 0x4B000000u, 0x7652)), -kBias), s1);
  y[3] = fmul_rn_noftz(fadd_rn_noftz(__uint_as_float(__byte_perm(vx, 0x4B000000u, 0x7653)), -kBias), s1);
}

template <bool kBF16>
__global__ void __launch_bounds__(kUnpackBlock) mx9_unpack_kernel(
    const uint32_t* __restrict__ q, const uint8_t* __restrict__ max_exp,
    const uint8_t* __restrict__ prime, void* __restrict__ y, int64_t nchunks) {
  using U = UnpackLane<kBF16>;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kUnpackBlock;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kUnpackBlock + (threadIdx.x - lane);
  // pairs handled by this lane inside its block, and their prime-bit shift
  const int pshift = (lane % U::kLanesPerBlock) * (U::kElems / 2);
  for (int64_t base = warp0; base < nchunks; base += stride * U::kUnroll) {
    uint32_t qv[U::kUnroll][U::kElems / 4], ev[U::kUnroll], pv[U::kUnroll];
#pragma unroll
    for (int u = 0; u < U::kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      if (c < nchunks) {
        if (kBF16) {
          const uint2 w = __ldcs(reinterpret_cast<const uint2*>(q) + c);
          qv[u][0] = w.x;
          qv[u][U::kElems / 4 - 1] = w.y;
        } else {
          qv[u][0] = __ldcs(q + c);
        }
        ev[u] = __ldg(max_exp + c / U::kLanesPerBlock);
        pv[u] = __ldg(prime + c / U::kLanesPerBlock);
      } else {
        qv[u][0] = qv[u][U::kElems / 4 - 1] = ev[u] = pv[u] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < U::kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      if (c >= nchunks) continue;
      const int E = static_cast<int>(ev[u]) - 127;
      const int pbits = static_cast<int>(pv[u] >> pshift);
      float s[U::kElems / 2];
      float v[U::kElems];
      if (kBF16 ? MXQ_MX9_UNPACK_PRMT_BF16 : MXQ_MX9_UNPACK_PRMT_F32) {
        // the two possible pair scales, then one select per pair
        const float s_keep = exp2_normal(max(E - 6, -126)), s_dem = exp2_normal(max(E - 7, -126));
#pragma unroll
        for (int k = 0; k < U::kElems / 2; ++k) s[k] = (pbits >> k) & 1 ? s_dem : s_keep;
#pragma unroll
        for (int k = 0; k < U::kElems / 4; ++k)
          unpack4_biased(qv[u][k] ^ 0x80808080u, s[2 * k], s[2 * k + 1], v + 4 * k);
      } else {
#pragma unroll
        for (int k = 0; k < U::kElems / 2; ++k)
          s[k] = exp2_normal(max(E - 6 - ((pbits >> k) & 1), -126));
#pragma unroll
        for (int k = 0; k < U::kElems / 4; ++k) unpack4(qv[u][k], s[2 * k], s[2 * k + 1], v + 4 * k);
      }
      if (kBF16) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)  // the high halves of two fp32 values
          o[k] = __byte_perm(__float_as_uint(v[2 * k]), __float_as_uint(v[2 * k + 1]), 0x7632);
        __stcs(reinterpret_cast<uint4*>(y) + c, make_uint4(o[0], o[1], o[2], o[3]));
      } else {
        __stcs(reinterpret_cast<float4*>(y) + c, make_float4(v[0], v[1], v[2], v[3]));
      }
    }
  }
}

// One full wave: as many resident blocks as the kernel's occupancy allows on
// every SM, or fewer when the problem is small.
template <typename Kernel>
unsigned unpack_grid(Kernel kernel, int64_t nchunks, int sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kUnpackBlock, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (nchunks + kUnpackBlock - 1) / kUnpackBlock;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<unsigned>(want < cap ? want : cap);
}

int check_dims(int dtype, int64_t rows, int64_t cols) {
  if (dtype != MXQ_F32 && dtype != MXQ_BF16) return MXQ_EBADDTYPE;
  if (rows < 0 || cols < 0 || cols % 16 != 0) return MXQ_EBADSHAPE;
  if (cols > 0 && rows > (INT64_MAX / 8) / cols) return MXQ_EBADSHAPE;
  return MXQ_OK;
}

template <bool kBF16>
cudaError_t launch_pack(const void* x, int64_t nb, int8_t* q, uint8_t* max_exp, uint8_t* prime,
                        int sms, int dev, cudaStream_t stream) {
  using S = PackShape<kBF16>;
  static bool attr_done[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {  // benign race: setting the same attribute twice is harmless
    const cudaError_t e = cudaFuncSetAttribute(
        mx9_pack_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t nchunks = (nb + S::kBlocksPerStage - 1) / S::kBlocksPerStage;
  const int64_t cap = static_cast<int64_t>(sms) * MXQ_MX9_PACK_CTAS_PER_SM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nchunks < cap ? nchunks : cap));
  cfg.blockDim = dim3(S::kThreads);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, mx9_pack_kernel<kBF16>, static_cast<const uint8_t*>(x), nb,
                            reinterpret_cast<uint4*>(q), max_exp, prime);
}

}  // namespace

namespace mxq {
// Read (and optionally clear) this file's status word; used by mxq_device_status.
int mx9_status_read(unsigned int* out, bool clear) {
  if (cudaMemcpyFromSymbol(out, g_mx9_status, sizeof *out) != cudaSuccess) return MXQ_ECUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_mx9_status, &zero, sizeof zero) != cudaSuccess) return MXQ_ECUDA;
  }
  return MXQ_OK;
}
}  // namespace mxq

extern "C" int mx9_pack(const void* x, int dtype, int64_t rows, int64_t cols, int8_t* q,
                        uint8_t* max_exp, uint8_t* prime, cudaStream_t stream) {
  int rc = check_dims(dtype, rows, cols);
  if (rc != MXQ_OK) return rc;
  const int64_t n = rows * cols;
  if (n == 0) return MXQ_OK;
  if (!x || !q || !max_exp || !prime) return MXQ_ENULL;
  if (!aligned_to(x, 16) || !aligned_to(q, 16)) return MXQ_EALIGN;
  const uint64_t esize = dtype == MXQ_F32 ? 4 : 2;
  const ByteRange r[4] = {
      {reinterpret_cast<uintptr_t>(x), esize * static_cast<uint64_t>(n)},
      {reinterpret_cast<uintptr_t>(q), static_cast<uint64_t>(n)},
      {reinterpret_cast<uintptr_t>(max_exp), static_cast<uint64_t>(n / 16)},
      {reinterpret_cast<uintptr_t>(prime), static_cast<uint64_t>(n / 16)},
  };
  if (ranges_overlap(r, 4)) return MXQ_EOVERLAP;
  int dev = 0;
  const int sms = sm_count_current_device(&dev);
  if (sms <= 0) return MXQ_ECUDA;
  const cudaError_t e = dtype == MXQ_F32
                            ? launch_pack<false>(x, n / 16, q, max_exp, prime, sms, dev, stream)
                            : launch_pack<true>(x, n / 16, q, max_exp, prime, sms, dev, stream);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}

extern "C" int mx9_unpack(const int8_t* q, const uint8_t* max_exp, const uint8_t* prime, void* y,
                          int dtype, int64_t rows, int64_t cols, cudaStream_t stream) {
  int rc = check_dims(dtype, rows, cols);
  if (rc != MXQ_OK) return rc;
  const int64_t n = rows * cols;
  if (n == 0) return MXQ_OK;
  if (!q || !max_exp || !prime || !y) return MXQ_ENULL;
  if (!aligned_to(y, 16) || !aligned_to(q, 16)) return MXQ_EALIGN;
  const uint64_t esize = dtype == MXQ_F32 ? 4 : 2;
  const ByteRange r[4] = {
      {reinterpret_cast<uintptr_t>(y), esize * static_cast<uint64_t>(n)},
      {reinterpret_cast<uintptr_t>(q), static_cast<uint64_t>(n)},
      {reinterpret_cast<uintptr_t>(max_exp), static_cast<uint64_t>(n / 16)},
      {reinterpret_cast<uintptr_t>(prime), static_cast<uint64_t>(n / 16)},
  };
  if (ranges_overlap(r, 4)) return MXQ_EOVERLAP;
  const int sms = sm_count_current_device(nullptr);
  if (sms <= 0) return MXQ_ECUDA;

  const int64_t nchunks = n / (dtype == MXQ_F32 ? UnpackLane<false>::kElems : UnpackLane<true>::kElems);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dtype == MXQ_F32 ? unpack_grid(mx9_unpack_kernel<false>, nchunks, sms)
                                      : unpack_grid(mx9_unpack_kernel<true>, nchunks, sms));
  cfg.blockDim = dim3(kUnpackBlock);
  cfg.stream = stream;
  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(q);
  const cudaError_t e =
      dtype == MXQ_F32
          ? cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<false>, q32, max_exp, prime, y, nchunks)
          : cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<true>, q32, max_exp, prime, y, nchunks);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}
