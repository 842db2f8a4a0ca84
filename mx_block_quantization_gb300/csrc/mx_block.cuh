// mx_block.cuh -- the shared-exponent block rule of MX9 and MX6 for the
// sm_103a kernels.
//
// AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
// pack/unpack" (Summary, "Key design choices"): blocks of 16 elements; the
// exponent byte is the block's largest exponent field; one prime bit per pair
// of elements, set when the pair's exponent is below the block's; scale
// exponent k = max(E - kOff - prime, -126); q = clamp(round_half_even(x / 2^k),
// -kQMax, kQMax).  MX9: kOff 6, kQMax 127 (int8).  MX6: the same rule with four
// magnitude bits, kOff 3, kQMax 15 (5-bit two's-complement codes).
//
// Finite blocks round with one FMA: for |v| < 2^22, 1.5 * 2^23 + v rounds once,
// half to even, to an integer whose two's-complement value is the low 16 bits
// of the result (a finite block gives |x / 2^k| < 2^8).  Two elements are then
// clamped at once as an int16 pair.  MX6 blocks of bf16 round in packed bf16
// instead (q_pair_bf16x2).  Blocks holding Inf or NaN (exponent field 255) take
// the general path: cvt.rni gives 0 for NaN and saturates +-Inf.
#pragma once

#include <stdint.h>

#include "mxq.h"
#include "mxq_device.cuh"

namespace mxq {

__device__ __forceinline__ float fma_rn_noftz(float a, float b, float c) {
  float r;
  asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// a * b + c (mod 2^32) as one integer multiply-add
__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

template <int kOff, int kQMax>
struct MxRule {
  static constexpr uint32_t kClampLo = static_cast<uint32_t>(static_cast<uint16_t>(-kQMax)) * 0x10001u;
  static constexpr uint32_t kClampHi = static_cast<uint32_t>(kQMax) * 0x10001u;
  // bf16 input of a 5-bit format: one packed bf16 FMA per pair (q_pair_bf16x2)
  static constexpr bool kPackedBf16 = kQMax == 15;

  // 2^-k of a pair from the block's exponent field eb8 (E = eb8 - 127) and the
  // pair's prime bit t: 127 - k = min(254 + kOff - eb8 + t, 253).
  static __device__ __forceinline__ float multiplier(uint32_t eb8, uint32_t t) {
    return __uint_as_float(min(254u + kOff - eb8 + t, 253u) << 23);
  }

  static __device__ __forceinline__ uint32_t clamp_pair(uint32_t h) {
    asm("max.s16x2 %0, %0, %1;" : "+r"(h) : "r"(kClampLo));
    asm("min.s16x2 %0, %0, %1;" : "+r"(h) : "r"(kClampHi));
    return h;
  }

  // Two elements of a finite block (fp32 bit patterns) -> clamped int16 pair.
  static __device__ __forceinline__ uint32_t q_pair(uint32_t a, uint32_t b, float mult) {
    const float ra = fma_rn_noftz(__uint_as_float(a), mult, 12582912.0f);
    const float rb = fma_rn_noftz(__uint_as_float(b), mult, 12582912.0f);
    return clamp_pair(__byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x5410));
  }

  // The same on the two bf16 halves of w without widening them: the
  // mixed-precision FMA takes bf16 factors and an fp32 addend and rounds once.
  // mult_bits: the fp32 power-of-two multiplier, exact as bf16 (its high half).
  static __device__ __forceinline__ uint32_t q_pair_bf16(uint32_t w, uint32_t mult_bits) {
    float ra, rb;
    asm("{\n\t.reg .b16 xl, xh, ml, mh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {ml, mh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, xl, mh, %4;\n\t"
        "fma.rn.f32.bf16 %1, xh, mh, %4;\n\t}"
        : "=f"(ra), "=f"(rb)
        : "r"(w), "r"(mult_bits), "f"(12582912.0f));
    return clamp_pair(__byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x5410));
  }

  // MX6 of bf16 (|x / 2^k| < 16 in a finite block): one packed bf16 FMA per
  // pair, against two mixed-precision FMAs and a byte permute.  192 + v stays
  // in the binade [128, 256), where the bf16 step is 1, so x * 2^-k + 192
  // rounds once, half to even, to 192 + round(v); as bits that is
  // 0x4340 + round(v), whose low five bits are the two's-complement code
  // (0x4340 is a multiple of 32).  Only +-16 needs the clamp to +-15.
  // mult2: the power-of-two multiplier as bf16 in both halves.
  static __device__ __forceinline__ uint32_t q_pair_bf16x2(uint32_t w, uint32_t mult2) {
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(mult2), "r"(0x43404340u));
    asm("max.s16x2 %0, %0, %1;" : "+r"(r) : "r"(0x43314331u));  // 192 - 15
    asm("min.s16x2 %0, %0, %1;" : "+r"(r) : "r"(0x434F434Fu));  // 192 + 15
    return r;
  }

  // General path for one element: x * 2^-k (exact, no flush), cvt.rni, clamp.
  static __device__ __forceinline__ uint32_t q_general(uint32_t x, float mult) {
    const int r = __float2int_rn(fmul_rn_noftz(__uint_as_float(x), mult));
    return static_cast<uint32_t>(max(-kQMax, min(kQMax, r))) & 0xFFFFu;
  }

  // 16 fp32 bit patterns -> 8 clamped int16 pairs (pair p = elements 2p, 2p+1),
  // exponent byte and prime byte (bit p = pair p).
  static __device__ __forceinline__ void block_f32(const uint32_t* f, uint32_t* h,
                                                   uint32_t* eb8_out, uint32_t* bits_out) {
    uint32_t pe[8], eb = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      pe[p] = max(f[2 * p] & 0x7F800000u, f[2 * p + 1] & 0x7F800000u);
      eb = max(eb, pe[p]);
    }
    const uint32_t eb8 = eb >> 23;
    const float m0 = multiplier(eb8, 0u), m1 = multiplier(eb8, 1u);
    uint32_t bits = 0;
    if (eb8 != 255u) {
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t t = pe[p] < eb;
        bits |= t << p;
        h[p] = q_pair(f[2 * p], f[2 * p + 1], t ? m1 : m0);
      }
    } else {
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint32_t t = pe[p] < eb;
        bits |= t << p;
        const float m = t ? m1 : m0;
        h[p] = q_general(f[2 * p], m) | (q_general(f[2 * p + 1], m) << 16);
      }
    }
    *eb8_out = eb8;
    *bits_out = bits;
  }

  // 16 bf16 elements as 8 words (word p = pair p, element 2p in the low half)
  // -> h as in block_f32, except that for a finite MX6 block each half of h
  // is 192 + q as bf16 bits, whose low five bits are the code.
  // Exponent fields are compared in place, two per word: with e16 = block
  // field << 7, the low half of (w & 0x7F80) + 0x8000 - e16 reaches bit 15
  // exactly when the element's field is >= the block's, likewise the high
  // half at bit 31 (the low half cannot carry); a pair is demoted when
  // neither bit is set.
  static __device__ __forceinline__ void block_bf16(const uint32_t* w, uint32_t* h,
                                                    uint32_t* eb8_out, uint32_t* bits_out) {
    uint32_t m[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) m[p] = w[p] & 0x7F807F80u;
    const uint32_t mx = vmax_u16x2(vmax_u16x2(vmax_u16x2(m[0], m[1]), vmax_u16x2(m[2], m[3])),
                                   vmax_u16x2(vmax_u16x2(m[4], m[5]), vmax_u16x2(m[6], m[7])));
    const uint32_t e16 = max(mx & 0xFFFFu, mx >> 16);
    const uint32_t eb8 = e16 >> 7;
    if (eb8 == 255u) {
      uint32_t f[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        f[2 * k] = w[k] << 16;  // exact widening of each bf16
        f[2 * k + 1] = w[k] & 0xFFFF0000u;
      }
      block_f32(f, h, eb8_out, bits_out);
      return;
    }
    const uint32_t d2 = (0x8000u - e16) * 0x10001u;
    const float m0 = multiplier(eb8, 0u), m1 = multiplier(eb8, 1u);
    const uint32_t mult0 = kPackedBf16 ? (__float_as_uint(m0) >> 16) * 0x10001u : __float_as_uint(m0);
    const uint32_t dmult = (kPackedBf16 ? (__float_as_uint(m1) >> 16) * 0x10001u : __float_as_uint(m1)) - mult0;
    uint32_t bits = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const bool keep = ((m[p] + d2) & 0x80008000u) != 0u;
      const uint32_t t = keep ? 0u : 1u;
      // prime bit and multiplier as integer multiply-adds, off the ALU pipe
      bits = mad_u32(t, 1u << p, bits);
      const uint32_t mult = mad_u32(t, dmult, mult0);
      h[p] = kPackedBf16 ? q_pair_bf16x2(w[p], mult) : q_pair_bf16(w[p], mult);
    }
    *eb8_out = eb8;
    *bits_out = bits;
  }
};

using Mx9Rule = MxRule<6, 127>;
using Mx6Rule = MxRule<3, 15>;

// 8 int16 pairs with values in [-127, 127] -> the 16 int8 bytes.
__device__ __forceinline__ uint4 pairs_to_bytes(const uint32_t* h) {
  return make_uint4(__byte_perm(h[0], h[1], 0x6420), __byte_perm(h[2], h[3], 0x6420),
                    __byte_perm(h[4], h[5], 0x6420), __byte_perm(h[6], h[7], 0x6420));
}


// 8 pairs of 16-bit halves whose low five bits are the 5-bit two's-complement
// codes (an int16 in [-15, 15], or 192 + q as bf16 bits) -> the 80 bits of the
// sixteen codes, element i at bits 5i..5i+4: bits 0-31, 32-63 and
// 64-79 (low half of *hi).  The disjoint fields are summed with multiply-adds,
// which leave the integer ALU pipe (the MX6 bf16 pack's limit) to the rest:
// measured +0.9% over shifts and ORs.
__device__ __forceinline__ void pairs_to_codes5(const uint32_t* h, uint32_t* lo, uint32_t* mid,
                                                uint32_t* hi) {
  uint32_t c[8];  // 10 bits per pair
#pragma unroll
  for (int p = 0; p < 8; ++p) c[p] = (h[p] & 0x1Fu) | ((h[p] >> 11) & 0x3E0u);
  *lo = mad_u32(c[3], 1u << 30, mad_u32(c[2], 1u << 20, mad_u32(c[1], 1u << 10, c[0])));
  *mid = mad_u32(c[6], 1u << 28, mad_u32(c[5], 1u << 18, mad_u32(c[4], 1u << 8, c[3] >> 2)));
  *hi = mad_u32(c[7], 1u << 6, c[6] >> 4);
}

__device__ __forceinline__ void sts16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Copy a warp's staged records (16-byte aligned on both sides, an even
// number of bytes) to global memory: 16-byte units, then 2-byte pieces.
__device__ __forceinline__ void copy_records_out(uint8_t* g, uint32_t s, uint32_t bytes, int lane) {
  const uint32_t n16 = bytes >> 4;
  for (uint32_t i = lane; i < n16; i += 32) __stcs(reinterpret_cast<uint4*>(g) + i, lds128(s + 16u * i));
  const uint32_t h0 = n16 * 8u, nh = bytes >> 1;
  for (uint32_t i = h0 + lane; i < nh; i += 32) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(s + 2u * i));
    reinterpret_cast<uint16_t*>(g)[i] = static_cast<uint16_t>(v);
  }
}

// Stage one block record at shared address a: [exponent, prime, data].
template <int kFmt>
__device__ __forceinline__ void stage_record(uint32_t a, uint32_t eb8, uint32_t bits,
                                             const uint32_t* h) {
  const uint32_t head = mad_u32(bits, 256u, eb8);  // eb8 | bits << 8
  if (kFmt == MXQ_FMT_MX9) {  // 18 bytes at a 2-byte aligned address
    const uint4 q = pairs_to_bytes(h);
    const uint32_t w[5] = {head | (q.x << 16), __byte_perm(q.x, q.y, 0x5432),
                           __byte_perm(q.y, q.z, 0x5432), __byte_perm(q.z, q.w, 0x5432), q.w >> 16};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      sts16(a + 4u * k, w[k] & 0xFFFFu);
      sts16(a + 4u * k + 2u, w[k] >> 16);
    }
    sts16(a + 16u, w[4]);
  } else {  // MX6: 12 bytes at a 4-byte aligned address
    uint32_t lo, mid, hi;
    pairs_to_codes5(h, &lo, &mid, &hi);
    sts32(a, mad_u32(lo, 1u << 16, head));  // head | lo << 16
    sts32(a + 4u, (lo >> 16) | (mid << 16));
    sts32(a + 8u, (mid >> 16) | (hi << 16));
  }
}

}  // namespace mxq
