// mx9.cu -- MX9 pack / unpack for sm_103a.
//
// Method: AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
// pack/unpack" (Summary, "Key design choices", review thread): blocks of 16
// elements along the last axis; shared E8M0 exponent E = the block's largest
// element exponent from the native bits; one prime bit per pair of elements
// (set when the pair's exponent is below E); scale exponent
// k = max(E - 6 - prime, -126); q = clamp(round_half_even(x / 2^k), -127, 127).
//
// Both kernels are streaming and HBM-bound: one full wave of resident blocks
// walks 16-byte chunks with several independent chunks in flight per thread;
// groups of neighbouring lanes that share a block (4 lanes for fp32 data, 2
// for bf16 data) combine exponents and prime bits with shuffles, so every
// load and store of a warp covers contiguous bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxq.h"
#include "mxq_device.cuh"
#include "mxq_host.h"

namespace {

using namespace mxq;

// Launch shape.  The defaults are the measured best on GB300; the macros only
// exist so that other shapes can be built for measurement.
#ifndef MXQ_MX9_UNROLL
#define MXQ_MX9_UNROLL 4
#endif
#ifndef MXQ_MX9_UNPACK_UNROLL
#define MXQ_MX9_UNPACK_UNROLL 4
#endif
#ifndef MXQ_MX9_PACK_MINBLOCKS
#define MXQ_MX9_PACK_MINBLOCKS 4
#endif
constexpr int kBlock = 256;
constexpr int kUnroll = MXQ_MX9_UNROLL;              // pack: 16-byte input chunks in flight
constexpr int kUnrollUnpack = MXQ_MX9_UNPACK_UNROLL;  // unpack: chunks per thread per iteration

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 2^e as fp32 for e in the normal range [-126, 127].
__device__ __forceinline__ float exp2_normal(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// round_half_even(v) clamped to [-127, 127]; NaN -> 0, +-Inf -> +-127.
__device__ __forceinline__ uint32_t q_byte(float v) {
  int r = __float2int_rn(v);  // cvt.rni.s32.f32: ties to even, NaN -> 0, saturating
  r = max(-127, min(127, r));
  return static_cast<uint32_t>(r) & 0xFFu;
}

// x / 2^k as an exact multiply by 2^-k (k in [-126, 122] makes 2^-k normal).
__device__ __forceinline__ uint32_t quant_elem(float x, int k) {
  return q_byte(fmul_rn_noftz(x, exp2_normal(-k)));
}

// ---------------------------------------------------------------------------
// pack, fp32 input: 4 lanes per 16-element block, 4 elements per lane
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock, MXQ_MX9_PACK_MINBLOCKS) mx9_pack_f32_kernel(const uint4* __restrict__ x,
                                                              int64_t nchunks,
                                                              uint32_t* __restrict__ q,
                                                              uint8_t* __restrict__ max_exp,
                                                              uint8_t* __restrict__ prime) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x - lane);
  for (int64_t base = warp0; base < nchunks; base += stride * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      v[u] = c < nchunks ? ldg_stream(x + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      const uint32_t b0 = (v[u].x >> 23) & 0xFF, b1 = (v[u].y >> 23) & 0xFF;
      const uint32_t b2 = (v[u].z >> 23) & 0xFF, b3 = (v[u].w >> 23) & 0xFF;
      const uint32_t p0 = max(b0, b1), p1 = max(b2, b3);
      uint32_t eb = max(p0, p1);
      eb = max(eb, __shfl_xor_sync(0xFFFFFFFFu, eb, 1));
      eb = max(eb, __shfl_xor_sync(0xFFFFFFFFu, eb, 2));  // biased E of the block
      const uint32_t t0 = p0 < eb, t1 = p1 < eb;
      const int E = static_cast<int>(eb) - 127;
      const int k0 = max(E - 6 - static_cast<int>(t0), -126);
      const int k1 = max(E - 6 - static_cast<int>(t1), -126);
      const uint32_t word = quant_elem(__uint_as_float(v[u].x), k0) |
                            (quant_elem(__uint_as_float(v[u].y), k0) << 8) |
                            (quant_elem(__uint_as_float(v[u].z), k1) << 16) |
                            (quant_elem(__uint_as_float(v[u].w), k1) << 24);
      uint32_t bits = (t0 | (t1 << 1)) << (2 * (lane & 3));
      bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
      bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
      if (c < nchunks) {
        __stcs(q + c, word);
        if ((lane & 3) == 0) {
          max_exp[c >> 2] = static_cast<uint8_t>(eb);
          prime[c >> 2] = static_cast<uint8_t>(bits);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// pack, bf16 input: 2 lanes per block, 8 elements per lane
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock, MXQ_MX9_PACK_MINBLOCKS) mx9_pack_bf16_kernel(const uint4* __restrict__ x,
                                                               int64_t nchunks,
                                                               uint2* __restrict__ q,
                                                               uint8_t* __restrict__ max_exp,
                                                               uint8_t* __restrict__ prime) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x - lane);
  for (int64_t base = warp0; base < nchunks; base += stride * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      v[u] = c < nchunks ? ldg_stream(x + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * stride + lane;
      const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t pe[4];  // biased exponent of each pair (one word = one pair)
#pragma unroll
      for (int i = 0; i < 4; ++i) pe[i] = max((wd[i] >> 7) & 0xFF, (wd[i] >> 23) & 0xFF);
      uint32_t eb = max(max(pe[0], pe[1]), max(pe[2], pe[3]));
      eb = max(eb, __shfl_xor_sync(0xFFFFFFFFu, eb, 1));
      const int E = static_cast<int>(eb) - 127;
      uint32_t tb = 0, lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t t = pe[i] < eb;
        tb |= t << i;
        const int k = max(E - 6 - static_cast<int>(t), -126);
        const uint32_t pair = quant_elem(bf16_lo_f32(wd[i]), k) |
                              (quant_elem(bf16_hi_f32(wd[i]), k) << 8);
        if (i < 2)
          lo |= pair << (16 * i);
        else
          hi |= pair << (16 * (i - 2));
      }
      uint32_t bits = tb << (4 * (lane & 1));
      bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
      if (c < nchunks) {
        __stcs(q + c, make_uint2(lo, hi));
        if ((lane & 1) == 0) {
          max_exp[c >> 1] = static_cast<uint8_t>(eb);
          prime[c >> 1] = static_cast<uint8_t>(bits);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// unpack: 4 lanes per block, 4 elements per lane; fp32 or bf16 output
// ---------------------------------------------------------------------------
template <bool kBF16>
__global__ void __launch_bounds__(kBlock) mx9_unpack_kernel(const uint32_t* __restrict__ q,
                                                            const uint8_t* __restrict__ max_exp,
                                                            const uint8_t* __restrict__ prime,
                                                            void* __restrict__ y,
                                                            int64_t nchunks) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x - lane);
  for (int64_t base = warp0; base < nchunks; base += stride * kUnrollUnpack) {
    uint32_t qv[kUnrollUnpack], ev[kUnrollUnpack], pv[kUnrollUnpack];
#pragma unroll
    for (int u = 0; u < kUnrollUnpack; ++u) {
      const int64_t c = base + u * stride + lane;
      if (c < nchunks) {
        qv[u] = __ldcs(q + c);
        ev[u] = __ldg(max_exp + (c >> 2));
        pv[u] = __ldg(prime + (c >> 2));
      } else {
        qv[u] = ev[u] = pv[u] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnrollUnpack; ++u) {
      const int64_t c = base + u * stride + lane;
      if (c >= nchunks) continue;
      const int E = static_cast<int>(ev[u]) - 127;
      const int pbits = static_cast<int>(pv[u] >> (2 * (lane & 3)));
      const float s0 = exp2_normal(max(E - 6 - (pbits & 1), -126));
      const float s1 = exp2_normal(max(E - 6 - ((pbits >> 1) & 1), -126));
      const float y0 = static_cast<float>(static_cast<int8_t>(qv[u] & 0xFF)) * s0;
      const float y1 = static_cast<float>(static_cast<int8_t>((qv[u] >> 8) & 0xFF)) * s0;
      const float y2 = static_cast<float>(static_cast<int8_t>((qv[u] >> 16) & 0xFF)) * s1;
      const float y3 = static_cast<float>(static_cast<int8_t>(qv[u] >> 24)) * s1;
      if (kBF16) {
        // q * 2^k has at most 7 significant bits: the top half of the fp32 is
        // the exact bf16 (Inf included)
        const uint32_t lo = (__float_as_uint(y0) >> 16) | (__float_as_uint(y1) & 0xFFFF0000u);
        const uint32_t hi = (__float_as_uint(y2) >> 16) | (__float_as_uint(y3) & 0xFFFF0000u);
        __stcs(reinterpret_cast<uint2*>(y) + c, make_uint2(lo, hi));
      } else {
        __stcs(reinterpret_cast<float4*>(y) + c, make_float4(y0, y1, y2, y3));
      }
    }
  }
}

// One full wave: as many resident blocks as the kernel's occupancy allows on
// every SM, or fewer when the problem is small.
template <typename Kernel>
unsigned grid_for(Kernel kernel, int64_t nchunks, int sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBlock, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (nchunks + kBlock - 1) / kBlock;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<unsigned>(want < cap ? want : cap);
}

int check_dims(int dtype, int64_t rows, int64_t cols) {
  if (dtype != MXQ_F32 && dtype != MXQ_BF16) return MXQ_EBADDTYPE;
  if (rows < 0 || cols < 0 || cols % 16 != 0) return MXQ_EBADSHAPE;
  if (cols > 0 && rows > (INT64_MAX / 8) / cols) return MXQ_EBADSHAPE;
  return MXQ_OK;
}

}  // namespace

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
  const int sms = sm_count_current_device(nullptr);
  if (sms <= 0) return MXQ_ECUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kBlock);
  cfg.stream = stream;
  cudaError_t e;
  if (dtype == MXQ_F32) {
    const int64_t nchunks = n / 4;
    cfg.gridDim = dim3(grid_for(mx9_pack_f32_kernel, nchunks, sms));
    e = cudaLaunchKernelEx(&cfg, mx9_pack_f32_kernel, static_cast<const uint4*>(x), nchunks,
                           reinterpret_cast<uint32_t*>(q), max_exp, prime);
  } else {
    const int64_t nchunks = n / 8;
    cfg.gridDim = dim3(grid_for(mx9_pack_bf16_kernel, nchunks, sms));
    e = cudaLaunchKernelEx(&cfg, mx9_pack_bf16_kernel, static_cast<const uint4*>(x), nchunks,
                           reinterpret_cast<uint2*>(q), max_exp, prime);
  }
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

  const int64_t nchunks = n / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dtype == MXQ_F32 ? grid_for(mx9_unpack_kernel<false>, nchunks, sms)
                                      : grid_for(mx9_unpack_kernel<true>, nchunks, sms));
  cfg.blockDim = dim3(kBlock);
  cfg.stream = stream;
  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(q);
  const cudaError_t e =
      dtype == MXQ_F32
          ? cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<false>, q32, max_exp, prime, y, nchunks)
          : cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<true>, q32, max_exp, prime, y, nchunks);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}
