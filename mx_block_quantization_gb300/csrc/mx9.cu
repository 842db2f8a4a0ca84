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
// mixed-precision FMA (MX6: one packed bf16 FMA per pair), which keeps the
// integer pipe (the limit for bf16) light.
// The same kernel writes the packed MX9 / MX6 record forms of mx_packed.cu
// (blocked rows read at a pitch: one bulk copy per row piece of a stage),
// staging each warp's 32 records and storing them with one bulk copy.
// unpack: a streaming kernel with a warp for every group of 32-block rounds
// over the whole tensor; each lane decodes whole 16-element blocks (exact
// q * 2^k built without conversion instructions) into a per-warp
// shared-memory stage, from which every store instruction writes 512
// contiguous output bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxq.h"
#include "mx_block.cuh"
#include "mxq_check.cuh"
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
#ifndef MXQ_MX9_REC_F32_WARPS
#define MXQ_MX9_REC_F32_WARPS 12
#endif
#ifndef MXQ_MX9_REC_F32_RING_KB
#define MXQ_MX9_REC_F32_RING_KB 96
#endif
#ifndef MXQ_MX9_REC_BF16_WARPS
#define MXQ_MX9_REC_BF16_WARPS 8
#endif
#ifndef MXQ_MX9_REC_BF16_RING_KB
#define MXQ_MX9_REC_BF16_RING_KB 64
#endif
#ifndef MXQ_MX9_REC_F32_PER_THREAD
#define MXQ_MX9_REC_F32_PER_THREAD 1
#endif
#ifndef MXQ_MX9_REC_BF16_PER_THREAD
#define MXQ_MX9_REC_BF16_PER_THREAD 4
#endif
#ifndef MXQ_MX9_PACK_CTAS_PER_SM
#define MXQ_MX9_PACK_CTAS_PER_SM 2
#endif
// Waves of resident blocks in the pack's grid (1: one persistent wave; more
// only where every block still gets MXQ_MX9_PACK_MIN_STAGES stages).
// Measured at 16384x8192 / 32768x16384 (fraction of the measured copy
// rate): the split bf16 pack 0.987 / 0.955 with one wave, 0.983-0.999 /
// 1.028-1.031 with 16; every other form was fastest with one (16 waves: split
// fp32 equal, records 9-21% slower; a block per stage: 20-50% slower).
#ifndef MXQ_MX9_PACK_WAVES_SPLIT_BF16
#define MXQ_MX9_PACK_WAVES_SPLIT_BF16 16
#endif
#ifndef MXQ_MX9_PACK_WAVES
#define MXQ_MX9_PACK_WAVES 1
#endif
#ifndef MXQ_MX9_PACK_MIN_STAGES
#define MXQ_MX9_PACK_MIN_STAGES 3
#endif
#ifndef MXQ_MX9_PACK_BF16_PER_THREAD
#define MXQ_MX9_PACK_BF16_PER_THREAD 2
#endif
#ifndef MXQ_MX9_PACK_F32_PER_THREAD
#define MXQ_MX9_PACK_F32_PER_THREAD 1
#endif
#ifndef MXQ_MX9_UNPACK_PRMT_F32
#define MXQ_MX9_UNPACK_PRMT_F32 0
#endif
#ifndef MXQ_MX9_UNPACK_PRMT_BF16
#define MXQ_MX9_UNPACK_PRMT_BF16 1
#endif
// Rounds of 32 blocks a warp of the unpack decodes (its loads all issued
// before the first decode).  Measured with the grid below at 16384x8192 and
// 32768x16384: fp32 1 or 2 alike (1.04-1.05 of the measured copy rate), 4
// slower; bf16 2 best (1.045-1.067), 4 and 8 slower.
#ifndef MXQ_MX9_UNPACK_UNROLL_F32
#define MXQ_MX9_UNPACK_UNROLL_F32 1
#endif
#ifndef MXQ_MX9_UNPACK_UNROLL_BF16
#define MXQ_MX9_UNPACK_UNROLL_BF16 2
#endif

constexpr int kUnpackBlock = 256;

// Sticky status word of this file's kernels (MXQ_DEV_* bits).
__device__ unsigned int g_mx9_status = 0;

// Output forms of the pack kernel: the split tensors (q, max_exp, prime), or
// one packed tensor of block records (MX9: 18 bytes, MX6: 12 bytes).
enum PackOut { kSplit = 0, kRecMx9 = MXQ_FMT_MX9, kRecMx6 = MXQ_FMT_MX6 };

// Pack kernel shape per input type: consumer warps (kPerThread 16-element
// blocks per consumer thread and stage), one producer warp, a ring of stages,
// and for record outputs a per-warp staging area of 32 records.  Rings deeper
// than these measured slower; the record forms, with more instructions per
// block, measured faster with more warps.
template <bool kBF16, int kOut>
struct PackShape {
  static constexpr int kWarps =
      kOut == kSplit ? (kBF16 ? MXQ_MX9_PACK_BF16_WARPS : MXQ_MX9_PACK_F32_WARPS)
                     : (kBF16 ? MXQ_MX9_REC_BF16_WARPS : MXQ_MX9_REC_F32_WARPS);
  static constexpr int kPerThread =
      kOut == kSplit ? (kBF16 ? MXQ_MX9_PACK_BF16_PER_THREAD : MXQ_MX9_PACK_F32_PER_THREAD)
                     : (kBF16 ? MXQ_MX9_REC_BF16_PER_THREAD : MXQ_MX9_REC_F32_PER_THREAD);
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kBlocksPerStage = kConsumers * kPerThread;
  static constexpr uint32_t kBlockBytes = kBF16 ? 32u : 64u;  // 16 elements
  static constexpr uint32_t kStageBytes = kBlocksPerStage * kBlockBytes;
  static constexpr uint32_t kRingBytes =
      (kOut == kSplit ? (kBF16 ? MXQ_MX9_PACK_BF16_RING_KB : MXQ_MX9_PACK_F32_RING_KB)
                      : (kBF16 ? MXQ_MX9_REC_BF16_RING_KB : MXQ_MX9_REC_F32_RING_KB)) *
      1024u;
  static constexpr int kStages = static_cast<int>(kRingBytes / kStageBytes);
  static constexpr int kWaves =
      kOut == kSplit && kBF16 ? MXQ_MX9_PACK_WAVES_SPLIT_BF16 : MXQ_MX9_PACK_WAVES;
  static constexpr uint32_t kRecord =
      kOut == kRecMx9 ? MXQ_MX9_RECORD_BYTES : kOut == kRecMx6 ? MXQ_MX6_RECORD_BYTES : 0u;
  static constexpr uint32_t kOffBar = kStages * kStageBytes;
  static constexpr uint32_t kOffFlag = kOffBar + 16u * kStages;
  static constexpr uint32_t kOffRec = kOffFlag + 16u;
  // record outputs: a warp owns kPerThread * 32 consecutive blocks of a stage
  static constexpr int kWarpBlocks = 32 * kPerThread;
  static constexpr uint32_t kWarpRecBytes = kWarpBlocks * kRecord;
  static constexpr uint32_t kSmemBytes = kOffRec + kWarps * 2u * kWarpRecBytes + 128u;  // + alignment
  static_assert(kStages >= 2, "ring too small");
  static_assert(kWarpRecBytes % 16u == 0, "record runs of a warp stay 16-byte aligned");
  static_assert(kSmemBytes * MXQ_MX9_PACK_CTAS_PER_SM <= 227u * 1024u, "shared memory budget");
};

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// x: nb blocks in rows of nbl blocks, rows pitch bytes apart (16-byte aligned
// starts).  kSplit: q [nb, 16] int8, max_exp [nb], prime [nb].  kRecMx9 /
// kRecMx6: out is the packed tensor of nb records (16-byte aligned); q_or_rec
// points to it.
template <bool kBF16, int kOut>
__global__ void __launch_bounds__(PackShape<kBF16, kOut>::kThreads, MXQ_MX9_PACK_CTAS_PER_SM)
    mx9_pack_kernel(const uint8_t* __restrict__ x, int64_t nb, int64_t nbl, int64_t pitch,
                    uint8_t* __restrict__ q_or_rec, uint8_t* __restrict__ max_exp,
                    uint8_t* __restrict__ prime) {
  using S = PackShape<kBF16, kOut>;
  using R = MxRule<kOut == kRecMx6 ? 3 : 6, kOut == kRecMx6 ? 15 : 127>;
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
  pdl_wait();  // x may be the previous kernel's output; outputs may still be read by it
  pdl_trigger_at_start();

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
      const uint32_t dst = base + static_cast<uint32_t>(s) * S::kStageBytes;
      // x: nb / nbl rows of nbl blocks, pitch bytes apart
      const uint64_t x_bytes = static_cast<uint64_t>(nb / nbl - 1) * pitch + nbl * S::kBlockBytes;
      if (pitch == nbl * static_cast<int64_t>(S::kBlockBytes)) {  // rows follow each other
        if (in_buf(x + b0 * S::kBlockBytes, bytes, x, x_bytes, &g_mx9_status))
          bulk_load_1d(dst, x + b0 * S::kBlockBytes, bytes, full(s));
        else
          mbar_complete_tx(full(s), bytes);
      } else {  // one copy per row piece of the stage's blocks
        int64_t row = b0 / nbl, j = b0 - row * nbl;
        for (int64_t b = b0; b < b0 + nblk; ++row, j = 0) {
          const int64_t n = b0 + nblk - b < nbl - j ? b0 + nblk - b : nbl - j;
          const uint32_t nbytes = static_cast<uint32_t>(n) * S::kBlockBytes;
          if (in_buf(x + row * pitch + j * S::kBlockBytes, nbytes, x, x_bytes, &g_mx9_status))
            bulk_load_1d(dst + static_cast<uint32_t>(b - b0) * S::kBlockBytes,
                         x + row * pitch + j * S::kBlockBytes, nbytes, full(s));
          else
            mbar_complete_tx(full(s), nbytes);
          b += n;
        }
      }
      issued = i + 1;
    }
    pdl_trigger_at_end();
    // drain (a no-op after a normal run: consumers waited for every stage)
    for (int64_t i = issued > S::kStages ? issued - S::kStages : 0; i < issued; ++i)
      mbar_wait_drain(full(static_cast<int>(i % S::kStages)),
                      static_cast<uint32_t>((i / S::kStages) & 1));
    return;
  }

  // -------------------------------------------------------------- consumers
  // Record outputs: a warp takes kWarpBlocks consecutive blocks of each stage,
  // stages their records in one of its two buffers (alternating over stages)
  // and lane 0 writes them with one bulk store.
  const uint32_t rec_stage = base + S::kOffRec + static_cast<uint32_t>(warp) * 2u * S::kWarpRecBytes;
  uint32_t runs = 0;
  for (int64_t i = 0; i < my; ++i) {
    const int s = static_cast<int>(i % S::kStages);
    const bool ok = mbar_wait_bounded(full(s), static_cast<uint32_t>((i / S::kStages) & 1),
                                      abort_flag, &g_mx9_status, MXQ_DEV_TIMEOUT);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    const int64_t blk0 = (blockIdx.x + i * static_cast<int64_t>(gridDim.x)) * S::kBlocksPerStage;
    const uint32_t stage_base = base + static_cast<uint32_t>(s) * S::kStageBytes;
    // 16-element block `local` of this stage -> its clamped int16 pairs
    auto quantize = [&](int local, uint32_t* h, uint32_t* eb8, uint32_t* bits) {
      const uint32_t src = stage_base + static_cast<uint32_t>(local) * S::kBlockBytes;
      if (kBF16) {
        const uint4 a = lds128(src), b = lds128(src + 16);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        R::block_bf16(w, h, eb8, bits);
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
        R::block_f32(f, h, eb8, bits);
      }
    };
    if (kOut == kSplit) {
#pragma unroll
      for (int j = 0; j < S::kPerThread; ++j) {
        const int local = j * S::kConsumers + tid;
        const int64_t blk = blk0 + local;
        if (blk >= nb) break;
        uint32_t h[8], eb8, bits;
        quantize(local, h, &eb8, &bits);
        if (in_buf(q_or_rec + 16 * blk, 16, q_or_rec, 16ull * nb, &g_mx9_status))
          __stcs(reinterpret_cast<uint4*>(q_or_rec) + blk, pairs_to_bytes(h));
        if (in_buf(max_exp + blk, 1, max_exp, nb, &g_mx9_status))
          max_exp[blk] = static_cast<uint8_t>(eb8);
        if (in_buf(prime + blk, 1, prime, nb, &g_mx9_status))
          prime[blk] = static_cast<uint8_t>(bits);
      }
    } else {
      const int64_t wrun0 = blk0 + static_cast<int64_t>(warp) * S::kWarpBlocks;
      if (wrun0 < nb) {  // warp-uniform
        const uint32_t buf = rec_stage + (runs & 1u) * S::kWarpRecBytes;
        ++runs;
        if (lane == 0) bulk_wait_read<1>();  // the store that last read buf is done with it
        __syncwarp();
#pragma unroll
        for (int j = 0; j < S::kPerThread; ++j) {
          const int r = j * 32 + lane;  // record of this warp's run
          if (wrun0 + r < nb) {
            uint32_t h[8], eb8, bits;
            quantize(warp * S::kWarpBlocks + r, h, &eb8, &bits);
            stage_record<kOut>(buf + static_cast<uint32_t>(r) * S::kRecord, eb8, bits, h);
          }
        }
        const int64_t nvalid = nb - wrun0 < S::kWarpBlocks ? nb - wrun0 : S::kWarpBlocks;
        const uint32_t bytes = static_cast<uint32_t>(nvalid) * S::kRecord;
        if (!in_buf(q_or_rec + wrun0 * S::kRecord, bytes, q_or_rec,
                    static_cast<uint64_t>(nb) * S::kRecord, &g_mx9_status)) {
          __syncwarp();
        } else if (bytes % 16u == 0) {
          fence_proxy_async_smem();  // staged records before the bulk store reads them
          __syncwarp();
          if (lane == 0) {
            bulk_store(q_or_rec + wrun0 * S::kRecord, buf, bytes);
            bulk_commit();
          }
        } else {  // the tensor's last, partial run
          __syncwarp();
          copy_records_out(q_or_rec + wrun0 * S::kRecord, buf, bytes, lane);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }
  pdl_trigger_at_end();
  if (kOut != kSplit && lane == 0) bulk_wait_all<0>();
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

// Unpack: a lane decodes whole 16-element blocks, one per round: one 16-byte
// load of q plus the block's own exponent and prime bytes (a warp's loads of a
// round are 512 contiguous q bytes and 32 contiguous bytes of each of the
// others), the loads of all kUnroll rounds issued before the first decode.
// The decoded block (64 bytes of fp32 or 32 of bf16) goes to a per-warp
// staging buffer in shared memory, from which each lane stores 16-byte pieces
// so that every store instruction writes 512 contiguous output bytes.  A warp
// takes kUnroll consecutive rounds and the grid has a warp for every group of
// them: blocks are scheduled as earlier ones leave, which measured 10-15%
// faster than one persistent wave of resident blocks walking the tensor.
// q * 2^k is exact (|q| <= 127, k >= -126) except for overflow in max_exp
// 255 blocks; a bf16 result has at most 7 significant bits, so the top half
// of the fp32 is the exact bf16.
template <bool kBF16>
struct UnpackShape {
  static constexpr int kChunks = kBF16 ? 2 : 4;  // 16-byte output pieces per block
  static constexpr int kUnroll = kBF16 ? MXQ_MX9_UNPACK_UNROLL_BF16 : MXQ_MX9_UNPACK_UNROLL_F32;
  static constexpr int kWarps = kUnpackBlock / 32;
  static constexpr int kGroup = 32 * kUnroll;                   // blocks per warp
  static constexpr uint32_t kStageBytes = 32u * kChunks * 16u;  // one round of a warp
};

// Slot of output piece c (piece c % kChunks of the round's block c / kChunks)
// in a warp's staging buffer.  XOR-ing bits 3.. of c into its low bits makes
// both access patterns conflict-free: the writes, where lane l stores the
// pieces of its own block, and the reads, where lane l loads piece 32r + l.
template <bool kBF16>
__device__ __forceinline__ uint32_t unpack_slot(int c) {
  return static_cast<uint32_t>(kBF16 ? c ^ ((c >> 3) & 1) : c ^ ((c >> 3) & 3));
}

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
    const uint4* __restrict__ q, const uint8_t* __restrict__ max_exp,
    const uint8_t* __restrict__ prime, uint4* __restrict__ y, int64_t nb) {
  using U = UnpackShape<kBF16>;
  __shared__ __align__(16) uint8_t stage[U::kWarps][U::kStageBytes];
  pdl_wait();
  pdl_trigger_at_start();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t st = smem_u32(stage[warp]);
  const int64_t gwarps = static_cast<int64_t>(gridDim.x) * U::kWarps;
  // warp gw takes groups gw, gw + gwarps, ... (one group when the grid covers
  // the tensor, as launched)
  for (int64_t g0 = (static_cast<int64_t>(blockIdx.x) * U::kWarps + warp) * U::kGroup; g0 < nb;
       g0 += gwarps * U::kGroup) {
    uint4 qv[U::kUnroll];
    uint32_t ev[U::kUnroll], pv[U::kUnroll];
#pragma unroll
    for (int u = 0; u < U::kUnroll; ++u) {
      const int64_t b = g0 + 32 * u + lane;
      qv[u] = make_uint4(0u, 0u, 0u, 0u);
      ev[u] = pv[u] = 0u;
      if (b < nb && in_buf(q + b, 16, q, 16ull * nb, &g_mx9_status) &&
          in_buf(max_exp + b, 1, max_exp, nb, &g_mx9_status) &&
          in_buf(prime + b, 1, prime, nb, &g_mx9_status)) {
        qv[u] = __ldcs(q + b);
        ev[u] = __ldg(max_exp + b);
        pv[u] = __ldg(prime + b);
      }
    }
#pragma unroll
    for (int u = 0; u < U::kUnroll; ++u) {
      const int64_t bu = g0 + 32 * u;  // first block of the round (warp-uniform)
      if (bu >= nb) break;
      const int E = static_cast<int>(ev[u]) - 127;
      const uint32_t w[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
      float v[16];  // word k holds elements 4k..4k+3, i.e. pairs 2k and 2k+1
      if (kBF16 ? MXQ_MX9_UNPACK_PRMT_BF16 : MXQ_MX9_UNPACK_PRMT_F32) {
        // the two possible pair scales, then one select per pair
        const float s_keep = exp2_normal(max(E - 6, -126)), s_dem = exp2_normal(max(E - 7, -126));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          unpack4_biased(w[k] ^ 0x80808080u, (pv[u] >> (2 * k)) & 1u ? s_dem : s_keep,
                         (pv[u] >> (2 * k + 1)) & 1u ? s_dem : s_keep, v + 4 * k);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          unpack4(w[k], exp2_normal(max(E - 6 - static_cast<int>((pv[u] >> (2 * k)) & 1u), -126)),
                  exp2_normal(max(E - 6 - static_cast<int>((pv[u] >> (2 * k + 1)) & 1u), -126)),
                  v + 4 * k);
      }
#pragma unroll
      for (int j = 0; j < U::kChunks; ++j) {
        const uint32_t a = st + 16u * unpack_slot<kBF16>(U::kChunks * lane + j);
        if (kBF16) {  // the high halves of fp32 pairs
          const float* h = v + 8 * j;
          sts128(a, __byte_perm(__float_as_uint(h[0]), __float_as_uint(h[1]), 0x7632),
                 __byte_perm(__float_as_uint(h[2]), __float_as_uint(h[3]), 0x7632),
                 __byte_perm(__float_as_uint(h[4]), __float_as_uint(h[5]), 0x7632),
                 __byte_perm(__float_as_uint(h[6]), __float_as_uint(h[7]), 0x7632));
        } else {
          sts128(a, __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                 __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
        }
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < U::kChunks; ++r) {
        const int c = 32 * r + lane;
        const uint4 o = lds128(st + 16u * unpack_slot<kBF16>(c));
        const int64_t piece = bu * U::kChunks + c;
        if (bu + c / U::kChunks < nb &&
            in_buf(y + piece, 16, y, 16ull * U::kChunks * nb, &g_mx9_status))
          __stcs(y + piece, o);
      }
      __syncwarp();  // the buffer is rewritten by the next round
    }
  }
  pdl_trigger_at_end();
}

// A warp for every kGroup blocks (grid capped at the hardware's limit).
template <bool kBF16>
unsigned unpack_grid(int64_t nb) {
  using U = UnpackShape<kBF16>;
  const int64_t warps = (nb + U::kGroup - 1) / U::kGroup;
  const int64_t want = (warps + U::kWarps - 1) / U::kWarps;
  return static_cast<unsigned>(want < INT32_MAX ? want : INT32_MAX);
}

int check_dims(int dtype, int64_t rows, int64_t cols) {
  if (dtype != MXQ_F32 && dtype != MXQ_BF16) return MXQ_EBADDTYPE;
  if (rows < 0 || cols < 0 || cols % 16 != 0) return MXQ_EBADSHAPE;
  if (cols > 0 && rows > (INT64_MAX / 8) / cols) return MXQ_EBADSHAPE;
  return MXQ_OK;
}

template <bool kBF16, int kOut>
cudaError_t launch_pack(const void* x, int64_t nb, int64_t nbl, int64_t pitch, uint8_t* q_or_rec,
                        uint8_t* max_exp, uint8_t* prime, int sms, int dev, cudaStream_t stream) {
  using S = PackShape<kBF16, kOut>;
  static bool attr_done[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {  // benign race: setting the same attribute twice is harmless
    const cudaError_t e = cudaFuncSetAttribute(
        mx9_pack_kernel<kBF16, kOut>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t nchunks = (nb + S::kBlocksPerStage - 1) / S::kBlocksPerStage;
  // one wave of resident blocks, or kWaves whole waves when every block then
  // still gets MXQ_MX9_PACK_MIN_STAGES stages (its ring set-up amortized);
  // a partial last wave measured slower (4096x4096 bf16: 0.80-0.93 against
  // 0.97 for one wave)
  const int64_t wave = static_cast<int64_t>(sms) * MXQ_MX9_PACK_CTAS_PER_SM;
  const int64_t cap =
      nchunks >= wave * S::kWaves * MXQ_MX9_PACK_MIN_STAGES ? wave * S::kWaves : wave;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nchunks < cap ? nchunks : cap));
  cfg.blockDim = dim3(S::kThreads);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  return cudaLaunchKernelEx(&cfg, mx9_pack_kernel<kBF16, kOut>, static_cast<const uint8_t*>(x),
                            nb, nbl, pitch, q_or_rec, max_exp, prime);
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

// The packed-record form of the pack kernel for a contiguous tensor blocked
// along its rows (x and packed 16-byte aligned, nb whole blocks); the caller
// has checked the arguments.
int launch_records_pack(const void* x, bool bf16, int fmt, int64_t nb, int64_t nbl, int64_t pitch,
                        uint8_t* packed, cudaStream_t stream) {
  int dev = 0;
  const int sms = sm_count_current_device(&dev);
  if (sms <= 0) return MXQ_ECUDA;
  cudaError_t e;
  if (fmt == MXQ_FMT_MX9)
    e = bf16 ? launch_pack<true, kRecMx9>(x, nb, nbl, pitch, packed, nullptr, nullptr, sms, dev, stream)
             : launch_pack<false, kRecMx9>(x, nb, nbl, pitch, packed, nullptr, nullptr, sms, dev, stream);
  else
    e = bf16 ? launch_pack<true, kRecMx6>(x, nb, nbl, pitch, packed, nullptr, nullptr, sms, dev, stream)
             : launch_pack<false, kRecMx6>(x, nb, nbl, pitch, packed, nullptr, nullptr, sms, dev, stream);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
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
  uint8_t* qb = reinterpret_cast<uint8_t*>(q);
  const int64_t nb = n / 16;  // one flat run of blocks
  const cudaError_t e =
      dtype == MXQ_F32
          ? launch_pack<false, kSplit>(x, nb, nb, nb * 64, qb, max_exp, prime, sms, dev, stream)
          : launch_pack<true, kSplit>(x, nb, nb, nb * 32, qb, max_exp, prime, sms, dev, stream);
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
  const int64_t nb = n / 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dtype == MXQ_F32 ? unpack_grid<false>(nb) : unpack_grid<true>(nb));
  cfg.blockDim = dim3(kUnpackBlock);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  const uint4* q16 = reinterpret_cast<const uint4*>(q);
  uint4* y16 = static_cast<uint4*>(y);
  const cudaError_t e =
      dtype == MXQ_F32
          ? cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<false>, q16, max_exp, prime, y16, nb)
          : cudaLaunchKernelEx(&cfg, mx9_unpack_kernel<true>, q16, max_exp, prime, y16, nb);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}
