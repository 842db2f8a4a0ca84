// mxq_mma_check.cu -- a block-scaled MXFP8 matrix product on the 5th-generation
// tensor cores that reads the cast's outputs exactly as they are stored: the
// consumer check of the layouts.
//
// pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct
// metadata" (description, first paragraph; "Uncovered tail" paragraph): the
// scale tensors are written in the blocked form that the block-scaled MMA
// reads, the colwise ones as one slab per K-group.  Here tcgen05.mma of kind
// mxf8f6f4 with E8M0 block scales (one scale per 32 K elements) consumes E4M3
// rows together with such blocked scale matrices; feeding it q_row/s_row and a
// group's q_col columns with that group's s_col slab and comparing with the
// product of the decoded values shows that the bytes are where the MMA looks.
//
// Not a production GEMM: one CTA of four warps per 128x128 output tile, K in
// steps of 128 with no overlap between loads and MMAs.
//   * A and B chunks (128 rows x 128 K bytes) are copied into shared memory in
//     the no-swizzle K-major layout of 8-row x 16-byte core matrices (core
//     (r/8, k/16) at (r/8)*1024 + (k/16)*128, rows 16 bytes apart inside it);
//   * a 128x4 scale atom (512 bytes: row r%32 holds 16 bytes, 4 scales of each
//     of the rows r%32 + 32g) goes to tensor memory as the 4-warp broadcast of
//     its 32 rows: lane r, column g holds the 4 scales of row 32g + r%32, so
//     row r finds its own at column r/32, byte = K block;
//   * one thread issues 4 MMAs (K = 32 each, scale byte k selected by the
//     instruction descriptor) and commits them to an mbarrier; the accumulator
//     (128 lanes x 128 fp32 columns) stays in tensor memory until the end.
// Every wait is bounded; on a timeout the kernel records MXQ_DEV_TIMEOUT,
// frees its tensor memory and returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxq.h"
#include "mxq_check.cuh"
#include "mxq_device.cuh"
#include "mxq_host.h"

namespace {

using namespace mxq;

__device__ unsigned int g_mma_status = 0;

constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;     // accumulator 128 columns + scales
constexpr uint32_t kColSfa = 128;       // scale columns of A (4 used)
constexpr uint32_t kColSfb = 160;       // scale columns of B (4 used)
constexpr uint32_t kCoreK = 128;        // bytes between K-adjacent core matrices
constexpr uint32_t kCoreRows = 1024;    // bytes between 8-row groups
// dynamic shared memory that keeps at most two CTAs on an SM, so that their
// tensor-memory allocations (2 x 256 of 512 columns) never wait on each other
constexpr uint32_t kPadSmem = 80 * 1024;

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint4 tmem_ld4(uint32_t taddr) {
  uint4 v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(taddr)
               : "memory");
  return v;
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// D (+)= A * B^T with per-32 E8M0 scales of A and B; A, B K-major E4M3 in
// shared memory (descriptors), D and the scales in tensor memory.
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred acc;\n\t"
      "setp.ne.b32 acc, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], acc;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor: start address, leading (K) and stride (8-row)
// byte offsets, all in 16-byte units; descriptor version 1; no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lead, uint32_t stride) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>(lead >> 4) << 16) | (static_cast<uint64_t>(stride >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind mxf8f6f4 with block scales: E4M3 A and B,
// both K-major, N = 128, M = 128, E8M0 scales, scale byte `k` of A and of B.
__host__ __device__ constexpr uint32_t mxf8_idesc(uint32_t k) {
  return (k << 4)              // scale byte of B
         | (0u << 7)           // A: E4M3
         | (0u << 10)          // B: E4M3
         | ((128u >> 3) << 17) // N / 8
         | (1u << 23)          // scales are E8M0
         | ((128u >> 4) << 24) // M / 16
         | (k << 29);          // scale byte of A
}

// One 128-row chunk (128 K bytes) of a K-major E4M3 matrix into the core-matrix
// layout; rows past `rows` of the matrix cannot occur (rows % 128 == 0).
__device__ __forceinline__ void stage_chunk(uint32_t dst, const uint8_t* src, int64_t ld,
                                            uint64_t src_bytes, const uint8_t* src_base, int tid) {
#pragma unroll 4
  for (int idx = tid; idx < 128 * 8; idx += kThreads) {
    const int r = idx >> 3, p = idx & 7;
    const uint8_t* g = src + r * ld + 16 * p;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (in_buf(g, 16, src_base, src_bytes, &g_mma_status)) v = __ldg(reinterpret_cast<const uint4*>(g));
    sts128(dst + static_cast<uint32_t>(r >> 3) * kCoreRows + static_cast<uint32_t>(p) * kCoreK +
               static_cast<uint32_t>(r & 7) * 16u,
           v.x, v.y, v.z, v.w);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    mxq_mma_check_kernel(const uint8_t* __restrict__ a, int64_t lda, const uint8_t* __restrict__ sa,
                         const uint8_t* __restrict__ b, int64_t ldb, const uint8_t* __restrict__ sb,
                         float* __restrict__ d, int64_t Ma, int64_t Nb, int64_t K) {
  __shared__ __align__(1024) uint8_t tile_a[128 * 128];
  __shared__ __align__(1024) uint8_t tile_b[128 * 128];
  __shared__ uint32_t tmem_base;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t tile_i = blockIdx.y, tile_j = blockIdx.x;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_sel = static_cast<uint32_t>(32 * warp) << 16;  // this warp's lanes
  const int64_t kchunks = K / 128;                                   // scale atoms along K
  const uint64_t a_bytes = static_cast<uint64_t>(Ma - 1) * lda + K;
  const uint64_t b_bytes = static_cast<uint64_t>(Nb - 1) * ldb + K;
  const uint64_t s_bytes_a = static_cast<uint64_t>(Ma) * K / 32;
  const uint64_t s_bytes_b = static_cast<uint64_t>(Nb) * K / 32;
  bool ok = true;
  for (int64_t kc = 0; kc < kchunks; ++kc) {
    stage_chunk(smem_u32(tile_a), a + tile_i * 128 * lda + kc * 128, lda, a_bytes, a, tid);
    stage_chunk(smem_u32(tile_b), b + tile_j * 128 * ldb + kc * 128, ldb, b_bytes, b, tid);
    // scale atoms (row block, K chunk): row lane of the 512 bytes, broadcast to
    // the lanes of all four warps
    const uint8_t* pa = sa + (tile_i * kchunks + kc) * 512 + 16 * lane;
    const uint8_t* pb = sb + (tile_j * kchunks + kc) * 512 + 16 * lane;
    uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
    if (in_buf(pa, 16, sa, s_bytes_a, &g_mma_status)) va = __ldg(reinterpret_cast<const uint4*>(pa));
    if (in_buf(pb, 16, sb, s_bytes_b, &g_mma_status)) vb = __ldg(reinterpret_cast<const uint4*>(pb));
    tmem_st4(tmem + lane_sel + kColSfa, va);
    tmem_st4(tmem + lane_sel + kColSfb, vb);
    tmem_wait_st();
    fence_proxy_async_smem();  // the staged tiles before the MMAs read them
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k) {
        const uint64_t da = smem_desc(smem_u32(tile_a) + 2u * kCoreK * k, kCoreK, kCoreRows);
        const uint64_t db = smem_desc(smem_u32(tile_b) + 2u * kCoreK * k, kCoreK, kCoreRows);
        mma_mxf8(tmem, da, db, mxf8_idesc(k), tmem + kColSfa, tmem + kColSfb, (kc | k) != 0);
      }
      mma_commit(smem_u32(&bar));
    }
    // the MMAs have read the tiles and the scale columns before they are refilled
    ok = mbar_wait_bounded(smem_u32(&bar), static_cast<uint32_t>(kc & 1), &abort_flag,
                           &g_mma_status, MXQ_DEV_TIMEOUT);
    tc_fence_after();
    if (!__syncthreads_and(ok)) break;
  }
  if (ok) {
    // lane l of warp w holds output row 32w + l of the tile
    const int64_t row = tile_i * 128 + 32 * warp + lane;
    float* out = d + row * Nb + tile_j * 128;
    for (uint32_t c = 0; c < 128; c += 4) {
      const uint4 v = tmem_ld4(tmem + lane_sel + c);
      tmem_wait_ld();
      if (in_buf(out + c, 16, d, static_cast<uint64_t>(Ma) * Nb * 4, &g_mma_status))
        *reinterpret_cast<uint4*>(out + c) = v;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace mxq {
int mma_status_read(unsigned int* out, bool clear) {
  if (cudaMemcpyFromSymbol(out, g_mma_status, sizeof *out) != cudaSuccess) return MXQ_ECUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_mma_status, &zero, sizeof zero) != cudaSuccess) return MXQ_ECUDA;
  }
  return MXQ_OK;
}
}  // namespace mxq

extern "C" int mxq_mxfp8_scaled_mm(const uint8_t* a, int64_t lda, const uint8_t* sa,
                                   const uint8_t* b, int64_t ldb, const uint8_t* sb, float* d,
                                   int64_t Ma, int64_t Nb, int64_t K, cudaStream_t stream) {
  if (Ma < 0 || Nb < 0 || K < 0 || Ma % 128 != 0 || Nb % 128 != 0 || K % 128 != 0 ||
      Ma > (int64_t{1} << 24) || Nb > (int64_t{1} << 24) || K > (int64_t{1} << 24))
    return MXQ_EBADSHAPE;
  if (Ma == 0 || Nb == 0) return MXQ_OK;
  // row pitches bounded so that no byte range below can wrap
  if (K == 0 || lda < K || ldb < K || lda % 16 != 0 || ldb % 16 != 0 ||
      lda > (int64_t{1} << 40) || ldb > (int64_t{1} << 40))
    return MXQ_EBADSHAPE;
  if (!a || !sa || !b || !sb || !d) return MXQ_ENULL;
  if (!aligned_to(a, 16) || !aligned_to(sa, 16) || !aligned_to(b, 16) || !aligned_to(sb, 16) ||
      !aligned_to(d, 16))
    return MXQ_EALIGN;
  const ByteRange r[5] = {
      {reinterpret_cast<uintptr_t>(d), static_cast<uint64_t>(Ma) * Nb * 4},
      {reinterpret_cast<uintptr_t>(a), static_cast<uint64_t>(Ma - 1) * lda + K},
      {reinterpret_cast<uintptr_t>(sa), static_cast<uint64_t>(Ma) * K / 32},
      {reinterpret_cast<uintptr_t>(b), static_cast<uint64_t>(Nb - 1) * ldb + K},
      {reinterpret_cast<uintptr_t>(sb), static_cast<uint64_t>(Nb) * K / 32},
  };
  // the output must not overlap an input; the inputs may share storage
  for (int i = 1; i < 5; ++i) {
    const ByteRange two[2] = {r[0], r[i]};
    if (ranges_overlap(two, 2)) return MXQ_EOVERLAP;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MXQ_ECUDA;
  static bool attr_done[64] = {};  // benign race: the same attribute set twice
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(mxq_mma_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPadSmem) != cudaSuccess)
      return MXQ_ECUDA;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(Nb / 128), static_cast<unsigned>(Ma / 128));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPadSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  return cudaLaunchKernelEx(&cfg, mxq_mma_check_kernel, a, lda, sa, b, ldb, sb, d, Ma, Nb, K) ==
                 cudaSuccess
             ? MXQ_OK
             : MXQ_ECUDA;
}
