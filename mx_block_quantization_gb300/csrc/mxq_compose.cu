// mxq_compose.cu -- the K-groups scale swizzle and the three-pass composition.
//
// pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct
// metadata" (description, first paragraph) replaces three kernels: a 1x32
// cast along N, a 32x1 cast along M, and a standalone K-groups swizzle of the
// colwise scales.  This file provides the swizzle and the composed call, so
// the fused kernel can be measured against the composition it replaces on the
// same GPU.  The composition writes the same bytes as the fused cast except in
// colwise blocks that hold NaN: the separate 32x1 cast skips NaN in its amax
// (description, NaN paragraph), the fused one poisons the block.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mxq.h"
#include "mxq_check.cuh"
#include "mxq_device.cuh"
#include "mxq_host.h"

extern "C" int mxq_quantize_1x32(const void* x, int64_t M, int64_t N, uint8_t* q_row,
                                 uint8_t* s_row, cudaStream_t stream);
extern "C" int mxq_quantize_32x1(const void* x, int64_t M, int64_t N, uint8_t* q_col,
                                 uint8_t* s_rm, cudaStream_t stream);

namespace {

using namespace mxq;

constexpr int kSwzThreads = 256;

// Sticky status word of this file's kernels (MXQ_DEV_* bits).
__device__ unsigned int g_compose_status = 0;

// First g with offs[g] > row.
__device__ __forceinline__ int group_of(const int32_t* s_offs, int G, int64_t row) {
  int lo = 0, hi = G;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(s_offs[mid]) > row)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// Every 16-byte unit of s_col is produced by one thread.  s_col is a sequence
// of 512-byte atoms; atom a of group g = [lo, hi) (a' = a - (N/128)*(lo/128)
// inside the group's slab, A = (hi - lo)/128 atoms per 128 rows of n) holds
// the scales of rows n = 128*(a'/A) + r and scale columns lo/32 + 4*(a'%A) + c,
// at byte r%32*16 + (r/32)*4 + c.  A 16-byte unit k (0..31) of the atom is rows
// r = k + 32*{0,1,2,3}, each row contributing its 4 adjacent scale bytes, one
// aligned 32-bit word of the row-major input.  Atoms from (N/128)*(end/128) on
// are the uncovered tail and are written as zeros.
__global__ void __launch_bounds__(kSwzThreads)
    mxq_swizzle_kernel(const uint8_t* __restrict__ s_rm, int64_t N, int64_t M,
                       const int32_t* __restrict__ offs, int G, uint8_t* __restrict__ s_col) {
  __shared__ int32_t s_offs[MXQ_MAX_GROUPS];
  pdl_wait();  // s_rm is the previous kernel's output
  pdl_trigger_at_start();
  int64_t end = M;
  if (offs != nullptr) {
    int bad = 0;
    for (int g = threadIdx.x; g < G; g += kSwzThreads) {
      const int32_t v = offs[g];
      const int32_t prev = g ? offs[g - 1] : 0;
      if (v < prev || (v & 127) != 0 || v > M) bad = 1;
      s_offs[g] = v;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_compose_status, MXQ_DEV_BADOFFS);
      return;
    }
    end = s_offs[G - 1];
  }
  const int64_t TN = N / 128;
  const int64_t pitch = M / 32;                // bytes per row of s_rm
  const int64_t units = N * M / 32 / 16;       // 16-byte units of s_col
  const int64_t tail_atom = TN * (end / 128);  // first atom of the uncovered tail
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kSwzThreads;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kSwzThreads + threadIdx.x; u < units;
       u += stride) {
    const int64_t a = u >> 5;
    const int k = static_cast<int>(u & 31);
    uint4 out = make_uint4(0, 0, 0, 0);
    if (a < tail_atom) {
      int64_t lo = 0, hi = M;
      if (offs != nullptr) {
        const int g = group_of(s_offs, G, 128 * (a / TN));
        lo = g ? s_offs[g - 1] : 0;
        hi = s_offs[g];
      }
      const int64_t A = (hi - lo) / 128;
      const int64_t al = a - TN * (lo / 128);
      const int64_t n0 = 128 * (al / A) + k;
      const int64_t col = lo / 32 + 4 * (al % A);
      const uint8_t* src = s_rm + n0 * pitch + col;
      if (in_buf(src, 96 * pitch + 4, s_rm, static_cast<uint64_t>(N) * M / 32, &g_compose_status)) {
        out.x = __ldg(reinterpret_cast<const uint32_t*>(src));
        out.y = __ldg(reinterpret_cast<const uint32_t*>(src + 32 * pitch));
        out.z = __ldg(reinterpret_cast<const uint32_t*>(src + 64 * pitch));
        out.w = __ldg(reinterpret_cast<const uint32_t*>(src + 96 * pitch));
      }
    }
    if (in_buf(s_col + 16 * u, 16, s_col, static_cast<uint64_t>(N) * M / 32, &g_compose_status))
      reinterpret_cast<uint4*>(s_col)[u] = out;
  }
}

int check_swizzle_args(const uint8_t* s_rm, int64_t N, int64_t M, const int32_t* offs, int32_t G,
                       const uint8_t* s_col) {
  if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0 || M > INT32_MAX || N > INT32_MAX)
    return MXQ_EBADSHAPE;
  if (offs == nullptr ? G != 0 : (G < 1 || G > MXQ_MAX_GROUPS)) return MXQ_EBADOFFS;
  if (offs != nullptr && !aligned_to(offs, 4)) return MXQ_EALIGN;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!s_rm || !s_col) return MXQ_ENULL;
  if (!aligned_to(s_rm, 16) || !aligned_to(s_col, 16)) return MXQ_EALIGN;
  const uint64_t bytes = static_cast<uint64_t>(N) * static_cast<uint64_t>(M) / 32;
  const ByteRange r[3] = {{reinterpret_cast<uintptr_t>(s_rm), bytes},
                          {reinterpret_cast<uintptr_t>(s_col), bytes},
                          {reinterpret_cast<uintptr_t>(offs), offs ? 4ull * G : 0ull}};
  if (ranges_overlap(r, 3)) return MXQ_EOVERLAP;
  return MXQ_OK;
}

int launch_swizzle(const uint8_t* s_rm, int64_t N, int64_t M, const int32_t* offs, int32_t G,
                   uint8_t* s_col, cudaStream_t stream) {
  const int sms = sm_count_current_device(nullptr);
  if (sms <= 0) return MXQ_ECUDA;
  const int64_t units = N * M / 32 / 16;
  const int64_t want = (units + kSwzThreads - 1) / kSwzThreads;
  const int64_t cap = static_cast<int64_t>(sms) * (2048 / kSwzThreads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
  cfg.blockDim = dim3(kSwzThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, mxq_swizzle_kernel, s_rm, N, M, offs, static_cast<int>(G), s_col);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}

}  // namespace

namespace mxq {
// Read (and optionally clear) this file's status word; used by mxq_device_status.
int compose_status_read(unsigned int* out, bool clear) {
  if (cudaMemcpyFromSymbol(out, g_compose_status, sizeof *out) != cudaSuccess) return MXQ_ECUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_compose_status, &zero, sizeof zero) != cudaSuccess)
      return MXQ_ECUDA;
  }
  return MXQ_OK;
}
}  // namespace mxq

extern "C" int mxq_swizzle_kgroups(const uint8_t* s_rm, int64_t N, int64_t M, const int32_t* offs,
                                   int32_t G, uint8_t* s_col, cudaStream_t stream) {
  const int rc = check_swizzle_args(s_rm, N, M, offs, G, s_col);
  if (rc != MXQ_OK || M == 0 || N == 0) return rc;
  return launch_swizzle(s_rm, N, M, offs, G, s_col, stream);
}

extern "C" int mxq_quantize_2d_dual_3pass(const void* x, int64_t M, int64_t N,
                                          const int32_t* offs, int32_t G, uint8_t* q_row,
                                          uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                          uint8_t* workspace, int64_t workspace_bytes,
                                          cudaStream_t stream) {
  if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0 || M > INT32_MAX || N > INT32_MAX)
    return MXQ_EBADSHAPE;
  if (offs == nullptr ? G != 0 : (G < 1 || G > MXQ_MAX_GROUPS)) return MXQ_EBADOFFS;
  if (offs != nullptr && !aligned_to(offs, 4)) return MXQ_EALIGN;
  if (M == 0 || N == 0) return MXQ_OK;
  const uint64_t MN = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  if (!x || !q_row || !s_row || !q_col || !s_col || !workspace) return MXQ_ENULL;
  if (workspace_bytes < 0 || static_cast<uint64_t>(workspace_bytes) < MN / 32)
    return MXQ_EBADSHAPE;
  if (!aligned_to(x, 16) || !aligned_to(q_row, 16) || !aligned_to(s_row, 16) ||
      !aligned_to(q_col, 16) || !aligned_to(s_col, 16) || !aligned_to(workspace, 16))
    return MXQ_EALIGN;
  const ByteRange r[7] = {
      {reinterpret_cast<uintptr_t>(x), 2 * MN},
      {reinterpret_cast<uintptr_t>(q_row), MN},
      {reinterpret_cast<uintptr_t>(q_col), MN},
      {reinterpret_cast<uintptr_t>(s_row), MN / 32},
      {reinterpret_cast<uintptr_t>(s_col), MN / 32},
      {reinterpret_cast<uintptr_t>(workspace), MN / 32},
      {reinterpret_cast<uintptr_t>(offs), offs ? 4ull * static_cast<uint64_t>(G) : 0ull},
  };
  if (ranges_overlap(r, 7)) return MXQ_EOVERLAP;
  int rc = mxq_quantize_1x32(x, M, N, q_row, s_row, stream);
  if (rc != MXQ_OK) return rc;
  rc = mxq_quantize_32x1(x, M, N, q_col, workspace, stream);
  if (rc != MXQ_OK) return rc;
  return launch_swizzle(workspace, N, M, offs, G, s_col, stream);
}

// ---------------------------------------------------------------------------
// The same three passes without any allocation by anyone.
//
// Some callers cannot allocate device memory at the moment they need this cast:
// work being recorded into a CUDA graph in global capture mode (allocation
// calls are illegal during such a capture), latency-critical paths where a
// cudaMalloc/cudaFree can synchronize the device, and plugins running inside a
// framework that owns all device memory through its own allocator, which the
// plugin cannot reach.  For them the workspace of the three-pass call lives in
// a static device array of this library instead of a caller buffer.
// ---------------------------------------------------------------------------
namespace {

// Holds the row-major colwise scales between the 32x1 pass and the swizzle.
// Every GPU that loads this library keeps it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MXQ_NOALLOC_SCRATCH_BYTES];

// The driver's cuCtxGetCurrent, reached through the runtime (no link-time
// dependency on libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of the array on device `dev` (the host-side name is only a
// stand-in for the symbol).  It is looked up with that device current on the
// first call, and again whenever the current context differs from the one it
// was looked up in: after a device reset the module can load at another
// address.  Later calls only compare the context, which is safe during a
// stream capture; the lookup itself may load the module, so the first call on
// a device (or in a new context) belongs before any capture.
uint8_t* noalloc_scratch(int dev) {
  static std::mutex mu;
  static uint8_t* addr[64] = {};
  static CUcontext ctx_of[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  if (addr[dev] == nullptr || ctx == nullptr || ctx != ctx_of[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    // the lookup makes the device's primary context current if none was
    if (get(&ctx) != CUDA_SUCCESS) return nullptr;
    addr[dev] = static_cast<uint8_t*>(p);
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

}  // namespace

extern "C" int mxq_quantize_2d_dual_3pass_noalloc(const void* x, int64_t M, int64_t N,
                                                  const int32_t* offs, int32_t G, uint8_t* q_row,
                                                  uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                                  cudaStream_t stream) {
  if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0 || M > INT32_MAX || N > INT32_MAX)
    return MXQ_EBADSHAPE;
  if (offs == nullptr ? G != 0 : (G < 1 || G > MXQ_MAX_GROUPS)) return MXQ_EBADOFFS;
  if (offs != nullptr && !aligned_to(offs, 4)) return MXQ_EALIGN;
  if (M == 0 || N == 0) return MXQ_OK;
  const uint64_t scratch_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N) / 32;
  if (scratch_bytes > MXQ_NOALLOC_SCRATCH_BYTES) return MXQ_ESCRATCH;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXQ_ECUDA;
  uint8_t* ws = noalloc_scratch(dev);
  if (ws == nullptr) return MXQ_ECUDA;
  // The 32x1 pass rewrites every byte of the scratch prefix that the swizzle
  // reads, so nothing left by an earlier call needs clearing.
  return mxq_quantize_2d_dual_3pass(x, M, N, offs, G, q_row, s_row, q_col, s_col, ws,
                                    static_cast<int64_t>(scratch_bytes), stream);
}
