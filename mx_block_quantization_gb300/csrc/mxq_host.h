// mxq_host.h -- host-side argument checks and device queries shared by the
// launch code.  Nothing here calls CUDA except the device-property helpers,
// which are only reached after every argument check has passed.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "mxq.h"

namespace mxq {

inline bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// A byte range [lo, lo + bytes) of one buffer; empty ranges never overlap.
struct ByteRange {
  uintptr_t lo;
  uint64_t bytes;
};

// A range that wraps past the top of the address space is no real buffer and
// counts as overlapping.
inline bool ranges_overlap(const ByteRange* r, int n) {
  for (int i = 0; i < n; ++i)
    if (r[i].bytes != 0 && r[i].lo + r[i].bytes <= r[i].lo) return true;
  for (int i = 0; i < n; ++i) {
    if (r[i].bytes == 0) continue;
    for (int j = i + 1; j < n; ++j) {
      if (r[j].bytes == 0) continue;
      const uintptr_t a0 = r[i].lo, a1 = r[i].lo + r[i].bytes;
      const uintptr_t b0 = r[j].lo, b1 = r[j].lo + r[j].bytes;
      if (a0 < b1 && b0 < a1) return true;
    }
  }
  return false;
}

// Programmatic dependent launch of every compute kernel (on by default; the
// macro exists so that a build without it can be measured against).
#ifndef MXQ_PDL
#define MXQ_PDL 1
#endif

// Marks a launch as allowed to start while the previous kernel of its stream
// is still running.  The kernel must call pdl_wait() (mxq_device.cuh) before
// touching global memory; with the attribute set, a predecessor that calls
// pdl_launch_dependents() lets this launch's CTAs be placed on SMs as its
// own CTAs leave, which hides the launch latency and set-up between kernels.
// `attr` must outlive the cudaLaunchKernelEx call.
inline void allow_programmatic_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr) {
  if (!MXQ_PDL) return;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link libcuda), looked up once; null if unavailable.
inline PFN_cuTensorMapEncodeTiled_v12000 driver_tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Number of SMs of the current device, cached per device ordinal.
inline int sm_count_current_device(int* out_device) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (out_device) *out_device = dev;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Launch the packed-record form of the TMA-fed pack kernel (mx9.cu) over nb
// whole 16-element blocks of a tensor blocked along its rows: rows of nbl
// blocks, pitch bytes apart; x, packed and pitch 16-byte aligned, arguments
// already checked.  Returns an MXQ_* code.
int launch_records_pack(const void* x, bool bf16, int fmt, int64_t nb, int64_t nbl, int64_t pitch,
                        uint8_t* packed, cudaStream_t stream);

// The TMA column-tile kernels (mx_cols_tma.cu) for a tensor blocked along its
// columns: taken when cols_tma_ok accepts the geometry (16-byte aligned x and
// packed, row pitch a multiple of 16 bytes, each column's records a multiple
// of 16 bytes, sizes within the int32 tile coordinates; for unpack, writes_x,
// also rows of a whole number of 16-byte pieces).  The launches return
// an MXQ_* code, or kColsTmaDeclined when a tensor map cannot be encoded (the
// caller then takes another kernel).  Arguments already checked.
constexpr int kColsTmaDeclined = 1;
bool cols_tma_ok(const void* x, int dtype, int fmt, int64_t rows, int64_t cols, int64_t ld,
                 const void* packed, bool writes_x);
int cols_tma_pack(const void* x, bool bf16, int fmt, int64_t rows, int64_t cols, int64_t ld,
                  uint8_t* packed, cudaStream_t stream);
int cols_tma_unpack(const uint8_t* packed, int fmt, void* y, bool bf16, int64_t rows, int64_t cols,
                    int64_t ld, cudaStream_t stream);
int cols_status_read(unsigned int* out, bool clear);

}  // namespace mxq
