// mxq_check.cuh -- bounds checks of the kernels' computed global accesses,
// compiled in with MXQ_DEBUG_BOUNDS=1 (a checked build of the library).
// Where no memory checker can run, the checked build stands in for one: an
// access whose byte range would leave its buffer is skipped and recorded as
// MXQ_DEV_OOB in the kernel file's status word (read by mxq_device_status).
// No trap, no assert.  In a release build every check is the constant `true`.
#pragma once

#include <stdint.h>

#include "mxq.h"

#ifndef MXQ_DEBUG_BOUNDS
#define MXQ_DEBUG_BOUNDS 0
#endif

namespace mxq {

// true when the bytes [p, p + n) lie inside the buffer [buf, buf + size).
__device__ __forceinline__ bool in_buf(const void* p, uint64_t n, const void* buf, uint64_t size,
                                       unsigned int* status) {
#if MXQ_DEBUG_BOUNDS
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), lo = reinterpret_cast<uintptr_t>(buf);
  if (a >= lo && n <= size && a - lo <= size - n) return true;
  atomicOr(status, MXQ_DEV_OOB);
  return false;
#else
  (void)p, (void)n, (void)buf, (void)size, (void)status;
  return true;
#endif
}

// Complete `bytes` of an mbarrier's expected transaction count without a
// copy (a checked build's stand-in for a load it skipped), so that the
// waiting consumers are released instead of timing out.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

}  // namespace mxq
