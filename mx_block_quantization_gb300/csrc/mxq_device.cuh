// mxq_device.cuh -- inline-PTX helpers shared by the sm_103a kernels:
// mbarriers with bounded waits, TMA tensor loads/stores, bulk copies, proxy
// fences, and the E8M0/E4M3 building blocks of the MXFP8 cast.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxq {

// ---------------------------------------------------------------------------
// shared-memory addresses, timers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// A kernel launched with programmatic stream serialization may be scheduled
// while the kernel before it on the stream is still running.  pdl_wait()
// returns once that kernel has completed and its memory writes are visible
// (at once when the launch has no such predecessor), so every kernel of the
// library calls it, in every thread, before its first global-memory access.
// Since no CTA gets past it early, a kernel never completes before its
// predecessor, which keeps the ordering transitive along a chain of launches.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel of the stream (if launched with programmatic stream
// serialization) be scheduled once every CTA of this grid has signalled or
// exited; its CTAs then take SMs as this grid's CTAs leave and run their
// set-up before their own pdl_wait().
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Where a kernel signals its dependents: 0 right after its set-up, 1 when a
// thread has finished its main loop (threads without work exit instead), 2
// never (the signal is then implied by the grid's completion).  2 is the
// measured best: an explicit signal let the next kernel's CTAs become resident
// beside the running ones, where they slowed it (the fp32 MX9 pack followed by
// the unpack: 98 -> 105 us at 16384x8192 with the signal at set-up, 111 us
// with it at the end of the main loops), while the kernels that follow gained
// less than that.
#ifndef MXQ_PDL_TRIGGER
#define MXQ_PDL_TRIGGER 2
#endif
__device__ __forceinline__ void pdl_trigger_at_start() {
  if (MXQ_PDL_TRIGGER == 0) pdl_launch_dependents();
}
__device__ __forceinline__ void pdl_trigger_at_end() {
  if (MXQ_PDL_TRIGGER == 1) pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Upper bound on any single pipeline wait.  A wait in a healthy launch lasts
// microseconds; the bound only exists so that a logic error ends the kernel
// with a status bit instead of hanging the GPU.  It is generous because the
// GPU may be time-sliced with other processes.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s

// Wait for the phase with the given parity to complete.  Gives up when the
// CTA-wide abort flag is raised by another role, or after kWaitLimitNs, in
// which case it raises the flag itself and records `timeout_bit` in *status.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag,
                                                  unsigned int* status, unsigned int timeout_bit,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1u;
        atomicOr(status, timeout_bit);
        return false;
      }
    }
  }
}

// Same, without the abort flag: used to drain copies already in flight while
// a CTA is shutting down.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA and bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load global -> shared, completing `bar`'s transaction count.
// c0 is the innermost coordinate (elements), c1 the outer one.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// L2 eviction-priority policy for data touched exactly once.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 cache-policy hint.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                                 int32_t c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// tma_store_2d with an L2 cache-policy hint.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, int32_t c0, int32_t c1,
                                                  uint32_t src, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(map),
      "r"(c0), "r"(c1), "r"(src), "l"(policy)
      : "memory");
}

// 2-D tiled store shared -> global, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t c0, int32_t c1,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          map),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
}

// Contiguous bulk store shared -> global (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed groups are incomplete (writes visible).
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// shared-memory vector access
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                       uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}

__device__ __forceinline__ void sts8(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// MXFP8 arithmetic
// ---------------------------------------------------------------------------

// E8M0 rceil scale byte from the block amax given as sign-masked bf16 bits
// (unsigned 16-bit order equals magnitude order for finite values; +Inf is
// 0x7F80 and every NaN is above it).  For finite amax with exponent field E
// and mantissa f, the smallest s with amax <= 448 * 2^(s-127) is
// E - 8 + [f > 0x60] (448 = 1.75 * 2^8 and 0.75 = 0x60/0x80), at least 0.
// `inf_code` is the byte for an Inf-only block: 255 rowwise, 254 colwise.
__device__ __forceinline__ uint32_t e8m0_rceil_from_bits(uint32_t a, uint32_t inf_code) {
  int e = static_cast<int>(a >> 7) - 8 + ((a & 0x7Fu) > 0x60u ? 1 : 0);
  uint32_t s = static_cast<uint32_t>(e < 0 ? 0 : e);
  s = (a == 0x7F80u) ? inf_code : s;
  s = (a > 0x7F80u) ? 255u : s;
  return s;
}

// The reciprocal multiplier 2^(127 - s) as an fp32: normal for s <= 253, the
// subnormal 2^-127 for s = 254 (used only by Inf-carrying colwise blocks).
// For s = 255 (the NaN rule) it is a NaN, so every product is NaN and every
// byte of the block casts to the E4M3 NaN 0x7F without a separate override.
__device__ __forceinline__ float e8m0_multiplier(uint32_t s) {
  return __uint_as_float(s == 255u ? 0x7FFFFFFFu : s == 254u ? 0x00400000u : (254u - s) << 23);
}

// Per-half max(|a|, |b|) of two bf16x2 words where a NaN operand loses to the
// other one (IEEE maxNum); the sign bit is masked off by the caller.
__device__ __forceinline__ uint32_t bf16x2_absmax_skip_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per-half max(|a|, |b|) of two bf16x2 words, NaN-propagating (the sign bit of
// the result is the xor of the inputs' signs and is masked off by the caller).
__device__ __forceinline__ uint32_t bf16x2_absmax_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// IEEE single multiply, round to nearest, subnormals kept (no flush).
__device__ __forceinline__ float fmul_rn_noftz(float a, float b) {
  float r;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Two fp32 -> two E4M3 bytes, round to nearest even, saturating finite.
// Result low byte = cvt(lo), high byte = cvt(hi).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

// Widen the two bf16 halves of a word to fp32 (exact).
__device__ __forceinline__ float bf16_lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace mxq
