// mxq_dual.cu -- one-pass dual-axis MXFP8 quantization for sm_103a.
//
// Method: pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with
// correct metadata" (description): read a bf16 [M, N] tensor once and emit
// E4M3 data cast in 1x32 blocks along N and in 32x1 blocks along M (stored
// transposed), plus both E8M0 rceil scale tensors already in the 128x4
// blocked layout of block-scaled MMA, the colwise scales placed per K-group
// slab and zeroed past offs[G-1].
//
// GB300 design (a persistent, warp-specialized, bandwidth-bound kernel; no
// tensor cores because there is no contraction):
//   * one CTA per SM walks 128x128 tiles t = blockIdx.x + k * gridDim.x;
//   * warp 16 (producer) streams tiles into a 3-stage shared-memory ring with
//     2-D TMA loads (two 64-column boxes per tile, 128-byte swizzle);
//   * warps 0..15 (consumers) run the rowwise and the colwise pass of a tile
//     from shared memory and write its four outputs into a double-buffered
//     shared staging area (E4M3 tiles in the same 128-byte swizzle, 512-byte
//     scale atoms already in blocked order);
//   * warp 17 (storer) drains each staged tile with two TMA tensor stores
//     (q_row, q_col) and two 512-byte bulk stores (the s_row atom and either
//     the s_col atom at its group slab or a zero atom for tail rows).
// Every pipeline wait is bounded; on a timeout the CTA raises a status bit,
// drains the copies it has in flight and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mxq.h"
#include "mxq_check.cuh"
#include "mxq_device.cuh"
#include "mxq_host.h"

namespace {

using namespace mxq;

// Pipeline shape.  The defaults are the measured best on GB300; the macros
// only exist so that other shapes can be built for measurement.
#ifndef MXQ_DUAL_STAGES
#define MXQ_DUAL_STAGES 3
#endif
#ifndef MXQ_DUAL_OUTBUFS
#define MXQ_DUAL_OUTBUFS 2
#endif
#ifndef MXQ_DUAL_GROUP_ROWS
#define MXQ_DUAL_GROUP_ROWS 8
#endif
// When the fused cast issues each tile's s_col atom store: 1 once the tile's
// data stores (q_row, q_col) have read their shared-memory tiles, from a
// 4-slot ring of atoms so that the data buffer is still released at that point;
// 0 together with the data stores.  1 measured 3.5-6% faster on grouped
// layouts at 65536x7168 (MoE groups 0.943 -> 0.976 of the measured copy rate,
// 64 groups of 1024 rows 0.916 -> 0.971) and the same on the dense layout
// (0.89); issuing the atom one tile later instead gained nothing.
#ifndef MXQ_DUAL_SCOL_DEFER
#define MXQ_DUAL_SCOL_DEFER 1
#endif
// 1: the s_row atom goes after the data stores too, from its own 4-slot ring
// (grouped layouts at 65536x7168: MoE 0.974 -> 0.982 of the measured copy rate,
// 64 groups 0.965 -> 0.983; dense unchanged)
#ifndef MXQ_DUAL_SROW_AFTER
#define MXQ_DUAL_SROW_AFTER 1
#endif
constexpr bool kSRowAfter = MXQ_DUAL_SCOL_DEFER && MXQ_DUAL_SROW_AFTER;
#ifndef MXQ_DUAL_L2_HINTS  // bit 0: evict-first on the input loads, bit 1: on the data stores
#define MXQ_DUAL_L2_HINTS 0
#endif
constexpr int kTile = 128;
constexpr int kStages = MXQ_DUAL_STAGES;              // input ring depth (tiles)
constexpr int kOutBufs = MXQ_DUAL_OUTBUFS;            // staged output tiles
constexpr int kPassWarps = 8;                         // consumer warps per pass
constexpr int kGroupRows = MXQ_DUAL_GROUP_ROWS;       // tile rows per rasterization group

// What one launch computes: both passes (the fused cast), or one of them
// alone (the separate 1x32 and 32x1 casts of the three-pass composition).
enum Mode : int { kDual = 0, kRowOnly = 1, kColOnly = 2 };

template <int kMode>
struct Roles {
  static constexpr bool kRow = kMode != kColOnly;
  static constexpr bool kCol = kMode != kRowOnly;
  static constexpr int kRowWarps = kRow ? kPassWarps : 0;  // warps [0, kRowWarps)
  static constexpr int kConsumerWarps = kRowWarps + (kCol ? kPassWarps : 0);
  static constexpr int kProducerWarp = kConsumerWarps;
  static constexpr int kStoreWarp = kConsumerWarps + 1;
  static constexpr int kThreads = (kConsumerWarps + 2) * 32;  // 576 for the fused cast
};

constexpr uint32_t kInStageBytes = kTile * kTile * 2;  // bf16 tile, 32 KiB
constexpr uint32_t kHalfBytes = kTile * 64 * 2;        // [128 rows][64 bf16] box, 16 KiB
constexpr uint32_t kQTileBytes = kTile * kTile;        // E4M3 tile, 16 KiB
constexpr uint32_t kAtomBytes = 512;                   // one 128x4 scale atom

// Shared-memory map (offsets from a 1024-byte aligned base; every swizzled
// buffer starts on a 1024-byte boundary as the 128-byte swizzle requires).
constexpr uint32_t kOffIn = 0;
constexpr uint32_t kOffQRow = kOffIn + kStages * kInStageBytes;
constexpr uint32_t kOffQCol = kOffQRow + kOutBufs * kQTileBytes;
constexpr uint32_t kOffSRow = kOffQCol + kOutBufs * kQTileBytes;
constexpr uint32_t kOffSCol = kOffSRow + kOutBufs * kAtomBytes;
constexpr int kSColSlots = 4;                          // deferred s_col atoms
constexpr uint32_t kOffSColRing = kOffSCol + kOutBufs * kAtomBytes;
constexpr uint32_t kOffSRowRing = kOffSColRing + kSColSlots * kAtomBytes;
constexpr uint32_t kOffZero = kOffSRowRing + (kSRowAfter ? kSColSlots : 0) * kAtomBytes;
constexpr uint32_t kOffOffs = kOffZero + kAtomBytes;
constexpr uint32_t kOffBar = kOffOffs + 4 * MXQ_MAX_GROUPS;
constexpr uint32_t kNumBars = 2 * kStages + 2 * kOutBufs;
constexpr uint32_t kOffFlag = kOffBar + 8 * kNumBars;
constexpr uint32_t kSmemUsed = kOffFlag + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffQRow % 1024 == 0 && kOffQCol % 1024 == 0, "swizzle alignment");

// Sticky per-device status word (MXQ_DEV_* bits), read by mxq_device_status.
__device__ unsigned int g_mxq_status = 0;

struct Bars {
  uint32_t base;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (kStages + s); }
  __device__ uint32_t ofull(int b) const { return base + 8u * (2 * kStages + b); }
  __device__ uint32_t oempty(int b) const { return base + 8u * (2 * kStages + kOutBufs + b); }
};

// Physical byte offset of 16-byte chunk `chunk` of row `row` in a buffer of
// 128-byte rows written with the 128-byte TMA swizzle (chunk ^= row % 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Amax of a run of bf16x2 words as sign-masked bf16 bits (per half): one
// NaN-propagating abs-max per word, then the sign bits cleared once.
template <int kWords>
__device__ __forceinline__ uint32_t absmax_bits(const uint32_t* w) {
  uint32_t m = w[0];
#pragma unroll
  for (int i = 1; i < kWords; ++i) m = bf16x2_absmax_nan(m, w[i]);
  return m & 0x7FFF7FFFu;
}

// The same amax with NaN skipped (the separate 32x1 cast's rule): the running
// maximum starts at 0 and a NaN operand never wins, so an all-NaN column gives 0.
template <int kWords>
__device__ __forceinline__ uint32_t absmax_bits_skip_nan(const uint32_t* w) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < kWords; ++i) m = bf16x2_absmax_skip_nan(m, w[i]);
  return m & 0x7FFF7FFFu;
}

// Cast one 1x32 row block (16 bf16x2 words, element order) with the
// multiplier of its scale and pack the E4M3 bytes in element order, four per
// output word.
__device__ __forceinline__ void cast_row_block(const uint32_t* w, float mult, uint32_t* o) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = w[2 * i], b = w[2 * i + 1];
    const uint32_t lo = cvt_e4m3x2(fmul_rn_noftz(bf16_hi_f32(a), mult),
                                   fmul_rn_noftz(bf16_lo_f32(a), mult));
    const uint32_t hi = cvt_e4m3x2(fmul_rn_noftz(bf16_hi_f32(b), mult),
                                   fmul_rn_noftz(bf16_lo_f32(b), mult));
    o[i] = lo | (hi << 16);
  }
}

// ---------------------------------------------------------------------------
// Rowwise warps (0..7): lane l of warp w takes tile row r = 16w + l/2 and the
// half-tile h = l%2, i.e. the two 1x32 blocks 2h and 2h+1.  Lanes with h = 1
// visit their eight 16-byte chunks in the order k ^ 4, so the 128-bit loads
// and stores of every 8-lane phase hit eight distinct bank groups; that only
// changes which block (jA, jB) each half of the registers belongs to.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rowwise_pass(uint32_t in_s, uint32_t qrow_s, uint32_t srow_s,
                                             int warp, int lane) {
  const int r = 16 * warp + (lane >> 1);
  const int h = lane & 1;
  const uint32_t half = in_s + static_cast<uint32_t>(h) * kHalfBytes;
  uint32_t w[32];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = lds128(half + swz(r, k ^ (4 * h)));
    w[4 * k + 0] = v.x;
    w[4 * k + 1] = v.y;
    w[4 * k + 2] = v.z;
    w[4 * k + 3] = v.w;
  }
  const int jA = 3 * h, jB = 2 * h + 1 - h;  // block of registers 0..15 / 16..31
  const uint32_t mA = absmax_bits<16>(w), mB = absmax_bits<16>(w + 16);
  const uint32_t sA = e8m0_rceil_from_bits(max(mA & 0xFFFFu, mA >> 16), 255u);
  const uint32_t sB = e8m0_rceil_from_bits(max(mB & 0xFFFFu, mB >> 16), 255u);
  uint32_t oA[8], oB[8];
  cast_row_block(w, e8m0_multiplier(sA), oA);
  cast_row_block(w + 16, e8m0_multiplier(sB), oB);
  sts128(qrow_s + swz(r, 2 * jA), oA[0], oA[1], oA[2], oA[3]);
  sts128(qrow_s + swz(r, 2 * jA + 1), oA[4], oA[5], oA[6], oA[7]);
  sts128(qrow_s + swz(r, 2 * jB), oB[0], oB[1], oB[2], oB[3]);
  sts128(qrow_s + swz(r, 2 * jB + 1), oB[4], oB[5], oB[6], oB[7]);
  const uint32_t at = static_cast<uint32_t>((r & 31) * 16 + (r >> 5) * 4);
  sts8(srow_s + at + jA, sA);
  sts8(srow_s + at + jB, sB);
}

// ---------------------------------------------------------------------------
// Colwise warps (8..15): warp 8 + w' takes row block i = w'/2 (rows 32i..+31)
// and lane l one column pair p (columns 2p, 2p+1) down all 32 rows.  Lanes
// 0..15 take pairs 16q + l of half-tile 0 and lanes 16..31 pairs
// 32 + 16(1-q) + (l-16) of half-tile 1 (q = w' % 2), so the two half-warps of
// every 32-bit load read different bank groups of the same row.  E4M3 bytes
// of four consecutive rows of one column form one word: each lane emits 32
// contiguous bytes of q_col per column.
// ---------------------------------------------------------------------------
template <bool kNaNPoisons>
__device__ __forceinline__ void colwise_pass(uint32_t in_s, uint32_t qcol_s, uint32_t scol_s,
                                             int cwarp, int lane) {
  const int i = cwarp >> 1;
  const int q = cwarp & 1;
  const int p = lane < 16 ? 16 * q + lane : 32 + 16 * (1 - q) + (lane - 16);
  const uint32_t half = in_s + (p >= 32 ? kHalfBytes : 0u);
  const int pp = p & 31;
  const int chunk = pp >> 2;
  const uint32_t within = static_cast<uint32_t>(pp & 3) * 4u;
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) w[j] = lds32(half + swz(32 * i + j, chunk) + within);

  const uint32_t m = kNaNPoisons ? absmax_bits<32>(w) : absmax_bits_skip_nan<32>(w);
  const uint32_t s_lo = e8m0_rceil_from_bits(m & 0xFFFFu, 254u);  // column 2p
  const uint32_t s_hi = e8m0_rceil_from_bits(m >> 16, 254u);      // column 2p+1
  const float mult_lo = e8m0_multiplier(s_lo);
  const float mult_hi = e8m0_multiplier(s_hi);
  uint32_t L[8], H[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t a = w[4 * g], b = w[4 * g + 1], c = w[4 * g + 2], d = w[4 * g + 3];
    const uint32_t l01 = cvt_e4m3x2(fmul_rn_noftz(bf16_lo_f32(b), mult_lo),
                                    fmul_rn_noftz(bf16_lo_f32(a), mult_lo));
    const uint32_t l23 = cvt_e4m3x2(fmul_rn_noftz(bf16_lo_f32(d), mult_lo),
                                    fmul_rn_noftz(bf16_lo_f32(c), mult_lo));
    const uint32_t h01 = cvt_e4m3x2(fmul_rn_noftz(bf16_hi_f32(b), mult_hi),
                                    fmul_rn_noftz(bf16_hi_f32(a), mult_hi));
    const uint32_t h23 = cvt_e4m3x2(fmul_rn_noftz(bf16_hi_f32(d), mult_hi),
                                    fmul_rn_noftz(bf16_hi_f32(c), mult_hi));
    L[g] = l01 | (l23 << 16);
    H[g] = h01 | (h23 << 16);
  }
  const int n_lo = 2 * p, n_hi = 2 * p + 1;  // tile-local columns = q_col tile rows
  sts128(qcol_s + swz(n_lo, 2 * i), L[0], L[1], L[2], L[3]);
  sts128(qcol_s + swz(n_lo, 2 * i + 1), L[4], L[5], L[6], L[7]);
  sts128(qcol_s + swz(n_hi, 2 * i), H[0], H[1], H[2], H[3]);
  sts128(qcol_s + swz(n_hi, 2 * i + 1), H[4], H[5], H[6], H[7]);
  sts8(scol_s + static_cast<uint32_t>((n_lo & 31) * 16 + (n_lo >> 5) * 4 + i), s_lo);
  sts8(scol_s + static_cast<uint32_t>((n_hi & 31) * 16 + (n_hi >> 5) * 4 + i), s_hi);
}

// Tile t of the persistent walk -> (tile row, tile column).  Tiles go in
// groups of kGroupRows tile rows, column by column inside a group, so the
// tiles in flight at one time cover a compact block: x rows and q_row rows
// are read/written in runs of several tiles, and so are the rows of the
// transposed q_col.
__device__ __forceinline__ void tile_coords(int64_t t, int64_t TM, int64_t TN, int64_t* ti,
                                            int64_t* tj) {
  const int64_t per_group = static_cast<int64_t>(kGroupRows) * TN;
  const int64_t g = t / per_group;
  const int64_t local = t - g * per_group;
  const int64_t rows = min(static_cast<int64_t>(kGroupRows), TM - g * kGroupRows);
  *ti = g * kGroupRows + local % rows;
  *tj = local / rows;
}

// First g with offs[g] > row (the group holding `row`), by binary search.
__device__ __forceinline__ int group_of_row(const int32_t* s_offs, int G, int64_t row) {
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

// One persistent launch over all 128x128 tiles.  kDual: the fused cast
// (q_row, s_row, q_col and grouped s_col).  kRowOnly: q_row and s_row.
// kColOnly: q_col and the colwise scales as a plain [N, M/32] row-major matrix
// written to `s_col` (the separate 32x1 cast, NaN skipped by its amax).
template <int kMode>
__global__ void __launch_bounds__(Roles<kMode>::kThreads, 1)
    mxq_tile_kernel(const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_qrow,
                    const __grid_constant__ CUtensorMap tm_qcol, const int32_t* __restrict__ offs,
                    int G, int M, int N, int grow0, int Mtot, uint8_t* __restrict__ s_row,
                    uint8_t* __restrict__ s_col) {
  using R = Roles<kMode>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t TN = N / kTile;
  const int64_t TM = M / kTile;
  const int64_t T = TM * TN;
  const int64_t my_tiles =
      (static_cast<int64_t>(blockIdx.x) < T) ? (T - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  const Bars bars{base + kOffBar};
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + kOffFlag);
  int32_t* s_offs = reinterpret_cast<int32_t*>(gbase + kOffOffs);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), R::kConsumerWarps);
    }
    for (int b = 0; b < kOutBufs; ++b) {
      mbar_init(bars.ofull(b), R::kConsumerWarps);
      mbar_init(bars.oempty(b), 1);
    }
    *abort_flag = 0u;
    mbar_init_fence();
  }
  if (tid < kAtomBytes / 4) {
    sts32(base + kOffZero + 4u * tid, 0u);
    fence_proxy_async_smem();
  }
  if (warp == R::kProducerWarp && lane == 0) tma_prefetch_desc(&tm_x);
  __syncthreads();
  // The set-up above touched only shared memory and the launch parameters, so
  // it may overlap the previous kernel of the stream; global memory may hold
  // that kernel's results only from here on.
  pdl_wait();
  pdl_trigger_at_start();

  // Producer prologue: start the first loads before the offsets check.
  int64_t issued = 0;
  const bool is_producer = (warp == R::kProducerWarp) && (lane == 0);
  auto issue_load = [&](int64_t k) {
    int64_t ti, tj;
    tile_coords(blockIdx.x + k * static_cast<int64_t>(gridDim.x), TM, TN, &ti, &tj);
    const int s = static_cast<int>(k % kStages);
    const uint32_t dst = base + kOffIn + static_cast<uint32_t>(s) * kInStageBytes;
    mbar_arrive_expect_tx(bars.full(s), kInStageBytes);
    const int32_t c0 = static_cast<int32_t>(tj * kTile), r0 = static_cast<int32_t>(ti * kTile);
    if (MXQ_DUAL_L2_HINTS & 1) {
      const uint64_t pol = l2_policy_evict_first();
      tma_load_2d_hint(dst, &tm_x, c0, r0, bars.full(s), pol);
      tma_load_2d_hint(dst + kHalfBytes, &tm_x, c0 + 64, r0, bars.full(s), pol);
    } else {
      tma_load_2d(dst, &tm_x, c0, r0, bars.full(s));
      tma_load_2d(dst + kHalfBytes, &tm_x, c0 + 64, r0, bars.full(s));
    }
  };
  auto drain_loads = [&]() {
    for (int64_t k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
      mbar_wait_drain(bars.full(static_cast<int>(k % kStages)),
                      static_cast<uint32_t>((k / kStages) & 1));
  };
  if (is_producer) {
    for (; issued < my_tiles && issued < kStages; ++issued) issue_load(issued);
  }

  // Device-side check of the group offsets (fused cast only): ascending,
  // multiples of 128, within [0, Mtot] (the full tensor's rows; this launch
  // casts its rows [grow0, grow0 + M)).  Every CTA reaches the same verdict;
  // on failure nothing is written and the status word records it.
  int64_t end_rows = Mtot;
  if (kMode == kDual && offs != nullptr) {
    int bad = 0;
    for (int g = tid; g < G; g += R::kThreads) {
      const int32_t v = offs[g];
      const int32_t prev = g ? offs[g - 1] : 0;
      if (v < prev || (v & (kTile - 1)) != 0 || v > Mtot) bad = 1;
      s_offs[g] = v;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      if (blockIdx.x == 0 && tid == 0) atomicOr(&g_mxq_status, MXQ_DEV_BADOFFS);
      if (is_producer) drain_loads();
      return;
    }
    end_rows = s_offs[G - 1];
  }

  if (warp < R::kConsumerWarps) {
    // ------------------------------------------------------------- consumers
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int s = static_cast<int>(k % kStages);
      const int b = static_cast<int>(k % kOutBufs);
      // every lane waits (acquiring the barrier's data); the warp leaves
      // together if any lane gave up, so no warp-collective runs short
      bool ok = mbar_wait_bounded(bars.full(s), static_cast<uint32_t>((k / kStages) & 1),
                                  abort_flag, &g_mxq_status, MXQ_DEV_TIMEOUT);
      if (ok && k >= kOutBufs)
        ok = mbar_wait_bounded(bars.oempty(b), static_cast<uint32_t>(((k / kOutBufs) - 1) & 1),
                               abort_flag, &g_mxq_status, MXQ_DEV_TIMEOUT);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      const uint32_t in_s = base + kOffIn + static_cast<uint32_t>(s) * kInStageBytes;
      if (warp < R::kRowWarps)
        rowwise_pass(in_s, base + kOffQRow + b * kQTileBytes,
                     (kMode == kDual && kSRowAfter)
                         ? base + kOffSRowRing + static_cast<uint32_t>(k % kSColSlots) * kAtomBytes
                         : base + kOffSRow + b * kAtomBytes,
                     warp, lane);
      else
        colwise_pass<kMode == kDual>(
            in_s, base + kOffQCol + b * kQTileBytes,
            (kMode == kDual && MXQ_DUAL_SCOL_DEFER)
                ? base + kOffSColRing + static_cast<uint32_t>(k % kSColSlots) * kAtomBytes
                : base + kOffSCol + b * kAtomBytes,
            warp - R::kRowWarps, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(s));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ofull(b));
    }
    pdl_trigger_at_end();
  } else if (warp == R::kProducerWarp) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      for (int64_t k = issued; k < my_tiles; ++k) {
        const int s = static_cast<int>(k % kStages);
        if (!mbar_wait_bounded(bars.empty(s), static_cast<uint32_t>(((k / kStages) - 1) & 1),
                               abort_flag, &g_mxq_status, MXQ_DEV_TIMEOUT)) {
          drain_loads();
          return;
        }
        issue_load(k);
        issued = k + 1;
      }
      pdl_trigger_at_end();
    }
  } else if (warp == R::kStoreWarp) {
    // ---------------------------------------------------------------- storer
    // Lane 0 issues the TMA and bulk stores.  For the 32x1 cast every lane
    // also copies the tile's 128 scale words (4 row blocks of one column are
    // adjacent in the staged atom) into the row-major scale matrix.
    if (kMode != kColOnly && lane != 0) return;
    if (lane == 0) {
      if (R::kRow) tma_prefetch_desc(&tm_qrow);
      if (R::kCol) tma_prefetch_desc(&tm_qcol);
    }
    const int64_t Mrows = M;
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int b = static_cast<int>(k % kOutBufs);
      bool ok = mbar_wait_bounded(bars.ofull(b), static_cast<uint32_t>((k / kOutBufs) & 1),
                                  abort_flag, &g_mxq_status, MXQ_DEV_TIMEOUT);
      if (kMode == kColOnly) ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      int64_t ti, tj;
      tile_coords(blockIdx.x + k * static_cast<int64_t>(gridDim.x), TM, TN, &ti, &tj);
      const int64_t row0 = ti * kTile;
      if (kMode == kColOnly) {
        const int64_t pitch = Mrows / 32;  // bytes per row of the [N, M/32] matrix
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int n = lane + 32 * r;
          const uint32_t word =
              lds32(base + kOffSCol + b * kAtomBytes + static_cast<uint32_t>((n & 31) * 16 + (n >> 5) * 4));
          uint8_t* const dst = s_col + (tj * kTile + n) * pitch + 4 * ti;
          if (in_buf(dst, 4, s_col, static_cast<uint64_t>(N) * Mrows / 32, &g_mxq_status))
            *reinterpret_cast<uint32_t*>(dst) = word;
        }
        __syncwarp();
      }
      if (lane == 0) {
        const uint64_t pol = (MXQ_DUAL_L2_HINTS & 2) ? l2_policy_evict_first() : 0ull;
        if (R::kRow) {
          if (MXQ_DUAL_L2_HINTS & 2)
            tma_store_2d_hint(&tm_qrow, static_cast<int32_t>(tj * kTile), static_cast<int32_t>(row0),
                              base + kOffQRow + b * kQTileBytes, pol);
          else
            tma_store_2d(&tm_qrow, static_cast<int32_t>(tj * kTile), static_cast<int32_t>(row0),
                         base + kOffQRow + b * kQTileBytes);
          if (!(kMode == kDual && kSRowAfter) &&
              in_buf(s_row + (ti * TN + tj) * kAtomBytes, kAtomBytes, s_row,
                     static_cast<uint64_t>(N) * Mrows / 32, &g_mxq_status))
            bulk_store(s_row + (ti * TN + tj) * kAtomBytes, base + kOffSRow + b * kAtomBytes,
                       kAtomBytes);
        }
        if (R::kCol) {
          if (MXQ_DUAL_L2_HINTS & 2)
            tma_store_2d_hint(&tm_qcol, static_cast<int32_t>(row0), static_cast<int32_t>(tj * kTile),
                              base + kOffQCol + b * kQTileBytes, pol);
          else
            tma_store_2d(&tm_qcol, static_cast<int32_t>(row0), static_cast<int32_t>(tj * kTile),
                         base + kOffQCol + b * kQTileBytes);
        }
        if (kMode == kDual) {
          // this tile's s_col atom: its place in the group's slab, or a zero
          // atom for rows past offs[G-1]
          const int64_t grow = grow0 + row0;  // the tile's first row in the full tensor
          uint8_t* dst;
          uint32_t src;
          if (grow < end_rows) {
            int64_t lo = 0, hi = Mtot;
            if (offs != nullptr) {
              const int g = group_of_row(s_offs, G, grow);
              lo = g ? s_offs[g - 1] : 0;
              hi = s_offs[g];
            }
            const int64_t atoms_per_nblock = (hi - lo) / kTile;  // (hi-lo)/32 scale cols / 4
            dst = s_col + static_cast<int64_t>(N) * lo / 32 +
                  (tj * atoms_per_nblock + (grow - lo) / kTile) * kAtomBytes;
            src = MXQ_DUAL_SCOL_DEFER
                      ? base + kOffSColRing + static_cast<uint32_t>(k % kSColSlots) * kAtomBytes
                      : base + kOffSCol + b * kAtomBytes;
          } else {
            dst = s_col + static_cast<int64_t>(N) * end_rows / 32 +
                  (((grow - end_rows) / kTile) * TN + tj) * kAtomBytes;
            src = base + kOffZero;
          }
          if (!in_buf(dst, kAtomBytes, s_col, static_cast<uint64_t>(N) * Mtot / 32, &g_mxq_status))
            dst = nullptr;
          if (MXQ_DUAL_SCOL_DEFER) {
            // the data stores first; the atom once they have read their
            // tiles.  Its ring slot is rewritten four tiles later, by then
            // well past this store (every wait_read<0> covers it).
            bulk_commit();
            bulk_wait_read<0>();
            if (dst != nullptr) bulk_store(dst, src, kAtomBytes);
            if (kSRowAfter && in_buf(s_row + (ti * TN + tj) * kAtomBytes, kAtomBytes, s_row,
                                     static_cast<uint64_t>(N) * Mrows / 32, &g_mxq_status))
              bulk_store(s_row + (ti * TN + tj) * kAtomBytes,
                         base + kOffSRowRing + static_cast<uint32_t>(k % kSColSlots) * kAtomBytes,
                         kAtomBytes);
            bulk_commit();
          } else {
            if (dst != nullptr) bulk_store(dst, src, kAtomBytes);
            bulk_commit();
            bulk_wait_read<0>();
          }
        } else {
          bulk_commit();
          bulk_wait_read<0>();
        }
        mbar_arrive(bars.oempty(b));
      }
    }
    pdl_trigger_at_end();
    if (lane == 0) bulk_wait_all<0>();
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kMode>
bool ensure_smem_attr(int dev) {
  static std::mutex mu;
  static bool done[64] = {};
  if (dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(mxq_tile_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

int check_shape(int64_t M, int64_t N) {
  if (M < 0 || N < 0 || M % kTile != 0 || N % kTile != 0 || M > INT32_MAX || N > INT32_MAX)
    return MXQ_EBADSHAPE;
  return MXQ_OK;
}

// Encode the tensor maps (unused ones get a valid map of x) and launch one
// persistent wave: min(tiles, SMs) CTAs.
template <int kMode>
int launch_tiles(const void* x, int64_t M, int64_t N, const int32_t* offs, int32_t G,
                 uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                 cudaStream_t stream, int64_t grow0 = 0, int64_t Mtot = -1) {
  if (Mtot < 0) Mtot = M;
  int dev = 0;
  const int sms = sm_count_current_device(&dev);
  if (sms <= 0 || !ensure_smem_attr<kMode>(dev)) return MXQ_ECUDA;
  CUtensorMap tm_x, tm_qrow, tm_qcol;
  if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, N, M, 2ull * N, 64, kTile))
    return MXQ_ECUDA;
  if (q_row) {
    if (!encode_2d(&tm_qrow, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_row, N, M, N, kTile, kTile))
      return MXQ_ECUDA;
  } else {
    tm_qrow = tm_x;
  }
  if (q_col) {
    if (!encode_2d(&tm_qcol, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_col, M, N, M, kTile, kTile))
      return MXQ_ECUDA;
  } else {
    tm_qcol = tm_x;
  }
  const int64_t T = (M / kTile) * (N / kTile);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T < sms ? T : sms));
  cfg.blockDim = dim3(Roles<kMode>::kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, mxq_tile_kernel<kMode>, tm_x, tm_qrow, tm_qcol, offs,
                         static_cast<int>(G), static_cast<int>(M), static_cast<int>(N),
                         static_cast<int>(grow0), static_cast<int>(Mtot), s_row, s_col);
  return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}

}  // namespace

extern "C" int mxq_quantize_2d_dual(const void* x, int64_t M, int64_t N, const int32_t* offs,
                                    int32_t G, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                    uint8_t* s_col, cudaStream_t stream) {
  int rc = check_shape(M, N);
  if (rc != MXQ_OK) return rc;
  if (offs == nullptr ? G != 0 : (G < 1 || G > MXQ_MAX_GROUPS)) return MXQ_EBADOFFS;
  if (offs != nullptr && !aligned_to(offs, 4)) return MXQ_EALIGN;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!x || !q_row || !s_row || !q_col || !s_col) return MXQ_ENULL;
  if (!aligned_to(x, 16) || !aligned_to(q_row, 16) || !aligned_to(s_row, 16) ||
      !aligned_to(q_col, 16) || !aligned_to(s_col, 16))
    return MXQ_EALIGN;
  const uint64_t MN = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  const ByteRange r[6] = {
      {reinterpret_cast<uintptr_t>(x), 2 * MN},
      {reinterpret_cast<uintptr_t>(q_row), MN},
      {reinterpret_cast<uintptr_t>(q_col), MN},
      {reinterpret_cast<uintptr_t>(s_row), MN / 32},
      {reinterpret_cast<uintptr_t>(s_col), MN / 32},
      {reinterpret_cast<uintptr_t>(offs), offs ? 4ull * static_cast<uint64_t>(G) : 0ull},
  };
  if (ranges_overlap(r, 6)) return MXQ_EOVERLAP;
  return launch_tiles<kDual>(x, M, N, offs, G, q_row, s_row, q_col, s_col, stream);
}

extern "C" int mxq_quantize_2d_dual_rows(const void* x, int64_t rows, int64_t N, int64_t row0,
                                         int64_t M, const int32_t* offs, int32_t G, uint8_t* q_row,
                                         uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                         cudaStream_t stream) {
  int rc = check_shape(rows, N);
  if (rc != MXQ_OK) return rc;
  rc = check_shape(M, N);
  if (rc != MXQ_OK) return rc;
  // the band inside [0, M), with no int64 sum that could wrap for a far row0
  if (row0 < 0 || row0 % kTile != 0 || row0 > M || rows > M - row0) return MXQ_EBADSHAPE;
  if (offs == nullptr ? G != 0 : (G < 1 || G > MXQ_MAX_GROUPS)) return MXQ_EBADOFFS;
  if (offs != nullptr && !aligned_to(offs, 4)) return MXQ_EALIGN;
  if (rows == 0 || N == 0) return MXQ_OK;
  if (!x || !q_row || !s_row || !q_col || !s_col) return MXQ_ENULL;
  if (!aligned_to(x, 16) || !aligned_to(q_row, 16) || !aligned_to(s_row, 16) ||
      !aligned_to(q_col, 16) || !aligned_to(s_col, 16))
    return MXQ_EALIGN;
  const uint64_t RN = static_cast<uint64_t>(rows) * static_cast<uint64_t>(N);
  const uint64_t MN = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  const ByteRange r[6] = {
      {reinterpret_cast<uintptr_t>(x), 2 * RN},
      {reinterpret_cast<uintptr_t>(q_row), RN},
      {reinterpret_cast<uintptr_t>(q_col), RN},
      {reinterpret_cast<uintptr_t>(s_row), RN / 32},
      {reinterpret_cast<uintptr_t>(s_col), MN / 32},
      {reinterpret_cast<uintptr_t>(offs), offs ? 4ull * static_cast<uint64_t>(G) : 0ull},
  };
  if (ranges_overlap(r, 6)) return MXQ_EOVERLAP;
  return launch_tiles<kDual>(x, rows, N, offs, G, q_row, s_row, q_col, s_col, stream, row0, M);
}

extern "C" int mxq_quantize_1x32(const void* x, int64_t M, int64_t N, uint8_t* q_row,
                                 uint8_t* s_row, cudaStream_t stream) {
  int rc = check_shape(M, N);
  if (rc != MXQ_OK) return rc;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!x || !q_row || !s_row) return MXQ_ENULL;
  if (!aligned_to(x, 16) || !aligned_to(q_row, 16) || !aligned_to(s_row, 16)) return MXQ_EALIGN;
  const uint64_t MN = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  const ByteRange r[3] = {{reinterpret_cast<uintptr_t>(x), 2 * MN},
                          {reinterpret_cast<uintptr_t>(q_row), MN},
                          {reinterpret_cast<uintptr_t>(s_row), MN / 32}};
  if (ranges_overlap(r, 3)) return MXQ_EOVERLAP;
  return launch_tiles<kRowOnly>(x, M, N, nullptr, 0, q_row, s_row, nullptr, nullptr, stream);
}

extern "C" int mxq_quantize_32x1(const void* x, int64_t M, int64_t N, uint8_t* q_col,
                                 uint8_t* s_rm, cudaStream_t stream) {
  int rc = check_shape(M, N);
  if (rc != MXQ_OK) return rc;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!x || !q_col || !s_rm) return MXQ_ENULL;
  if (!aligned_to(x, 16) || !aligned_to(q_col, 16) || !aligned_to(s_rm, 16)) return MXQ_EALIGN;
  const uint64_t MN = static_cast<uint64_t>(M) * static_cast<uint64_t>(N);
  const ByteRange r[3] = {{reinterpret_cast<uintptr_t>(x), 2 * MN},
                          {reinterpret_cast<uintptr_t>(q_col), MN},
                          {reinterpret_cast<uintptr_t>(s_rm), MN / 32}};
  if (ranges_overlap(r, 3)) return MXQ_EOVERLAP;
  return launch_tiles<kColOnly>(x, M, N, nullptr, 0, nullptr, nullptr, q_col, s_rm, stream);
}

namespace {
// Diagnostic kernel: one warp waits, with the pipelines' bounded wait, on an
// mbarrier that nothing ever arrives on, so the wait runs out after limit_ns
// and records MXQ_DEV_TIMEOUT exactly as a stalled pipeline would.
__global__ void mxq_selftest_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    mbar_init_fence();
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, &g_mxq_status,
                                    MXQ_DEV_TIMEOUT, limit_ns);
  (void)__all_sync(0xFFFFFFFFu, ok);
}

}  // namespace

extern "C" int mxq_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1000000ull || limit_ns > 4000000000ull) return MXQ_EBADSHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, mxq_selftest_timeout_kernel, limit_ns) == cudaSuccess
             ? MXQ_OK
             : MXQ_ECUDA;
}

namespace mxq {
int mx9_status_read(unsigned int* out, bool clear);      // mx9.cu
int compose_status_read(unsigned int* out, bool clear);  // mxq_compose.cu
int cols_status_read(unsigned int* out, bool clear);     // mx_cols_tma.cu
int packed_status_read(unsigned int* out, bool clear);   // mx_packed.cu
int mma_status_read(unsigned int* out, bool clear);      // mxq_mma_check.cu
}

// The device status word is the OR of the per-file words of the kernels.
extern "C" int mxq_device_status(uint32_t* out, int clear) {
  if (!out) return MXQ_ENULL;
  unsigned int v = 0, w = 0;
  if (cudaMemcpyFromSymbol(&v, g_mxq_status, sizeof v) != cudaSuccess) return MXQ_ECUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_mxq_status, &zero, sizeof zero) != cudaSuccess) return MXQ_ECUDA;
  }
  unsigned int c = 0;
  int rc = mxq::mx9_status_read(&w, clear != 0);
  if (rc != MXQ_OK) return rc;
  rc = mxq::compose_status_read(&c, clear != 0);
  if (rc != MXQ_OK) return rc;
  unsigned int t = 0, k = 0;
  rc = mxq::cols_status_read(&t, clear != 0);
  if (rc != MXQ_OK) return rc;
  rc = mxq::packed_status_read(&k, clear != 0);
  if (rc != MXQ_OK) return rc;
  unsigned int g = 0;
  rc = mxq::mma_status_read(&g, clear != 0);
  if (rc != MXQ_OK) return rc;
  *out = v | w | c | t | k | g;
  return MXQ_OK;
}

extern "C" int mxq_last_device_status(uint32_t* out, int clear) {
  return mxq_device_status(out, clear);
}
