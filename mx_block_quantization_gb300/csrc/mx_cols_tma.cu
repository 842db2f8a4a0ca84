// mx_cols_tma.cu -- MX9 / MX6 records blocked along columns (axis 0) for
// tensors that TMA moves as tiles: a persistent, warp-specialized transpose
// with 2-D TMA loads and stores.
//
// AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
// pack/unpack": the packed single-tensor form and its suite's blocking along
// an axis.  Block b = c * ceil(rows / 16) + j covers rows 16j..16j+15 of
// column c, so the packed tensor is [cols, nbl * R] bytes (nbl = blocks per
// column, R = record bytes) and one 128-row tile of a column is one run of 8
// consecutive records.
//
// Pack (x -> records):
// * producer warp: a tile is 128 rows x 512 bytes of x (128 fp32 or 256 bf16
//   columns), four 128-byte wide boxes loaded with the 128-byte swizzle (16-byte
//   chunk c of row r at c ^ (r % 8)) into a ring of stages;
// * 16 consumer warps: lane (box, chunk c, half h, block j) reads 16 rows x 8
//   bytes with 64-bit shared loads (a half-warp covers the 16 (c, h) of a box:
//   no bank conflict), releases the stage, quantizes its 2 fp32 or 4 bf16
//   blocks and stages their records at their place in the tile's runs, laid out
//   exactly as the packed tensor's [columns, 8 R] box;
// * storer warp: one 2-D TMA store per tile writes the runs (box: 8 R bytes x
//   the tile's columns); rows past the tensor end were zero-filled on load and
//   records past it are clipped by the store.
// Unpack (records -> x): the producer loads a tile's runs with one 2-D TMA
// load into a ring; consumer lanes decode their records into a swizzled tile
// (two buffers), and after one barrier of the consumer warps each warp writes
// whole tile rows, 16 bytes per lane: 512 contiguous bytes per store.  Two
// other forms measured slower: 2-D TMA stores of the staged tile (per-tile
// waits on the store reads; also, a swizzled TMA store clips a row in 16-byte
// units: a row of 37 fp32 had its last 16 bytes written whole), and stores
// straight from the decoding lanes (8 bytes per lane, 8 separate 32-byte
// sectors per store instruction, one L2 request each).  Unpack takes rows of
// whole 16-byte pieces.  Pack has no such limit: what its loads read past a
// row end reaches only records past the last column, which its store drops.
//
// Lane layout: warp w takes box w % 4; its lane with chunk c, half h and
// jh = lane / 16 takes block j = ((c / 2 + w / 4) % 4) + 4 jh.  Among the lanes
// that share a record word offset class, the 8 blocks are all different, so
// staging a record (and reading one back) costs at most 2 wavefronts; bf16
// lanes with odd c visit their columns in the order e ^ 1 for the same reason.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_block.cuh"
#include "mxq_check.cuh"
#include "mxq.h"
#include "mxq_device.cuh"
#include "mxq_host.h"

#ifndef MXQ_COLS_TMA_STAGES
#define MXQ_COLS_TMA_STAGES 2
#endif
#ifndef MXQ_COLS_TMA_UNPACK_RING_KB
#define MXQ_COLS_TMA_UNPACK_RING_KB 72
#endif
// unpack tile order (tile_at): tile rows per group, 1 = across a band of rows
// first (x rows move as one run), 0 = down whole columns first (a column's
// records move as one run)
#ifndef MXQ_COLS_TMA_UNPACK_GROUP
#define MXQ_COLS_TMA_UNPACK_GROUP 1
#endif
#ifndef MXQ_COLS_TMA_UNPACK_GROUP_MX9_F32  // the MX9 fp32 unpack measured faster in groups
#define MXQ_COLS_TMA_UNPACK_GROUP_MX9_F32 3
#endif

namespace {

using namespace mxq;

// Sticky status word of this file's kernels (MXQ_DEV_* bits).
__device__ unsigned int g_cols_status = 0;

constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 2) * 32;  // pack: + producer warp + storer warp
constexpr int kUnpackThreads = (kConsumerWarps + 1) * 32;  // unpack: + producer warp
constexpr int kTileRows = 128;                        // 8 blocks of 16 rows
constexpr int kBoxes = 4;                             // 128-byte wide boxes per tile
constexpr uint32_t kBoxBytes = kTileRows * 128u;      // 16 KB
constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;   // 64 KB

template <bool kBF16, int kFmt>
struct ColsTma {
  static constexpr int kEsize = kBF16 ? 2 : 4;
  static constexpr int kBoxCols = 128 / kEsize;
  static constexpr int kTileCols = kBoxes * kBoxCols;
  static constexpr int kColsPerLane = 8 / kEsize;  // columns in 8 bytes of a row
  static constexpr int kRecord = kFmt == MXQ_FMT_MX9 ? MXQ_MX9_RECORD_BYTES : MXQ_MX6_RECORD_BYTES;
  static constexpr int kOffset = kFmt == MXQ_FMT_MX9 ? 6 : 3;
  // unpack tile order (tile_at): tile rows per group
  static constexpr int kUnpackGroup = kFmt == MXQ_FMT_MX9 && !kBF16 ? MXQ_COLS_TMA_UNPACK_GROUP_MX9_F32
                                                                    : MXQ_COLS_TMA_UNPACK_GROUP;
  static constexpr int kQMax = kFmt == MXQ_FMT_MX9 ? 127 : 15;
  static constexpr uint32_t kRunBytes = 8u * kRecord;               // one column of a tile
  static constexpr uint32_t kRecTileBytes = kTileCols * kRunBytes;  // one tile's records
  // pack: ring of x tiles, two record buffers; unpack: a ring of record
  // tiles of about MXQ_COLS_TMA_UNPACK_RING_KB (2 to 8 stages), two x tiles
  static constexpr int kPackStages = MXQ_COLS_TMA_STAGES;
  static constexpr uint32_t kPackData = kPackStages * kTileBytes + 2u * kRecTileBytes;
  static constexpr int kRingFit = static_cast<int>(MXQ_COLS_TMA_UNPACK_RING_KB * 1024u / kRecTileBytes);
  static constexpr int kUnpackStages = kRingFit < 2 ? 2 : kRingFit > 8 ? 8 : kRingFit;
  static constexpr uint32_t kUnpackData = kUnpackStages * kRecTileBytes + 2u * kTileBytes;
  // barriers (full, empty per stage; out-full, out-free per buffer), abort flag
  static constexpr uint32_t kBarBytes = 8u * (2 * 8 + 4) + 16u;
  static constexpr uint32_t kPackSmem = kPackData + kBarBytes + 1024u;  // + alignment
  static constexpr uint32_t kUnpackSmem = kUnpackData + kBarBytes + 1024u;
  static_assert(kRecTileBytes % 1024u == 0, "buffers stay 1024-byte aligned");
  static_assert(kPackSmem <= 227u * 1024u && kUnpackSmem <= 227u * 1024u, "shared memory budget");
};

__device__ __forceinline__ void lds64(uint32_t a, uint32_t* x, uint32_t* y) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(*x), "=r"(*y) : "r"(a));
}

__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}

// Exact float of a small integer (|q| < 2^22): the bits of 1.5 * 2^23 + q,
// minus 1.5 * 2^23.
__device__ __forceinline__ float int_float_exact(int32_t q) {
  float r;
  asm("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(__int_as_float(0x4B400000 + q)), "f"(-12582912.0f));
  return r;
}

// The 16 values q * 2^k of the record at shared address rec.
template <int kFmt>
__device__ __forceinline__ void decode_record(uint32_t rec, float* v) {
  constexpr int kOff = kFmt == MXQ_FMT_MX9 ? 6 : 3;
  uint32_t head;
  int q[16];
  if (kFmt == MXQ_FMT_MX9) {
    // five aligned words cover the 18 bytes; the record starts 0 or 2 bytes in
    const uint32_t a = rec & ~3u, odd = rec & 2u;
    uint32_t w[5];
#pragma unroll
    for (int m = 0; m < 5; ++m) w[m] = lds32(a + 4u * m);
    head = __byte_perm(w[0], 0u, odd ? 0x4432 : 0x4410);
    const uint32_t sel = odd ? 0x7654u : 0x5432u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int32_t d = static_cast<int32_t>(__byte_perm(w[k], w[k + 1], sel));
      q[4 * k] = (d << 24) >> 24;
      q[4 * k + 1] = (d << 16) >> 24;
      q[4 * k + 2] = (d << 8) >> 24;
      q[4 * k + 3] = d >> 24;
    }
  } else {
    const uint32_t w0 = lds32(rec), w1 = lds32(rec + 4u), w2 = lds32(rec + 8u);
    head = w0 & 0xFFFFu;
    const uint64_t d = static_cast<uint64_t>(w0 >> 16) | (static_cast<uint64_t>(w1) << 16) |
                       (static_cast<uint64_t>(w2) << 48);
    const uint32_t d_hi = w2 >> 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = 5 * i;
      const uint32_t c = b + 5 <= 64 ? static_cast<uint32_t>(d >> b) & 0x1Fu
                         : b >= 64   ? (d_hi >> (b - 64)) & 0x1Fu
                                     : (static_cast<uint32_t>(d >> b) | (d_hi << (64 - b))) & 0x1Fu;
      q[i] = static_cast<int>(c << 27) >> 27;
    }
  }
  // 2^k with k = max(E - off - prime, -126): exponent field max(eb8 - off - prime, 1)
  const int eb8 = static_cast<int>(head & 0xFFu);
  const uint32_t bits = head >> 8;
  const float s_keep = __uint_as_float(static_cast<uint32_t>(max(eb8 - kOff, 1)) << 23);
  const float s_dem = __uint_as_float(static_cast<uint32_t>(max(eb8 - kOff - 1, 1)) << 23);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    v[i] = fmul_rn_noftz(int_float_exact(q[i]), (bits >> (i / 2)) & 1u ? s_dem : s_keep);
}

// Per-lane geometry shared by both directions.
template <bool kBF16, int kFmt>
struct LaneGeo {
  using C = ColsTma<kBF16, kFmt>;
  int c, j, cx;     // chunk, block, column-order flip (bf16, odd chunks)
  int col0;         // this lane's first column in the tile
  uint32_t xoff;    // byte offset of (row 16j, chunk c, half h) in a tile, before the swizzle
  uint32_t recoff;  // byte offset of this lane's first column's record j in a record tile
  __device__ __forceinline__ LaneGeo(int warp, int lane) {
    const int bx = warp & 3, rot = warp >> 2;
    c = lane & 7;
    const int h = (lane >> 3) & 1, jh = lane >> 4;
    j = (((c >> 1) + rot) & 3) + 4 * jh;
    cx = kBF16 ? (c & 1) : 0;
    xoff = static_cast<uint32_t>(bx) * kBoxBytes + static_cast<uint32_t>(16 * j) * 128u + 8u * h;
    col0 = bx * C::kBoxCols + c * (16 / C::kEsize) + h * C::kColsPerLane;
    recoff = static_cast<uint32_t>(col0) * C::kRunBytes + static_cast<uint32_t>(j) * C::kRecord;
  }
  // row i (0..15) of this lane's block in the swizzled tile ((16j + i) % 8 == i % 8)
  __device__ __forceinline__ uint32_t row(int i) const {
    return xoff + static_cast<uint32_t>(i) * 128u + (static_cast<uint32_t>(c ^ (i & 7)) << 4);
  }
};

// mbarriers after the data: full / empty per ring stage, and out-full /
// out-free per staged record buffer (pack only), then the CTA's abort flag.
struct Barriers {
  uint32_t base;
  int stages;
  __device__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ uint32_t empty(int s) const { return base + 8u * (stages + s); }
  __device__ uint32_t ofull(int b) const { return base + 8u * (2 * stages + b); }
  __device__ uint32_t ofree(int b) const { return base + 8u * (2 * stages + 2 + b); }
  __device__ uint32_t flag() const { return base + 8u * (2 * stages + 4); }
};

__device__ __forceinline__ void init_barriers(const Barriers& b, volatile uint32_t* abort_flag) {
  for (int s = 0; s < b.stages; ++s) {
    mbar_init(b.full(s), 1);
    mbar_init(b.empty(s), kConsumerWarps);
  }
  for (int o = 0; o < 2; ++o) {
    mbar_init(b.ofull(o), kConsumerWarps);
    mbar_init(b.ofree(o), 1);
  }
  *abort_flag = 0u;
  mbar_init_fence();
}

// tiles_r x tiles_c tiles; CTA b takes tiles b, b + grid, ... of the
// visiting order
__device__ __forceinline__ int64_t tiles_of_cta(int64_t ntiles) {
  return static_cast<int64_t>(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
}

// Barrier of the consumer warps (named barrier 1) returning the AND of every
// consumer thread's flag.
__device__ __forceinline__ bool consumers_sync_and(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(flag)), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}

// Tile t in the visiting order: `group` tile rows at a time, column by
// column inside a group (group 1: across a band of rows first; 0: down whole
// columns first).
__device__ __forceinline__ void tile_at_rows(int64_t t, int64_t tiles_r, int64_t tiles_c,
                                             int64_t group, int64_t* tr, int64_t* tc) {
  if (group == 0) {
    *tc = t / tiles_r;
    *tr = t - *tc * tiles_r;
  } else if (group == 1) {
    *tr = t / tiles_c;
    *tc = t - *tr * tiles_c;
  } else {
    const int64_t per_group = group * tiles_c;
    const int64_t g = t / per_group;
    const int64_t local = t - g * per_group;
    const int64_t rows = tiles_r - g * group < group ? tiles_r - g * group : group;
    *tr = g * group + local % rows;
    *tc = local / rows;
  }
}

template <int kGroup>
__device__ __forceinline__ void tile_at(int64_t t, int64_t tiles_r, int64_t tiles_c, int64_t* tr,
                                        int64_t* tc) {
  tile_at_rows(t, tiles_r, tiles_c, kGroup, tr, tc);
}

template <bool kBF16, int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
    mx_pack_cols_tma_kernel(const __grid_constant__ CUtensorMap tm_x,
                            const __grid_constant__ CUtensorMap tm_rec, int32_t tiles_r,
                            int32_t tiles_c, int32_t group) {
  using C = ColsTma<kBF16, kFmt>;
  using R = MxRule<C::kOffset, C::kQMax>;
  constexpr int kStages = C::kPackStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t rec_base = base + kStages * kTileBytes;
  const Barriers bars{rec_base + 2u * C::kRecTileBytes, kStages};
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem_raw + (bars.flag() - raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t my = tiles_of_cta(static_cast<int64_t>(tiles_r) * tiles_c);
  if (tid == 0) init_barriers(bars, abort_flag);
  __syncthreads();
  pdl_wait();  // inputs may be the previous kernel's output
  pdl_trigger_at_start();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    tma_prefetch_desc(&tm_x);
    int64_t issued = 0;
    for (int64_t i = 0; i < my; ++i) {
      const int s = static_cast<int>(i % kStages);
      if (i >= kStages &&
          !mbar_wait_bounded(bars.empty(s), static_cast<uint32_t>(((i / kStages) - 1) & 1),
                             abort_flag, &g_cols_status, MXQ_DEV_TIMEOUT))
        break;
      int64_t tr, tc;
      tile_at_rows(blockIdx.x + i * static_cast<int64_t>(gridDim.x), tiles_r, tiles_c, group, &tr, &tc);
      mbar_arrive_expect_tx(bars.full(s), kTileBytes);
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)
        tma_load_2d(base + s * kTileBytes + b * kBoxBytes, &tm_x,
                    static_cast<int32_t>(tc * C::kTileCols + b * C::kBoxCols),
                    static_cast<int32_t>(tr * kTileRows), bars.full(s));
      issued = i + 1;
    }
    // drain (a no-op after a normal run: consumers waited for every stage)
    for (int64_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
      mbar_wait_drain(bars.full(static_cast<int>(i % kStages)), static_cast<uint32_t>((i / kStages) & 1));
    return;
  }
  if (warp == kConsumerWarps + 1) {
    // -------------------------------------------------------------- storer
    if (lane != 0) return;
    tma_prefetch_desc(&tm_rec);
    for (int64_t i = 0; i < my; ++i) {
      const int ob = static_cast<int>(i & 1);
      if (!mbar_wait_bounded(bars.ofull(ob), static_cast<uint32_t>((i >> 1) & 1), abort_flag,
                             &g_cols_status, MXQ_DEV_TIMEOUT))
        break;
      int64_t tr, tc;
      tile_at_rows(blockIdx.x + i * static_cast<int64_t>(gridDim.x), tiles_r, tiles_c, group, &tr, &tc);
      tma_store_2d(&tm_rec, static_cast<int32_t>(tr * C::kRunBytes),
                   static_cast<int32_t>(tc * C::kTileCols), rec_base + ob * C::kRecTileBytes);
      bulk_commit();
      bulk_wait_read<1>();  // the store of tile i - 1 is done reading its buffer
      if (i >= 1) mbar_arrive(bars.ofree(ob ^ 1));
    }
    bulk_wait_all<0>();
    return;
  }

  // -------------------------------------------------------------- consumers
  const LaneGeo<kBF16, kFmt> geo(warp, lane);
  for (int64_t i = 0; i < my; ++i) {
    const int s = static_cast<int>(i % kStages);
    bool ok = mbar_wait_bounded(bars.full(s), static_cast<uint32_t>((i / kStages) & 1), abort_flag,
                                &g_cols_status, MXQ_DEV_TIMEOUT);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    const uint32_t tile = base + s * kTileBytes;
    uint32_t u[16], v[16];  // rows 16j..16j+15, the two words of this lane's 8 bytes
#pragma unroll
    for (int r = 0; r < 16; ++r) lds64(tile + geo.row(r), &u[r], &v[r]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.empty(s));
    const int ob = static_cast<int>(i & 1);
    if (i >= 2)
      ok = mbar_wait_bounded(bars.ofree(ob), static_cast<uint32_t>(((i >> 1) - 1) & 1), abort_flag,
                             &g_cols_status, MXQ_DEV_TIMEOUT);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    const uint32_t rec = rec_base + ob * C::kRecTileBytes + geo.recoff;
    if (kBF16) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ep = e ^ geo.cx;  // column of this lane handled now
        const uint32_t* src = e < 2 ? u : v;
        const uint32_t sel = (ep & 1) ? 0x7632u : 0x5410u;
        uint32_t w[8], h[8], eb8, bits;
#pragma unroll
        for (int p = 0; p < 8; ++p) w[p] = __byte_perm(src[2 * p], src[2 * p + 1], sel);
        R::block_bf16(w, h, &eb8, &bits);
        stage_record<kFmt>(rec + static_cast<uint32_t>(ep) * C::kRunBytes, eb8, bits, h);
      }
    } else {
      uint32_t h[8], eb8, bits;
      R::block_f32(u, h, &eb8, &bits);
      stage_record<kFmt>(rec, eb8, bits, h);
      R::block_f32(v, h, &eb8, &bits);
      stage_record<kFmt>(rec + C::kRunBytes, eb8, bits, h);
    }
    fence_proxy_async_smem();  // staged records before the TMA store reads them
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.ofull(ob));
  }
}

template <bool kBF16, int kFmt>
__global__ void __launch_bounds__(kUnpackThreads, 1)
    mx_unpack_cols_tma_kernel(const __grid_constant__ CUtensorMap tm_rec, uint8_t* __restrict__ y,
                              int64_t rows, int64_t cols, int64_t ld, int32_t tiles_r,
                              int32_t tiles_c) {
  using C = ColsTma<kBF16, kFmt>;
  constexpr int kStages = C::kUnpackStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ytile_base = base + kStages * C::kRecTileBytes;
  const Barriers bars{ytile_base + 2u * kTileBytes, kStages};
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem_raw + (bars.flag() - raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t my = tiles_of_cta(static_cast<int64_t>(tiles_r) * tiles_c);
  if (tid == 0) init_barriers(bars, abort_flag);
  __syncthreads();
  pdl_wait();  // inputs may be the previous kernel's output
  pdl_trigger_at_start();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    tma_prefetch_desc(&tm_rec);
    int64_t issued = 0;
    for (int64_t i = 0; i < my; ++i) {
      const int s = static_cast<int>(i % kStages);
      if (i >= kStages &&
          !mbar_wait_bounded(bars.empty(s), static_cast<uint32_t>(((i / kStages) - 1) & 1),
                             abort_flag, &g_cols_status, MXQ_DEV_TIMEOUT))
        break;
      int64_t tr, tc;
      tile_at<C::kUnpackGroup>(blockIdx.x + i * static_cast<int64_t>(gridDim.x), tiles_r, tiles_c, &tr, &tc);
      mbar_arrive_expect_tx(bars.full(s), C::kRecTileBytes);
      tma_load_2d(base + s * C::kRecTileBytes, &tm_rec, static_cast<int32_t>(tr * C::kRunBytes),
                  static_cast<int32_t>(tc * C::kTileCols), bars.full(s));
      issued = i + 1;
    }
    for (int64_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
      mbar_wait_drain(bars.full(static_cast<int>(i % kStages)), static_cast<uint32_t>((i / kStages) & 1));
    return;
  }

  // -------------------------------------------------------------- consumers
  // Each lane decodes its 2 (fp32) or 4 (bf16) records into the swizzled tile
  // buffer of this tile (two buffers, alternating); after one barrier of the
  // 16 consumer warps, warp w writes rows w, w + 16, ... of the tile, a lane
  // one 16-byte piece (box lane / 8, chunk lane % 8): 512 contiguous bytes per
  // store instruction.  The barrier also ANDs every thread's wait result, so
  // that on a timeout all consumer warps leave together.
  const LaneGeo<kBF16, kFmt> geo(warp, lane);
  const int64_t pitch = ld * C::kEsize;
  const int pbox = lane >> 3, pchunk = lane & 7;
  const int64_t pcol = pbox * C::kBoxCols + pchunk * (16 / C::kEsize);  // piece column in a tile
  for (int64_t i = 0; i < my; ++i) {
    const int s = static_cast<int>(i % kStages);
    const bool ok = mbar_wait_bounded(bars.full(s), static_cast<uint32_t>((i / kStages) & 1),
                                      abort_flag, &g_cols_status, MXQ_DEV_TIMEOUT);
    const uint32_t ytile = ytile_base + static_cast<uint32_t>(i & 1) * kTileBytes;
    if (ok) {
      const uint32_t rec = base + s * C::kRecTileBytes + geo.recoff;
      uint32_t u[16], v[16];
      if (kBF16) {
        // columns e ^ cx: decode two, keep their bf16 halves (exact: at most 8
        // significant bits), the first pair into u, the second into v
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float a[16], b[16];
          decode_record<kFmt>(rec + static_cast<uint32_t>((2 * half) ^ geo.cx) * C::kRunBytes, a);
          decode_record<kFmt>(rec + static_cast<uint32_t>((2 * half + 1) ^ geo.cx) * C::kRunBytes, b);
          const uint32_t sel = geo.cx ? 0x3276u : 0x7632u;
          uint32_t* dst = half ? v : u;
#pragma unroll
          for (int r = 0; r < 16; ++r) dst[r] = __byte_perm(__float_as_uint(a[r]), __float_as_uint(b[r]), sel);
        }
      } else {
        float a[16];
        decode_record<kFmt>(rec, a);
#pragma unroll
        for (int r = 0; r < 16; ++r) u[r] = __float_as_uint(a[r]);
        decode_record<kFmt>(rec + C::kRunBytes, a);
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = __float_as_uint(a[r]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(s));
#pragma unroll
      for (int r = 0; r < 16; ++r) sts64(ytile + geo.row(r), u[r], v[r]);
    }
    // the tile complete (and buffer i & 1 of tile i - 2 no longer read: each
    // warp read it before its writes of tile i - 1 and this barrier's previous
    // round); all threads' wait results
    if (!consumers_sync_and(ok)) break;
    int64_t tr, tc;
    tile_at<C::kUnpackGroup>(blockIdx.x + i * static_cast<int64_t>(gridDim.x), tiles_r, tiles_c, &tr, &tc);
    const int64_t col = tc * C::kTileCols + pcol;
    if (col < cols) {  // whole 16-byte pieces: cols * element size is a multiple of 16
      const int64_t row0 = tr * kTileRows;
      uint8_t* p = y + row0 * pitch + col * C::kEsize;
#pragma unroll
      for (int k = 0; k < kTileRows / kConsumerWarps; ++k) {
        const int r = warp + kConsumerWarps * k;
        if (row0 + r < rows) {
          const uint4 q = lds128(ytile + static_cast<uint32_t>(pbox) * kBoxBytes +
                                 static_cast<uint32_t>(r) * 128u +
                                 (static_cast<uint32_t>(pchunk ^ (r & 7)) << 4));
          if (in_buf(p + r * pitch, 16, y, static_cast<uint64_t>((rows - 1) * ld + cols) * C::kEsize,
                     &g_cols_status))
            __stcs(reinterpret_cast<uint4*>(p + r * pitch), q);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

bool encode(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto enc = driver_tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encode the two tensor maps (x or y, and the packed tensor) of a tensor
// that cols_tma_ok accepted.
template <bool kBF16, int kFmt>
bool encode_maps(const void* x, int64_t rows, int64_t cols, int64_t ld, const void* packed,
                 CUtensorMap* tm_x, CUtensorMap* tm_rec) {
  using C = ColsTma<kBF16, kFmt>;
  const int64_t line = (rows + 15) / 16 * C::kRecord;
  return encode(tm_x, kBF16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, x,
                static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                static_cast<uint64_t>(ld) * C::kEsize, C::kBoxCols, kTileRows,
                CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode(tm_rec, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, static_cast<uint64_t>(line),
                static_cast<uint64_t>(cols), static_cast<uint64_t>(line), C::kRunBytes, C::kTileCols,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// One persistent wave: min(tiles, SMs) CTAs of one per SM.
template <auto kernel, typename... Args>
int launch_wave(uint32_t smem, int64_t tiles, int threads, cudaStream_t stream, Args... args) {
  int dev = 0;
  const int sms = sm_count_current_device(&dev);
  if (sms <= 0 || dev < 0 || dev >= 64) return MXQ_ECUDA;
  static bool attr_done[64] = {};  // benign race: the same attribute set twice
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MXQ_ECUDA;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  allow_programmatic_launch(&cfg, &attr);
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? MXQ_OK : MXQ_ECUDA;
}

// Tile rows per group of the pack's tile order.  An MX9 run of 8 records (144
// bytes) starts 16 bytes into a 32-byte sector on every other tile row, so the
// two halves of such a sector come from tiles (tr, tc) and (tr + 1, tc).  In
// row-band order the bf16 MX9 pack fell to 4100-4180 GB/s at 32768x16384 and
// 5263 at 24576x16384 (6430 walking pairs of tile rows), while at 8192 columns
// the row-band order measured best (pairs cost 3.5%): pairs from 16384 columns
// on, measured; fp32 MX9 measured as well or better in pairs at every size;
// MX6 runs (96 bytes) never split a sector and keep the row-band order.
template <bool kBF16, int kFmt>
int pack_group(int64_t cols) {
  if (kFmt != MXQ_FMT_MX9) return 1;
  return kBF16 && cols <= 8192 ? 1 : 2;
}

template <bool kBF16, int kFmt>
int launch_pack(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* packed,
                cudaStream_t stream) {
  using C = ColsTma<kBF16, kFmt>;
  CUtensorMap tm_x, tm_rec;
  if (!encode_maps<kBF16, kFmt>(x, rows, cols, ld, packed, &tm_x, &tm_rec)) return kColsTmaDeclined;
  const int64_t tiles_r = (rows + kTileRows - 1) / kTileRows;
  const int64_t tiles_c = (cols + C::kTileCols - 1) / C::kTileCols;
  return launch_wave<mx_pack_cols_tma_kernel<kBF16, kFmt>>(
      C::kPackSmem, tiles_r * tiles_c, kThreads, stream, tm_x, tm_rec,
      static_cast<int32_t>(tiles_r), static_cast<int32_t>(tiles_c),
      static_cast<int32_t>(pack_group<kBF16, kFmt>(cols)));
}

template <bool kBF16, int kFmt>
int launch_unpack(const uint8_t* packed, void* y, int64_t rows, int64_t cols, int64_t ld,
                  cudaStream_t stream) {
  using C = ColsTma<kBF16, kFmt>;
  CUtensorMap tm_y, tm_rec;
  if (!encode_maps<kBF16, kFmt>(y, rows, cols, ld, packed, &tm_y, &tm_rec)) return kColsTmaDeclined;
  const int64_t tiles_r = (rows + kTileRows - 1) / kTileRows;
  const int64_t tiles_c = (cols + C::kTileCols - 1) / C::kTileCols;
  return launch_wave<mx_unpack_cols_tma_kernel<kBF16, kFmt>>(
      C::kUnpackSmem, tiles_r * tiles_c, kUnpackThreads, stream, tm_rec, static_cast<uint8_t*>(y),
      rows, cols, ld, static_cast<int32_t>(tiles_r), static_cast<int32_t>(tiles_c));
}

}  // namespace

namespace mxq {

bool cols_tma_ok(const void* x, int dtype, int fmt, int64_t rows, int64_t cols, int64_t ld,
                 const void* packed, bool writes_x) {
  const int64_t esize = dtype == MXQ_F32 ? 4 : 2;
  const int64_t rec = fmt == MXQ_FMT_MX9 ? MXQ_MX9_RECORD_BYTES : MXQ_MX6_RECORD_BYTES;
  if (!aligned_to(x, 16) || !aligned_to(packed, 16) || (ld * esize) % 16 != 0) return false;
  // unpack stores whole 16-byte pieces of a row (what pack loads past a row
  // end only feeds records past the last column, which its store drops)
  if (writes_x && (cols * esize) % 16 != 0) return false;
  // tile coordinates stay in int32; row pitches below the tensor-map limit
  if (rows <= 0 || cols <= 0 || rows > INT32_MAX - 2 * kTileRows || cols > INT32_MAX - 1024)
    return false;
  if (ld * esize >= (int64_t{1} << 40)) return false;
  const int64_t line = (rows + 15) / 16 * rec;  // bytes of one column's records
  return line % 16 == 0 && line <= INT32_MAX;
}

int cols_tma_pack(const void* x, bool bf16, int fmt, int64_t rows, int64_t cols, int64_t ld,
                  uint8_t* packed, cudaStream_t stream) {
  if (bf16)
    return fmt == MXQ_FMT_MX9 ? launch_pack<true, MXQ_FMT_MX9>(x, rows, cols, ld, packed, stream)
                              : launch_pack<true, MXQ_FMT_MX6>(x, rows, cols, ld, packed, stream);
  return fmt == MXQ_FMT_MX9 ? launch_pack<false, MXQ_FMT_MX9>(x, rows, cols, ld, packed, stream)
                            : launch_pack<false, MXQ_FMT_MX6>(x, rows, cols, ld, packed, stream);
}

int cols_tma_unpack(const uint8_t* packed, int fmt, void* y, bool bf16, int64_t rows, int64_t cols,
                    int64_t ld, cudaStream_t stream) {
  if (bf16)
    return fmt == MXQ_FMT_MX9 ? launch_unpack<true, MXQ_FMT_MX9>(packed, y, rows, cols, ld, stream)
                              : launch_unpack<true, MXQ_FMT_MX6>(packed, y, rows, cols, ld, stream);
  return fmt == MXQ_FMT_MX9 ? launch_unpack<false, MXQ_FMT_MX9>(packed, y, rows, cols, ld, stream)
                            : launch_unpack<false, MXQ_FMT_MX6>(packed, y, rows, cols, ld, stream);
}

int cols_status_read(unsigned int* out, bool clear) {
  if (cudaMemcpyFromSymbol(out, g_cols_status, sizeof *out) != cudaSuccess) return MXQ_ECUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_cols_status, &zero, sizeof zero) != cudaSuccess) return MXQ_ECUDA;
  }
  return MXQ_OK;
}

}  // namespace mxq
