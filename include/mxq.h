/*
 * mxq.h -- C ABI of the GB300 MX block-quantization library (libmxq.so).
 *
 * Plain pointers and sizes only.  Every data pointer is a DEVICE pointer that
 * the caller owns (allocated, for example, with torch or cudaMalloc); the
 * library never allocates, never frees and never synchronizes inside these
 * calls.  Work is enqueued on the caller's `stream` (0 = legacy default
 * stream), so every call can be captured in a CUDA graph and ordered with the
 * caller's own work.  Kernels are launched with programmatic dependent launch:
 * one may be scheduled, and run its shared-memory set-up, while the previous
 * kernel on the stream is still running, but it touches no global memory
 * before that kernel has completed, so stream order is kept exactly.
 *
 * Return value: MXQ_OK (0) when the work was enqueued, a negative MXQ_E* code
 * when an argument was rejected (nothing is enqueued and no byte of any output
 * is touched) or when the launch failed.  Argument checks run on the host and
 * make no CUDA call, so a rejected call is safe on any thread and any device.
 * The library never aborts, throws or raises a device trap.
 *
 * Checks that need device data (the group offsets of mxq_quantize_2d_dual) are
 * made by the kernel itself: on failure it writes nothing and sets a bit in
 * the device status word of the current device (mxq_device_status).
 *
 * Sources for the operations (page title, section):
 *   [AO]  pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct
 *         metadata" -- description and review replies.
 *   [MX9] AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
 *         pack/unpack" -- Summary, "Key design choices", review thread.
 */
#ifndef MXQ_H_
#define MXQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t (a repeated identical typedef
   is legal in C11 and C++). */
typedef struct CUstream_st *cudaStream_t;

/* ---- status codes ------------------------------------------------------ */
#define MXQ_OK 0
#define MXQ_EBADSHAPE (-1) /* a size is negative, too large, or violates the method's multiples */
#define MXQ_EBADDTYPE (-2) /* dtype code is not MXQ_F32 / MXQ_BF16 */
#define MXQ_EBADOFFS (-3)  /* group count out of range, or offs/G inconsistent */
#define MXQ_EALIGN (-4)    /* a pointer is not 16-byte aligned (offs: 4-byte) */
#define MXQ_EOVERLAP (-5)  /* two buffers' byte ranges overlap (or one wraps past the top of memory) */
#define MXQ_ECUDA (-6)     /* the CUDA runtime refused the launch */
#define MXQ_ENULL (-7)     /* a required pointer is NULL */
#define MXQ_ESCRATCH (-8)  /* needs more than the static scratch of the no-allocation call */

/* ---- dtype codes ------------------------------------------------------- */
#define MXQ_F32 0
#define MXQ_BF16 1

/* ---- limits ------------------------------------------------------------ */
#define MXQ_MAX_GROUPS 1024 /* largest G accepted by mxq_quantize_2d_dual */

/* ---- device status word bits (see mxq_device_status) ------------------- */
#define MXQ_DEV_BADOFFS 0x1u /* offs failed the device-side check: no output written */
#define MXQ_DEV_TIMEOUT 0x2u /* an internal pipeline wait gave up: outputs incomplete */
#define MXQ_DEV_OOB 0x4u     /* checked build only: a store out of its buffer was skipped */

/*
 * Dual-axis MXFP8 quantization of one bf16 matrix, reading it once.
 * [AO] description: one read of x emits four outputs -- E4M3 data cast in 1x32
 * blocks along N (rowwise) and in 32x1 blocks along M (colwise), and the two
 * E8M0 "rceil" scale tensors already in the blocked layout that block-scaled
 * MMA consumes, with the colwise scales grouped by the K-group offsets and
 * zeroed for the uncovered tail past offs[G-1].
 *
 *   x      bf16 [M, N] row-major (2*M*N bytes), 16-byte aligned.
 *   M, N   multiples of 128, >= 0 (the [AO] description requires both sizes and
 *          every group size to be multiples of 128).  M == 0 or N == 0 is a
 *          no-op.
 *   offs   device int32 [G]: cumulative group ends, non-decreasing, each a
 *          multiple of 128, offs[G-1] <= M (empty groups allowed); 4-byte
 *          aligned.  NULL selects dense placement (one group [0, M)); then G
 *          must be 0.  1 <= G <= MXQ_MAX_GROUPS otherwise.
 *   q_row  E4M3 [M*N]: q_row[m*N + n]; 16-byte aligned.
 *   s_row  E8M0 [M*N/32]: the [M, N/32] scale matrix in the 128x4 blocked
 *          layout: scale (r, c) at ((r/128)*(C/4) + c/4)*512 + (r%32)*16 +
 *          ((r%128)/32)*4 + c%4 with C = N/32.
 *   q_col  E4M3 [N*M]: q_col[n*M + m], i.e. [N, M] row-major ("logically
 *          transposed colwise store").
 *   s_col  E8M0 [N*M/32]: group g = [lo, hi) owns bytes [N*lo/32, N*hi/32),
 *          its [N, (hi-lo)/32] colwise scale matrix in the same blocked
 *          layout; bytes from N*offs[G-1]/32 to the end are written as 0.
 *          Rows in the tail are still quantized in q_row, s_row and q_col.
 *   stream CUDA stream for the launch.
 * Scale and data rules ([AO] description, "Bug-compatible" list): the scale
 * byte is the smallest s with amax <= 448*2^(s-127); data is x*2^(127-s) cast
 * to E4M3 with round-to-nearest-even; a block with any NaN gets scale 255 and
 * all-NaN (0x7F) data on both axes; a block with +-Inf and no NaN gets scale
 * 255 and 0x7F data rowwise, and scale 254 with +-Inf saturated to +-448
 * colwise.
 * Buffers must not overlap one another, x or offs.  Every byte of every output
 * is written (for valid offs); outputs need no initialisation.
 */
int mxq_quantize_2d_dual(const void *x, int64_t M, int64_t N, const int32_t *offs, int32_t G,
                         uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                         cudaStream_t stream);

/*
 * The same cast on a band of rows [row0, row0 + rows) of a full [M, N] tensor,
 * for data-parallel shards along M.  The pages' tiles and blocks are
 * independent, so the band's outputs are exactly the full call's bytes at the
 * band's places; only s_col needs the band's position, because a group's slab
 * offset and width come from the full tensor's offs.
 *
 *   x      bf16 [rows, N]: the band (row0 .. row0+rows-1 of the full tensor).
 *   rows, row0, M, N   multiples of 128 with row0 + rows <= M; rows == 0 is a
 *          no-op.
 *   offs, G  the full tensor's K-group offsets (as for mxq_quantize_2d_dual,
 *          checked on the device against M); NULL and 0 for dense.
 *   q_row  E4M3 [rows*N]: rows row0.. of the full q_row.
 *   s_row  E8M0 [rows*N/32]: bytes [row0*N/32, (row0+rows)*N/32) of the full
 *          s_row (the blocked layout keeps a band of 128-row blocks together).
 *   q_col  E4M3 [N*rows]: [N, rows] row-major, columns row0.. of the full q_col.
 *   s_col  E8M0 [N*M/32]: the FULL colwise scale buffer; the call writes the
 *          512-byte atoms of its rows (and the zero atoms of its tail rows) and
 *          leaves every other byte alone, so bands that cover [0, M) once write
 *          every byte once, with no exchange between them.
 * Errors and device status as for mxq_quantize_2d_dual; MXQ_EBADSHAPE also for
 * a band outside [0, M).
 */
int mxq_quantize_2d_dual_rows(const void *x, int64_t rows, int64_t N, int64_t row0, int64_t M,
                              const int32_t *offs, int32_t G, uint8_t *q_row, uint8_t *s_row,
                              uint8_t *q_col, uint8_t *s_col, cudaStream_t stream);

/*
 * MX9 pack.  [MX9] Summary / "Key design choices": blocks of 16 consecutive
 * elements along the last axis (block b = r*(cols/16) + j); per block a
 * shared exponent E = max over the block of the element exponents taken from
 * the native bits (biased exponent field - 127: fp32 bits 30..23, bf16 bits
 * 14..7), stored as max_exp[b] = E + 127; per pair p of elements (2p, 2p+1) a
 * prime bit (bit p of prime[b], LSB = pair 0) set when the pair's exponent is
 * below E; scale exponent k_p = max(E - 6 - prime_p, -126); data
 * q = clamp(round_half_even(x / 2^k_p), -127, 127).  NaN packs to 0, +-Inf to
 * +-127 (max_exp 255).
 *
 *   x        fp32 or bf16 [rows, cols] row-major, 16-byte aligned.
 *   dtype    MXQ_F32 or MXQ_BF16 (type of x).
 *   rows, cols  rows >= 0, cols >= 0 and cols % 16 == 0.
 *   q        int8 [n_blocks, 16], n_blocks = rows*cols/16; 16-byte aligned.
 *   max_exp  uint8 [n_blocks].
 *   prime    uint8 [n_blocks] (the page's [n_blocks, 1]).
 * Buffers must not overlap.  9 bits per element in total.
 */
int mx9_pack(const void *x, int dtype, int64_t rows, int64_t cols, int8_t *q, uint8_t *max_exp,
             uint8_t *prime, cudaStream_t stream);

/*
 * MX9 unpack: y = q * 2^k_p with k_p rebuilt from max_exp and prime as in
 * mx9_pack ([MX9] Summary: the packed form is dequantized back to fp32/bf16;
 * the caller passes the shape back because it is not stored).  The result is
 * exact in fp32 and bf16; a block with max_exp 255 can give +-Inf.
 *
 *   q, max_exp, prime  as produced by mx9_pack (q 16-byte aligned).
 *   y        fp32 or bf16 [rows, cols] row-major output, 16-byte aligned.
 *   dtype    MXQ_F32 or MXQ_BF16 (type of y).
 */
int mx9_unpack(const int8_t *q, const uint8_t *max_exp, const uint8_t *prime, void *y, int dtype,
               int64_t rows, int64_t cols, cudaStream_t stream);

/*
 * MX9 and MX6 in one packed uint8 tensor ([MX9] commits: MX9 packed into one
 * uint8 tensor with MX6 and MX9 sent to the packed kernels, and strided inputs
 * accepted; the suite's axis, non-contiguous and padding tests).  One record per 16-element block, [exponent byte, prime
 * byte, data] (the review excerpt stores the exponent at the record start):
 *   MXQ_FMT_MX9: data = 16 int8 q as in mx9_pack; 18-byte records, 9 bits/elem.
 *   MXQ_FMT_MX6: the same rule with 4 magnitude bits, k = max(E - 3 - prime,
 *     -126), q clamped to [-15, 15], stored as sixteen 5-bit two's-complement
 *     codes (element i at bits 5i..5i+4 of the 10 data bytes read as one
 *     little-endian number); 12-byte records, 6 bits/elem.
 * The 2-D tensor has `rows` x `cols` elements, element (r, c) at x[r*ld + c]
 * (ld >= cols, any element-aligned x: strided views are accepted).  Blocks
 * run along `axis`: 1 = along each row, block b = r*ceil(cols/16) + j over
 * columns 16j..16j+15; 0 = down each column, b = c*ceil(rows/16) + j over rows
 * 16j..16j+15 (the tensor with the blocked axis moved last).  A partial last
 * block is zero-padded and then follows the normal rule; unpack writes only
 * the tensor's own elements.  packed: n_blocks * record bytes, 2-byte (MX9) or
 * 4-byte (MX6) aligned.  Any allowed alignment gives the same bytes; 16-byte
 * aligned packed, x and row pitch (ld * element size) select the faster
 * kernels.  Shape and axis are not stored: the caller passes them back to
 * unpack.  Errors: MXQ_EBADDTYPE (dtype or fmt), MXQ_EBADSHAPE (negative
 * sizes, ld < cols, axis not 0/1), MXQ_ENULL, MXQ_EALIGN (x not element-
 * aligned, packed below the sizes above), MXQ_EOVERLAP, MXQ_ECUDA.
 */
#define MXQ_FMT_MX9 9
#define MXQ_FMT_MX6 6
#define MXQ_MX9_RECORD_BYTES 18
#define MXQ_MX6_RECORD_BYTES 12
int mx_pack_packed(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld, int axis,
                   int fmt, uint8_t *packed, cudaStream_t stream);
int mx_unpack_packed(const uint8_t *packed, int fmt, void *y, int dtype, int64_t rows,
                     int64_t cols, int64_t ld, int axis, cudaStream_t stream);

/*
 * The three-pass composition that the fused cast replaces ([AO] description,
 * first paragraph: a 1x32 cast along N, a 32x1 cast along M and a standalone
 * K-groups swizzle of the colwise scales, reading x twice).  Kept so that the
 * fused kernel can be measured against it and for callers that want one axis.
 *
 * mxq_quantize_1x32: q_row and s_row exactly as mxq_quantize_2d_dual writes
 *   them.  Arguments as there.
 * mxq_quantize_32x1: q_col as mxq_quantize_2d_dual writes it, and the colwise
 *   scales as a plain row-major [N, M/32] matrix s_rm (byte n*(M/32) + i for
 *   the 32x1 block of rows 32i..32i+31 of column n).  Its block rule is the
 *   separate 32x1 cast's ([AO] description, NaN paragraph): the amax skips NaN
 *   (an all-NaN block takes scale 0), +-Inf gives scale 254 and +-448 data,
 *   a NaN element stays a NaN byte.  So it differs from the fused cast only in
 *   blocks that hold NaN.
 * mxq_swizzle_kgroups: s_rm [N, M/32] -> s_col in the fused cast's layout:
 *   per-group blocked slabs, zeros from N*offs[G-1]/32 on (offs/G as for
 *   mxq_quantize_2d_dual; invalid offs are detected on the device, nothing is
 *   written and MXQ_DEV_BADOFFS is set).
 * mxq_quantize_2d_dual_3pass: the three launches in order on `stream`, with
 *   the caller's `workspace` (>= N*M/32 bytes, 16-byte aligned, not
 *   overlapping any other buffer; returns MXQ_EBADSHAPE if too small) holding
 *   s_rm between the second and third.
 * All pointers are device pointers; 16-byte alignment as for the fused cast.
 */
int mxq_quantize_1x32(const void *x, int64_t M, int64_t N, uint8_t *q_row, uint8_t *s_row,
                      cudaStream_t stream);
int mxq_quantize_32x1(const void *x, int64_t M, int64_t N, uint8_t *q_col, uint8_t *s_rm,
                      cudaStream_t stream);
int mxq_swizzle_kgroups(const uint8_t *s_rm, int64_t N, int64_t M, const int32_t *offs, int32_t G,
                        uint8_t *s_col, cudaStream_t stream);
int mxq_quantize_2d_dual_3pass(const void *x, int64_t M, int64_t N, const int32_t *offs, int32_t G,
                               uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                               uint8_t *workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * mxq_quantize_2d_dual_3pass without any allocation.  The pages have no
 * counterpart: this is a library convenience.  It is for callers that cannot
 * allocate device memory when they need the cast -- work recorded into a CUDA
 * graph in global capture mode (allocation is illegal there), latency-critical
 * paths where cudaMalloc/cudaFree can synchronize the device, and plugins inside
 * a framework that owns all device memory through an allocator they cannot
 * reach.  The three passes' workspace is a static device array of
 * MXQ_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library holds until the process exits; the call makes no cudaMalloc or
 * cudaFree and calls no allocating routine.
 *   Arguments, outputs and errors as mxq_quantize_2d_dual_3pass minus the
 *   workspace; returns MXQ_ESCRATCH, enqueuing nothing, when M*N/32 exceeds
 *   MXQ_NOALLOC_SCRATCH_BYTES (16 MiB: M*N up to 2^29 elements).
 *   The first call on a device looks up the array's device address with that
 *   device current; make that first call before any stream capture.  The
 *   address is looked up again when the current context changes (after a
 *   device reset, say), so the first call in a new context also belongs
 *   before any capture.
 *   All calls share the one array and each overwrites the part it uses before
 *   reading it: calls that may overlap on the GPU (different streams without
 *   ordering between them) race on it and must be serialized by the caller.
 */
#define MXQ_NOALLOC_SCRATCH_BYTES (16u << 20)
int mxq_quantize_2d_dual_3pass_noalloc(const void *x, int64_t M, int64_t N, const int32_t *offs,
                                       int32_t G, uint8_t *q_row, uint8_t *s_row, uint8_t *q_col,
                                       uint8_t *s_col, cudaStream_t stream);

/*
 * Block-scaled MXFP8 matrix product on the tensor cores, reading E4M3 rows and
 * E8M0 scale matrices exactly as mxq_quantize_2d_dual stores them: the consumer
 * check of the layouts ([AO] description, first paragraph: the scales are
 * written in the blocked form the block-scaled MMA reads; "Uncovered tail"
 * paragraph: one slab per K-group).  tcgen05.mma of kind mxf8f6f4 with one
 * E8M0 scale per 32 K elements; a checking tool, not a tuned GEMM (one CTA per
 * 128x128 output tile, no overlap of loads and MMAs).
 *   D[i, j] = sum_k A(i, k) * 2^(sa(i, k/32) - 127) * B(j, k) * 2^(sb(j, k/32) - 127)
 *   a      E4M3 [Ma, K], row i at a + i*lda (K contiguous bytes); e.g. q_row
 *          (lda = N), or a K-group's columns of q_col (a = q_col + lo, lda = M).
 *   sa     E8M0 [Ma, K/32] in the 128x4 blocked layout (s_row, or the group's
 *          s_col slab at s_col + N*lo/32).
 *   b, ldb, sb   likewise for B [Nb, K].
 *   d      fp32 [Ma, Nb] row-major.
 *   Ma, Nb, K    multiples of 128, at most 2^24 (Ma == 0 or Nb == 0: no-op;
 *          K == 0 with Ma, Nb > 0: MXQ_EBADSHAPE); lda, ldb >= K, multiples of 16
 *          and at most 2^40; every pointer 16-byte aligned; d must not overlap an
 *          input.
 * Every internal wait is bounded (MXQ_DEV_TIMEOUT in the status word).
 */
int mxq_mxfp8_scaled_mm(const uint8_t *a, int64_t lda, const uint8_t *sa, const uint8_t *b,
                        int64_t ldb, const uint8_t *sb, float *d, int64_t Ma, int64_t Nb, int64_t K,
                        cudaStream_t stream);

/*
 * Device status word of the current device: a sticky OR of MXQ_DEV_* bits set
 * by kernels since the last clear.  Writes it to *out and clears it when
 * `clear` is non-zero.  This call synchronizes the device (it reads device
 * memory); use it for diagnostics and tests, not inside captured work.
 * Returns MXQ_OK, MXQ_ENULL or MXQ_ECUDA.
 * mxq_last_device_status is the same call under the boundary's other name: the
 * word lives in device memory and is read by a copy (hence the synchronization)
 * instead of in a library-owned pinned host flag, so that no compute call
 * needs an allocation.
 */
int mxq_device_status(uint32_t *out, int clear);
int mxq_last_device_status(uint32_t *out, int clear);

/*
 * Self-test of failure detection, on the GPU and without a fault: launches one
 * warp that waits, with the same bounded wait the pipelines use, on an
 * mbarrier nothing ever completes.  The wait gives up after `limit_ns`
 * nanoseconds (1e6 .. 4e9, else MXQ_EBADSHAPE), the kernel records
 * MXQ_DEV_TIMEOUT in the device status word and returns, and the context stays
 * usable.  The production kernels use a 4 s limit per wait.
 */
int mxq_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/*
 * Checked builds.  A library compiled with MXQ_DEBUG_BOUNDS=1 (the
 * package's build step makes it as libmxq_checked.so beside libmxq.so)
 * tests the byte range of every global store its kernels make outside the
 * TMA tensor stores (whose bounds the tensor maps enforce) against the
 * output buffer it belongs to; a range that would leave the buffer is not
 * written and MXQ_DEV_OOB is set in the device status word.  Results are
 * otherwise identical.  mxq_debug_bounds() returns 1 in a checked build and
 * 0 in a release build.  mxq_selftest_bounds() launches one thread that
 * tests a range lying past a 64-byte dummy buffer, without any access: a
 * checked build records MXQ_DEV_OOB, a release build records nothing.
 * Returns MXQ_OK or MXQ_ECUDA.
 */
int mxq_debug_bounds(void);
int mxq_selftest_bounds(cudaStream_t stream);

/* Static description of a status code (never NULL). */
const char *mxq_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
int mxq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H_ */
