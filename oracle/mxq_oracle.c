/*
 * mxq_oracle.c -- CPU oracle for MX block quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, scalar, obviously-correct
 * statement of what the GPU library computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg load it.  It shares no source, header,
 * table or helper with the CUDA library; the two agree only because both follow
 * the same published definitions.
 *
 * Arithmetic is carried out in IEEE binary64, where every value that occurs here
 * (bf16/fp32 inputs, their products with powers of two, E4M3 grid points) is
 * exact.  Rounding is done by nearbyint() in the default round-to-nearest-even
 * mode; ldexp()/frexp() are exact.
 *
 * Sources (cited by page title and section):
 *   [AO]  pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct
 *         metadata" -- description and review replies.
 *   [MX9] AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
 *         pack/unpack" -- Summary, "Key design choices", review thread.
 *
 * Readings where the pages are silent are marked READING and listed in the
 * design notes of the repository.
 *
 * Parity unpinned (the pages print none of these, so no pin outside this file
 * can fix them; the GPU library follows the same readings):
 *   - the bit order of the MX9 / MX6 prime byte (bit p = pair p, LSB first);
 *   - the sign of the E4M3 NaN data byte (0x7F);
 *   - the MX6 code layout (sixteen 5-bit two's-complement codes, element i at
 *     bits 5i..5i+4 of the 10 data bytes read little-endian).
 * Every other result here has at least one pin outside this file.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Status codes (values match the library's documented codes; no shared header). */
#define ORC_OK 0
#define ORC_EBADSHAPE (-1)
#define ORC_EBADDTYPE (-2)
#define ORC_EBADOFFS (-3)

#define ORC_F32 0
#define ORC_BF16 1

/* ------------------------------------------------------------------------- */
/* Input decoding                                                            */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double f32_to_double(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* E4M3 (OCP FP8 "e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3       */
/* mantissa bits, no infinities, NaN = S.1111.111, largest finite 448.       */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code, from the format definition. */
double oracle_e4m3_value(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);             /* subnormal: m/8 * 2^-6 */
    else
        mag = ldexp(8.0 + (double)m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/*
 * Encode v to E4M3 with round-to-nearest, ties to the even mantissa, and
 * saturation of finite overflow and of +-Inf to +-448 (the "satfinite" cast
 * named in [AO] description, second paragraph).  NaN encodes as 0x7F.  The
 * sign bit always follows v, so -0 and negative values that round to zero give
 * 0x80 (READING: the pages do not print signed-zero bytes; IEEE casts keep the
 * sign).
 */
uint8_t oracle_e4m3_encode(double v) {
    uint8_t sign;
    double a;
    int code;
    if (isnan(v)) return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs(v);
    if (a > 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9; a count of 8 steps is the smallest
           normal 2^-6, whose code is also 8 */
        code = (int)nearbyint(ldexp(a, 9));
    } else {
        int e2;
        double n;
        (void)frexp(a, &e2);      /* a = f * 2^e2, f in [0.5, 1) */
        int E = e2 - 1;           /* a in [2^E, 2^(E+1)), E in [-6, 8] */
        n = nearbyint(ldexp(a, 3 - E)); /* significand in steps of 1/8: 8..16 */
        /* n == 16 carries into the next binade; the formula stays correct */
        code = (E + 7) * 8 + ((int)n - 8);
    }
    if (code > 0x7E) code = 0x7E; /* unreachable for a <= 448; kept explicit */
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------- */
/* E8M0 rceil scale (the [AO] description supports the rceil rounding mode   */
/* alone; review reply on the scale 0/1 cutoff 448*2^-127).                   */
/* ------------------------------------------------------------------------- */

/*
 * Smallest s in [0, 254] such that amax <= 448 * 2^(s-127): the block's
 * largest magnitude, divided by the scale 2^(s-127), fits the E4M3 range
 * without saturating.  amax must be finite and non-negative.
 */
int oracle_e8m0_rceil(double amax) {
    int lo = 0, hi = 254;
    while (lo < hi) { /* the predicate is monotone in s: binary search */
        int mid = (lo + hi) / 2;
        if (amax <= ldexp(448.0, mid - 127))
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

/*
 * One MXFP8 block of 32 bf16 elements read with a stride (1 for a 1x32 row
 * block, N for a 32x1 column block).  Writes the E8M0 scale byte and the 32
 * E4M3 data bytes (with a stride for the output).
 *
 * Non-finite rules, [AO] description, "Bug-compatible" list and the NaN
 * paragraph after it:
 *   - any NaN in the block: scale 255 and every data byte NaN, on both axes
 *     (the fused kernel's deliberate choice: NaN poisons the colwise block too);
 *   - otherwise any +-Inf: rowwise (non-saturating cast) gives scale 255 and
 *     all-NaN data; colwise (saturating cast) gives scale 254 and finite data,
 *     i.e. Inf saturates to +-448 after the 2^-127 multiplier.
 *   - a finite block whose amax is small enough to reach scale byte 0 is
 *     multiplied by 2^127 (the "254 - scale_biased" reciprocal).
 * Data for scale s < 255 is x * 2^(127-s), encoded by oracle_e4m3_encode.
 * READING: a NaN data byte is always 0x7F (the pages leave NaN signs to a
 * contract they do not print).
 */
void oracle_mxfp8_block(const uint16_t *x, int64_t stride, int colwise,
                        uint8_t *scale_out, uint8_t *q, int64_t qstride) {
    int any_nan = 0, any_inf = 0, s, i;
    double amax = 0.0;
    for (i = 0; i < 32; ++i) {
        double v = bf16_to_double(x[i * stride]);
        if (isnan(v))
            any_nan = 1;
        else if (isinf(v))
            any_inf = 1;
        else if (fabs(v) > amax)
            amax = fabs(v);
    }
    if (any_nan)
        s = 255;
    else if (any_inf)
        s = colwise ? 254 : 255;
    else
        s = oracle_e8m0_rceil(amax);
    *scale_out = (uint8_t)s;
    for (i = 0; i < 32; ++i) {
        if (s == 255) {
            q[i * qstride] = 0x7F;
        } else {
            double v = bf16_to_double(x[i * stride]);
            q[i * qstride] = oracle_e4m3_encode(ldexp(v, 127 - s));
        }
    }
}

/*
 * The colwise block of the separate 32x1 cast that the fused kernel replaces
 * ([AO] description, NaN paragraph): its amax skips NaN entirely, so a block
 * holding NaN still gets the scale its other elements imply (0 when every
 * element is NaN: the maximum over no values is taken as 0, READING); the
 * cast saturates, so +-Inf gives scale 254 and +-448 data, and a NaN element
 * stays a NaN byte (0x7F).
 */
void oracle_mxfp8_block_nan_dropped(const uint16_t *x, int64_t stride, uint8_t *scale_out,
                                    uint8_t *q, int64_t qstride) {
    int any_inf = 0, s, i;
    double amax = 0.0;
    for (i = 0; i < 32; ++i) {
        double v = bf16_to_double(x[i * stride]);
        if (isnan(v)) continue;
        if (isinf(v))
            any_inf = 1;
        else if (fabs(v) > amax)
            amax = fabs(v);
    }
    s = any_inf ? 254 : oracle_e8m0_rceil(amax);
    *scale_out = (uint8_t)s;
    for (i = 0; i < 32; ++i) {
        double v = bf16_to_double(x[i * stride]);
        q[i * qstride] = isnan(v) ? 0x7F : oracle_e4m3_encode(ldexp(v, 127 - s));
    }
}

/* ------------------------------------------------------------------------- */
/* Blocked scale layout                                                       */
/* ------------------------------------------------------------------------- */

/*
 * Byte offset of scale (r, c) of an R x C scale matrix stored in the blocked
 * layout consumed by block-scaled MMA: 128 x 4 atoms of 512 bytes ([AO]
 * description: scales are written "in the blocked layouts their consumers
 * expect"; one atom is the "512-byte line" of the uncovered-tail paragraph),
 * atoms ordered row-block-major, and inside an atom row r sits at
 * (r % 32) * 16 + ((r % 128) / 32) * 4 and column c at c % 4.
 * READING: the formula itself is not printed on the pages; this is the public
 * 128x4 scale-factor layout of block-scaled tensor-core MMA.
 * Requires R % 128 == 0 and C % 4 == 0.
 */
int64_t oracle_blocked_index(int64_t r, int64_t c, int64_t R, int64_t C) {
    (void)R;
    return ((r / 128) * (C / 4) + c / 4) * 512 + (r % 32) * 16 +
           ((r % 128) / 32) * 4 + (c % 4);
}

/* ------------------------------------------------------------------------- */
/* Dual-axis MXFP8 quantization ([AO] description)                            */
/* ------------------------------------------------------------------------- */

/*
 * Validation of the group offsets (the [AO] description requires each group
 * size to be a multiple of 128; review replies: offsets are checked for
 * ordering and bounds; empty groups are valid).  offs == NULL selects dense placement and
 * then G must be 0.
 */
int oracle_check_offs(const int32_t *offs, int32_t G, int64_t M) {
    int32_t g;
    int64_t prev = 0;
    if (offs == NULL) return G == 0 ? ORC_OK : ORC_EBADOFFS;
    if (G < 1) return ORC_EBADOFFS;
    for (g = 0; g < G; ++g) {
        int64_t o = offs[g];
        if (o < prev || o % 128 != 0 || o > M) return ORC_EBADOFFS;
        prev = o;
    }
    return ORC_OK;
}

/*
 * x: bf16 bit patterns, [M, N] row-major.  Outputs (all written in full):
 *   q_row [M*N]      E4M3, q_row[m*N + n]            (1x32 blocks along N)
 *   s_row [M*N/32]   E8M0, blocked as an [M, N/32] scale matrix
 *   q_col [N*M]      E4M3, q_col[n*M + m]            (32x1 blocks along M,
 *                    stored transposed, as the [AO] description's
 *                    colwise store is)
 *   s_col [N*M/32]   E8M0 colwise scales grouped by offs:
 *       group g covers rows [lo, hi) = [offs[g-1] (0 for g = 0), offs[g]);
 *       its scales form an [N, (hi-lo)/32] matrix, blocked, stored as one
 *       contiguous slab starting at byte N*lo/32 (READING of the [AO]
 *       description's per-group slabs and compact column scales);
 *       every byte from N*offs[G-1]/32 to the end is 0 ([AO] description,
 *       "Uncovered tail": rows past offs[-1] are still quantized, their column
 *       scale bytes are zeroed).
 * Dense (offs == NULL) is the single group [0, M).
 */
int oracle_mxfp8_dual(const uint16_t *x, int64_t M, int64_t N,
                      const int32_t *offs, int32_t G, uint8_t *q_row,
                      uint8_t *s_row, uint8_t *q_col, uint8_t *s_col) {
    int64_t m, n, j, i, b;
    int rc;
    if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0) return ORC_EBADSHAPE;
    rc = oracle_check_offs(offs, G, M);
    if (rc != ORC_OK) return rc;

    /* rowwise: block (m, j) = x[m, 32j .. 32j+31] */
    for (m = 0; m < M; ++m) {
        for (j = 0; j < N / 32; ++j) {
            uint8_t s;
            oracle_mxfp8_block(x + m * N + 32 * j, 1, 0, &s,
                               q_row + m * N + 32 * j, 1);
            s_row[oracle_blocked_index(m, j, M, N / 32)] = s;
        }
    }

    /* colwise: block (i, n) = x[32i .. 32i+31, n] */
    {
        int64_t end = offs ? offs[G - 1] : M;
        for (i = 0; i < M / 32; ++i) {
            int64_t row = 32 * i, lo = 0, hi = M;
            int in_group = row < end;
            if (offs && in_group) {
                /* the group holding this row block: offs[g-1] <= row < offs[g] */
                int32_t g = 0;
                while (offs[g] <= row) ++g;
                lo = g == 0 ? 0 : offs[g - 1];
                hi = offs[g];
            }
            for (n = 0; n < N; ++n) {
                uint8_t s;
                oracle_mxfp8_block(x + row * N + n, N, 1, &s,
                                   q_col + n * M + row, 1);
                if (in_group)
                    s_col[N * lo / 32 +
                          oracle_blocked_index(n, i - lo / 32, N, (hi - lo) / 32)] = s;
            }
        }
        for (b = N * end / 32; b < N * M / 32; ++b) s_col[b] = 0;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* The three-pass composition ([AO] description, first paragraph): a 1x32     */
/* cast, a 32x1 cast with plain row-major scales, and a K-groups swizzle of   */
/* those scales into the blocked per-group slabs.                             */
/* ------------------------------------------------------------------------- */

/* 1x32 pass: q_row and s_row exactly as in oracle_mxfp8_dual. */
int oracle_mxfp8_1x32(const uint16_t *x, int64_t M, int64_t N, uint8_t *q_row, uint8_t *s_row) {
    int64_t m, j;
    if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0) return ORC_EBADSHAPE;
    for (m = 0; m < M; ++m)
        for (j = 0; j < N / 32; ++j) {
            uint8_t s;
            oracle_mxfp8_block(x + m * N + 32 * j, 1, 0, &s, q_row + m * N + 32 * j, 1);
            s_row[oracle_blocked_index(m, j, M, N / 32)] = s;
        }
    return ORC_OK;
}

/* 32x1 pass: q_col[n*M + m] and the scales as a plain [N, M/32] row-major
   matrix s_rm[n*(M/32) + i], with the NaN-dropping block rule above. */
int oracle_mxfp8_32x1(const uint16_t *x, int64_t M, int64_t N, uint8_t *q_col, uint8_t *s_rm) {
    int64_t i, n;
    if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0) return ORC_EBADSHAPE;
    for (i = 0; i < M / 32; ++i)
        for (n = 0; n < N; ++n)
            oracle_mxfp8_block_nan_dropped(x + 32 * i * N + n, N, &s_rm[n * (M / 32) + i],
                                           q_col + n * M + 32 * i, 1);
    return ORC_OK;
}

/* K-groups swizzle: s_rm [N, M/32] row-major -> s_col with group g's columns
   [lo/32, hi/32) blocked as one slab at byte N*lo/32, and zeros from
   N*offs[G-1]/32 on (the separate pass "iterates groups and returns
   new_zeros", [AO] "Uncovered tail" paragraph).  offs == NULL: one group. */
int oracle_swizzle_kgroups(const uint8_t *s_rm, int64_t N, int64_t M, const int32_t *offs,
                           int32_t G, uint8_t *s_col) {
    int64_t b, n, c, lo = 0;
    int32_t g, ng = offs ? G : 1;
    int rc;
    if (M < 0 || N < 0 || M % 128 != 0 || N % 128 != 0) return ORC_EBADSHAPE;
    rc = oracle_check_offs(offs, G, M);
    if (rc != ORC_OK) return rc;
    for (b = 0; b < N * M / 32; ++b) s_col[b] = 0;
    for (g = 0; g < ng; ++g) {
        int64_t hi = offs ? offs[g] : M;
        for (n = 0; n < N; ++n)
            for (c = lo / 32; c < hi / 32; ++c)
                s_col[N * lo / 32 + oracle_blocked_index(n, c - lo / 32, N, (hi - lo) / 32)] =
                    s_rm[n * (M / 32) + c];
        lo = hi;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* MX9 ([MX9] Summary and "Key design choices")                               */
/* ------------------------------------------------------------------------- */

/*
 * Element exponent taken from the native bits ([MX9] "Key design choices":
 * the exponent comes from the input type's own bit fields): the biased
 * exponent field minus 127, so zero and
 * subnormals give -127 and Inf/NaN give 128.
 */
static int mx9_t(const void *x, int dtype, int64_t idx) {
    if (dtype == ORC_F32) {
        uint32_t u = ((const uint32_t *)x)[idx];
        return (int)((u >> 23) & 0xFF) - 127;
    } else {
        uint16_t u = ((const uint16_t *)x)[idx];
        return (int)((u >> 7) & 0xFF) - 127;
    }
}

static double mx9_value(const void *x, int dtype, int64_t idx) {
    if (dtype == ORC_F32) return f32_to_double(((const uint32_t *)x)[idx]);
    return bf16_to_double(((const uint16_t *)x)[idx]);
}

/*
 * Scale exponent of pair p: the shared exponent E less 6 (8-bit signed
 * elements with 7 magnitude bits cover |x| < 2^(E+1)), less one more for a
 * pair flagged in the prime bitmap, clamped below at -126, the smallest fp32
 * normal exponent ([MX9] "Key design choices").
 * READING: the offset 6 and the prime polarity are fixed by nine bits per element
 * (8-bit value, 1/2 bit shared exponent, 1/2 bit prime) and by the quality the
 * page reports; the page does not print them.
 */
static int mx9_k(int E, int tau) {
    int k = E - 6 - tau;
    return k < -126 ? -126 : k;
}

/*
 * Pack rows x cols elements (cols % 16 == 0) in blocks of 16 consecutive
 * elements along the last axis; block b = r * (cols/16) + j.
 *   max_exp[b] = E + 127 where E = max_i t(x_i)           (E8M0 shared exponent)
 *   prime[b]   bit p (LSB = pair 0) = 1 iff max(t_2p, t_2p+1) < E
 *   q[16b + i] = clamp(round_half_even(x_i / 2^k_p), -127, 127)
 * The division is by a power of two, hence exact ([MX9] review: IEEE
 * round-nearest division), and the rounding is ties-to-even.  The clamp is
 * symmetric at +-127 ([MX9] "Key design choices").
 * READING for non-finite inputs (the page only says NaN produces garbage):
 * NaN packs to q = 0; +-Inf to +-127; the block's max_exp is 255.
 */
int oracle_mx9_pack(const void *x, int dtype, int64_t rows, int64_t cols,
                    int8_t *q, uint8_t *max_exp, uint8_t *prime) {
    int64_t nb, b;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EBADDTYPE;
    if (rows < 0 || cols < 0 || cols % 16 != 0) return ORC_EBADSHAPE;
    nb = rows * (cols / 16);
    for (b = 0; b < nb; ++b) {
        int t[16], E = -127, p, i;
        uint8_t bits = 0;
        for (i = 0; i < 16; ++i) {
            t[i] = mx9_t(x, dtype, 16 * b + i);
            if (t[i] > E) E = t[i];
        }
        max_exp[b] = (uint8_t)(E + 127);
        for (p = 0; p < 8; ++p) {
            int tp = t[2 * p] > t[2 * p + 1] ? t[2 * p] : t[2 * p + 1];
            int tau = tp < E;
            int k = mx9_k(E, tau);
            bits |= (uint8_t)(tau << p);
            for (i = 2 * p; i < 2 * p + 2; ++i) {
                double v = mx9_value(x, dtype, 16 * b + i);
                double r;
                if (isnan(v)) {
                    q[16 * b + i] = 0;
                    continue;
                }
                r = nearbyint(ldexp(v, -k));
                if (r > 127.0) r = 127.0;
                if (r < -127.0) r = -127.0;
                q[16 * b + i] = (int8_t)r;
            }
        }
        prime[b] = bits;
    }
    return ORC_OK;
}

/* Round a binary64 value to bf16 bits, nearest-even (used only where the
   value is already exact in bf16, or overflows). */
static uint16_t double_to_bf16_bits(double y) {
    float f = (float)y;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return 0x7FC0;
    {
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
    }
    return (uint16_t)(u >> 16);
}

/*
 * Unpack: y_i = q_i * 2^k_p with k_p rebuilt from max_exp and the prime bit,
 * as in pack.  The product is exact in fp32 and bf16 (7-bit magnitudes,
 * exponents >= -126); a block with max_exp 255 can overflow to +-Inf.
 */
int oracle_mx9_unpack(const int8_t *q, const uint8_t *max_exp,
                      const uint8_t *prime, void *y, int dtype, int64_t rows,
                      int64_t cols) {
    int64_t nb, b;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EBADDTYPE;
    if (rows < 0 || cols < 0 || cols % 16 != 0) return ORC_EBADSHAPE;
    nb = rows * (cols / 16);
    for (b = 0; b < nb; ++b) {
        int E = (int)max_exp[b] - 127, i;
        for (i = 0; i < 16; ++i) {
            int tau = (prime[b] >> (i / 2)) & 1;
            double v = ldexp((double)q[16 * b + i], mx9_k(E, tau));
            if (fabs(v) >= ldexp(1.0, 128)) v = v > 0 ? INFINITY : -INFINITY;
            if (dtype == ORC_F32) {
                float f = (float)v;
                memcpy((uint32_t *)y + 16 * b + i, &f, sizeof f);
            } else {
                ((uint16_t *)y)[16 * b + i] = double_to_bf16_bits(v);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* MX9 and MX6 in the single packed tensor, blocked along either axis of a    */
/* strided 2-D tensor, with a zero-padded partial last block ([MX9] commits: */
/* MX9 packed into one uint8 tensor with MX6 and MX9 sent to the packed       */
/* kernels, strided inputs accepted; the axis and padding tests of the suite; */
/* the exponent byte is stored at the block record's start).                  */
/*                                                                             */
/* READINGS: a record is [exponent byte, prime byte, data]; MX9 data is the    */
/* 16 int8 q; MX6 uses the same rule with 4 magnitude bits (offset 3 instead   */
/* of 6, clamp +-15) and stores sixteen 5-bit two's-complement codes, element  */
/* i at bits 5i..5i+4 of the 10 data bytes read as one little-endian number.   */
/* Blocks run along `axis` (1: along a row, 0: down a column); the element    */
/* (r, c) is at x[r * ld + c].  Block order: axis 1 -> b = r * ceil(cols/16) + */
/* j; axis 0 -> b = c * ceil(rows/16) + j, i.e. blocks of the tensor with the  */
/* blocked axis moved last.  A partial last block is padded with zeros and     */
/* then follows the normal rule; unpack writes only real elements.             */
/* ------------------------------------------------------------------------- */

#define ORC_FMT_MX9 9
#define ORC_FMT_MX6 6

static int mx_record_bytes(int fmt) { return fmt == ORC_FMT_MX9 ? 18 : 12; }

/* the block rule of oracle_mx9_pack with a format-dependent offset and clamp */
static void mx_block(const double *v, const int *t, int fmt, uint8_t *e_out, uint8_t *p_out,
                     int *q) {
    int E = -127, p, i, d = fmt == ORC_FMT_MX9 ? 6 : 3, qmax = fmt == ORC_FMT_MX9 ? 127 : 15;
    uint8_t bits = 0;
    for (i = 0; i < 16; ++i)
        if (t[i] > E) E = t[i];
    *e_out = (uint8_t)(E + 127);
    for (p = 0; p < 8; ++p) {
        int tp = t[2 * p] > t[2 * p + 1] ? t[2 * p] : t[2 * p + 1];
        int tau = tp < E;
        int k = E - d - tau;
        if (k < -126) k = -126;
        bits |= (uint8_t)(tau << p);
        for (i = 2 * p; i < 2 * p + 2; ++i) {
            double r;
            if (isnan(v[i])) {
                q[i] = 0;
                continue;
            }
            r = nearbyint(ldexp(v[i], -k));
            if (r > qmax) r = qmax;
            if (r < -qmax) r = -qmax;
            q[i] = (int)r;
        }
    }
    *p_out = bits;
}

static int64_t mx_blocks_per_line(int64_t len) { return (len + 15) / 16; }

int oracle_mx_pack(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld, int axis,
                   int fmt, uint8_t *packed) {
    int64_t lines, line_len, nbl, b;
    int RB = mx_record_bytes(fmt);
    if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EBADDTYPE;
    if (fmt != ORC_FMT_MX9 && fmt != ORC_FMT_MX6) return ORC_EBADDTYPE;
    if (rows < 0 || cols < 0 || ld < cols || (axis != 0 && axis != 1)) return ORC_EBADSHAPE;
    lines = axis == 1 ? rows : cols;
    line_len = axis == 1 ? cols : rows;
    nbl = mx_blocks_per_line(line_len);
    for (b = 0; b < lines * nbl; ++b) {
        int64_t line = b / nbl, j = b % nbl;
        double v[16];
        int t[16], q[16], i;
        uint8_t *rec = packed + b * RB;
        for (i = 0; i < 16; ++i) {
            int64_t pos = 16 * j + i;
            if (pos >= line_len) { /* zero padding */
                v[i] = 0.0;
                t[i] = -127;
            } else {
                int64_t idx = axis == 1 ? line * ld + pos : pos * ld + line;
                v[i] = mx9_value(x, dtype, idx);
                t[i] = mx9_t(x, dtype, idx);
            }
        }
        mx_block(v, t, fmt, &rec[0], &rec[1], q);
        if (fmt == ORC_FMT_MX9) {
            for (i = 0; i < 16; ++i) rec[2 + i] = (uint8_t)(int8_t)q[i];
        } else {
            for (i = 0; i < 10; ++i) rec[2 + i] = 0;
            for (i = 0; i < 16; ++i) {
                unsigned code = (unsigned)q[i] & 0x1Fu; /* 5-bit two's complement */
                int bit;
                for (bit = 0; bit < 5; ++bit)
                    if (code & (1u << bit)) {
                        int pos = 5 * i + bit;
                        rec[2 + pos / 8] |= (uint8_t)(1u << (pos % 8));
                    }
            }
        }
    }
    return ORC_OK;
}

int oracle_mx_unpack(const uint8_t *packed, int fmt, void *y, int dtype, int64_t rows,
                     int64_t cols, int64_t ld, int axis) {
    int64_t lines, line_len, nbl, b;
    int RB = mx_record_bytes(fmt), d = fmt == ORC_FMT_MX9 ? 6 : 3;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EBADDTYPE;
    if (fmt != ORC_FMT_MX9 && fmt != ORC_FMT_MX6) return ORC_EBADDTYPE;
    if (rows < 0 || cols < 0 || ld < cols || (axis != 0 && axis != 1)) return ORC_EBADSHAPE;
    lines = axis == 1 ? rows : cols;
    line_len = axis == 1 ? cols : rows;
    nbl = mx_blocks_per_line(line_len);
    for (b = 0; b < lines * nbl; ++b) {
        int64_t line = b / nbl, j = b % nbl;
        const uint8_t *rec = packed + b * RB;
        int E = (int)rec[0] - 127, i;
        for (i = 0; i < 16; ++i) {
            int64_t pos = 16 * j + i, idx;
            int tau = (rec[1] >> (i / 2)) & 1, q, k;
            double v;
            if (pos >= line_len) continue;
            if (fmt == ORC_FMT_MX9) {
                q = (int8_t)rec[2 + i];
            } else {
                unsigned code = 0;
                int bit;
                for (bit = 0; bit < 5; ++bit) {
                    int p = 5 * i + bit;
                    code |= (unsigned)((rec[2 + p / 8] >> (p % 8)) & 1u) << bit;
                }
                q = code >= 16 ? (int)code - 32 : (int)code;
            }
            k = E - d - tau;
            if (k < -126) k = -126;
            v = ldexp((double)q, k);
            if (fabs(v) >= ldexp(1.0, 128)) v = v > 0 ? INFINITY : -INFINITY;
            idx = axis == 1 ? line * ld + pos : pos * ld + line;
            if (dtype == ORC_F32) {
                float f = (float)v;
                memcpy((uint32_t *)y + idx, &f, sizeof f);
            } else {
                ((uint16_t *)y)[idx] = double_to_bf16_bits(v);
            }
        }
    }
    return ORC_OK;
}

/* Rounding-mode guard: the oracle relies on round-to-nearest-even. */
int oracle_rounding_is_nearest_even(void) { return fegetround() == FE_TONEAREST; }
