/*
 * Serial CPU oracle for device-wide prefix scan, stream compaction and the
 * radix-sort one-bit split.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or constant with the
 * CUDA library; it is written directly from the definitions on the pages:
 *
 *   [P1] geek-doc.cn, "并行前缀和 scan: Hillis-Steele、Blelloch 与 warp
 *        shuffle 三种写法" -- section 一 (inclusive / exclusive definitions,
 *        the serial accumulate loop, compaction by exclusive scan, the radix
 *        split and the bracket check).
 *   [P2] lpnh.cn/news/2866224, "并行扫描 Scan/Prefix Sum" -- section 2.1
 *        (sequential_scan), section 2.2 and 3.3 (any associative operator),
 *        section 4.1 (stream_compact pseudo-code).
 *   [P3] pgsm.cn/news/414823, "SIMT数据依赖与并行前缀和" -- section 4.1/4.2
 *        (compaction of int values by a bool validity array, count output).
 *
 * Every routine is the plain serial definition: one pass, one accumulator,
 * no blocking and no reordering.
 *
 * Readings taken where the pages are silent:
 *   - exclusive scan starts from the identity of the operator (P1 section 一
 *     fixes z[0] = 0 for addition only): 0 for add and xor, INT32_MIN for
 *     int32 max, 0 for uint32 max, -infinity for fp32 max;
 *   - int32 addition wraps modulo 2^32 (computed in uint32_t, no signed
 *     overflow);
 *   - fp32 addition is accumulated in fp64 (this is the tolerance reference,
 *     not an fp32 result); fp32 max keeps fmaxf semantics and is exact;
 *   - a compaction flag keeps its element when it is nonzero.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_ADD 0
#define ORACLE_MAX 1
#define ORACLE_XOR 2

/* Return codes: 0 = ok, -1 = operator not defined for the type. */

/* ---- int32 --------------------------------------------------------------
 * P1 section 一: y[i] = x[0] + ... + x[i] (inclusive), z[i] = x[0] + ... +
 * x[i-1] with z[0] the identity (exclusive).  P2 section 2.2 / 3.3: the same
 * loop for any associative operator. */
static uint32_t op_i32(int op, uint32_t a, uint32_t b)
{
    switch (op) {
    case ORACLE_ADD: return a + b; /* wraps mod 2^32 */
    case ORACLE_MAX: return ((int32_t)a >= (int32_t)b) ? a : b;
    default:         return a ^ b;
    }
}

int oracle_scan_i32(const int32_t *x, int32_t *y, size_t n, int op, int inclusive)
{
    if (op != ORACLE_ADD && op != ORACLE_MAX && op != ORACLE_XOR) return -1;
    uint32_t acc = (op == ORACLE_MAX) ? (uint32_t)INT32_MIN : 0u;
    for (size_t i = 0; i < n; ++i) {
        uint32_t xi = (uint32_t)x[i];
        if (inclusive) {
            acc = op_i32(op, acc, xi);
            y[i] = (int32_t)acc;
        } else {
            y[i] = (int32_t)acc;
            acc = op_i32(op, acc, xi);
        }
    }
    return 0;
}

/* ---- uint32 ------------------------------------------------------------- */
static uint32_t op_u32(int op, uint32_t a, uint32_t b)
{
    switch (op) {
    case ORACLE_ADD: return a + b;
    case ORACLE_MAX: return (a >= b) ? a : b;
    default:         return a ^ b;
    }
}

int oracle_scan_u32(const uint32_t *x, uint32_t *y, size_t n, int op, int inclusive)
{
    if (op != ORACLE_ADD && op != ORACLE_MAX && op != ORACLE_XOR) return -1;
    uint32_t acc = 0u; /* identity of add, xor and unsigned max */
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc = op_u32(op, acc, x[i]);
            y[i] = acc;
        } else {
            y[i] = acc;
            acc = op_u32(op, acc, x[i]);
        }
    }
    return 0;
}

/* ---- fp32 inputs, fp64 reference outputs ---------------------------------
 * Addition accumulates in double: the reference against which the fp32
 * device result is judged (P1 pitfalls: floating point is not associative,
 * so a parallel order is accepted within a bound).  Max is exact in either
 * precision; the result is widened to double without rounding. */
int oracle_scan_f32(const float *x, double *y, size_t n, int op, int inclusive)
{
    if (op == ORACLE_ADD) {
        double acc = 0.0;
        for (size_t i = 0; i < n; ++i) {
            if (inclusive) {
                acc += (double)x[i];
                y[i] = acc;
            } else {
                y[i] = acc;
                acc += (double)x[i];
            }
        }
        return 0;
    }
    if (op == ORACLE_MAX) {
        float acc = -INFINITY;
        for (size_t i = 0; i < n; ++i) {
            if (inclusive) {
                acc = fmaxf(acc, x[i]);
                y[i] = (double)acc;
            } else {
                y[i] = (double)acc;
                acc = fmaxf(acc, x[i]);
            }
        }
        return 0;
    }
    return -1; /* xor is not defined on floating point values */
}

/* Running sum of |x[j]| for j <= i in double: the scale of the fp32
 * tolerance |gpu_i - ref_i| <= 1e-5 * sum_{j<=i} |x_j|. */
void oracle_abs_prefix_f32(const float *x, double *s, size_t n)
{
    double acc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        acc += fabs((double)x[i]);
        s[i] = acc;
    }
}

/* ---- segmented scan --------------------------------------------------------
 * P2 section 7.2 names the segmented scan as the building block for sparse
 * data.  Its definition: a nonzero head flag heads[i] starts a new segment at
 * i (element 0 always starts one), and each segment is scanned on its own --
 * the accumulator returns to the operator's identity at every segment start.
 * Operators, identities and fp32 precision as the plain scans above. */
int oracle_segscan_i32(const int32_t *x, const uint8_t *heads, int32_t *y, size_t n, int op, int inclusive)
{
    if (op != ORACLE_ADD && op != ORACLE_MAX && op != ORACLE_XOR) return -1;
    const uint32_t id = (op == ORACLE_MAX) ? (uint32_t)INT32_MIN : 0u;
    uint32_t acc = id;
    for (size_t i = 0; i < n; ++i) {
        if (heads[i] != 0) acc = id;
        uint32_t xi = (uint32_t)x[i];
        if (inclusive) {
            acc = op_i32(op, acc, xi);
            y[i] = (int32_t)acc;
        } else {
            y[i] = (int32_t)acc;
            acc = op_i32(op, acc, xi);
        }
    }
    return 0;
}

int oracle_segscan_u32(const uint32_t *x, const uint8_t *heads, uint32_t *y, size_t n, int op, int inclusive)
{
    if (op != ORACLE_ADD && op != ORACLE_MAX && op != ORACLE_XOR) return -1;
    uint32_t acc = 0u;
    for (size_t i = 0; i < n; ++i) {
        if (heads[i] != 0) acc = 0u;
        if (inclusive) {
            acc = op_u32(op, acc, x[i]);
            y[i] = acc;
        } else {
            y[i] = acc;
            acc = op_u32(op, acc, x[i]);
        }
    }
    return 0;
}

int oracle_segscan_f32(const float *x, const uint8_t *heads, double *y, size_t n, int op, int inclusive)
{
    if (op == ORACLE_ADD) {
        double acc = 0.0;
        for (size_t i = 0; i < n; ++i) {
            if (heads[i] != 0) acc = 0.0;
            if (inclusive) {
                acc += (double)x[i];
                y[i] = acc;
            } else {
                y[i] = acc;
                acc += (double)x[i];
            }
        }
        return 0;
    }
    if (op == ORACLE_MAX) {
        float acc = -INFINITY;
        for (size_t i = 0; i < n; ++i) {
            if (heads[i] != 0) acc = -INFINITY;
            if (inclusive) {
                acc = fmaxf(acc, x[i]);
                y[i] = (double)acc;
            } else {
                y[i] = (double)acc;
                acc = fmaxf(acc, x[i]);
            }
        }
        return 0;
    }
    return -1;
}

/* Running sum of |x[j]| over the segment of i up to i, in double: the scale
 * of the fp32 tolerance of the segmented scan. */
void oracle_seg_abs_prefix_f32(const float *x, const uint8_t *heads, double *s, size_t n)
{
    double acc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        if (heads[i] != 0) acc = 0.0;
        acc += fabs((double)x[i]);
        s[i] = acc;
    }
}

/* ---- stream compaction -----------------------------------------------------
 * P2 section 4.1 and P3 section 4.1: keep in[i] when its flag is set, in
 * input order; the number kept is the count.  Returns the count. */
int64_t oracle_compact_i32(const int32_t *in, const uint8_t *flags, int32_t *out, size_t n)
{
    int64_t k = 0;
    for (size_t i = 0; i < n; ++i) {
        if (flags[i] != 0) {
            out[k] = in[i];
            ++k;
        }
    }
    return k;
}

/* ---- radix one-bit split ---------------------------------------------------
 * P1 section 一 (radix sort): the keys whose bit `bit` is 0 come first, then
 * the keys whose bit is 1, each group in input order (a stable partition).
 * Returns the number of zeros. */
int64_t oracle_split_bit_u32(const uint32_t *keys, uint32_t *out, int bit, size_t n)
{
    int64_t k = 0;
    for (size_t i = 0; i < n; ++i)
        if (((keys[i] >> bit) & 1u) == 0u) out[k++] = keys[i];
    int64_t zeros = k;
    for (size_t i = 0; i < n; ++i)
        if (((keys[i] >> bit) & 1u) != 0u) out[k++] = keys[i];
    return zeros;
}

/* Least-significant-bit-first radix sort: 32 one-bit splits, bit 0 to 31,
 * ping-ponging between `keys` and `tmp`.  After an even number of passes the
 * sorted keys are back in `keys`. */
void oracle_sort_lsd_u32(uint32_t *keys, uint32_t *tmp, size_t n)
{
    uint32_t *src = keys, *dst = tmp;
    for (int bit = 0; bit < 32; ++bit) {
        oracle_split_bit_u32(src, dst, bit, n);
        uint32_t *t = src;
        src = dst;
        dst = t;
    }
}

/* ---- bracket check --------------------------------------------------------
 * P1 section 一: with '(' as +1 and ')' as -1, a negative running sum means a
 * surplus ')', and a nonzero final sum means the brackets do not pair up.
 * Input: the inclusive add-scan of the +1/-1 sequence. */
void oracle_bracket_flags(const int32_t *incl, size_t n, int *neg_prefix, int *unbalanced)
{
    int neg = 0;
    for (size_t i = 0; i < n; ++i)
        if (incl[i] < 0) neg = 1;
    *neg_prefix = neg;
    *unbalanced = (n > 0 && incl[n - 1] != 0) ? 1 : 0;
}
