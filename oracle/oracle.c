/*
 * CPU oracle for the Purlin collectives -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference leg may load this library.  The product path (libpurlin1) never
 * calls it, links it or shares code with it.
 *
 * Source: "Purlin: Separating Orchestration from the Datapath of Collectives"
 * (paper pages).  The abstract states that a collective is named by an input
 * layout, an output layout and a copy or reduction operation; the Figure 4
 * caption fixes the placements on three ranks:
 *   - ReduceScatter combines partition k of every input into y_k at rank k;
 *   - AllGather places every y_k, in rank order, at every rank;
 *   - AllToAll gives rank j partition j of every source.
 * The Figure 6 caption composes AllReduce as ReduceScatter then AllGather.
 * Table 2 adds the variable-length (V) forms.
 *
 * Readings taken where the pages say nothing (each listed in the design notes):
 *   - outputs are placed in source-rank order at prefix-sum offsets;
 *   - a sum is accumulated in fp32, in rank order 0..R-1, starting from the
 *     rank-0 value (so -0 + -0 stays -0), with IEEE round-to-nearest-even on
 *     every add and no flush of subnormals, then rounded ONCE to the output type;
 *   - the composed AllReduce's intermediate y_k is that once-rounded value, so
 *     AllReduce equals the direct per-element definition bit for bit.
 *   - the maximum is a rank-ordered fold that takes rank r's value when it is
 *     greater (IEEE comparison), so NaN counts only from rank 0 and of two
 *     zeros the earlier rank's sign is kept;
 *   - fp16 follows the same fp32-accumulate, round-once rule as bf16; 1-byte
 *     (fp8) elements are only moved, never reduced.
 *
 * Everything here is a plain loop over elements; nothing is blocked, fused or
 * reordered.  Build: plain C11, -O2 -fno-fast-math -ffp-contract=off.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs fp32 arithmetic evaluated in fp32 (FLT_EVAL_METHOD == 0)"
#endif

enum { ORC_BF16 = 0, ORC_FP32 = 1, ORC_FP16 = 2, ORC_U8 = 3 };
enum { ORC_COPY = 0, ORC_SUM = 1, ORC_MAX = 2 };

/* ---------------------------------------------------------------- bf16 --- */

/* A bf16 number is the upper half of the fp32 number with the same value. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Exact value of the bf16 bit pattern held in the upper half of `bits`, with
 * an unbounded exponent: the all-ones exponent with a zero fraction stands for
 * 2^128, the number one step above the largest finite bf16. */
static double bf16_pattern_value(uint32_t bits)
{
    uint32_t e = (bits >> 23) & 0xFFu;
    uint32_t f = (bits >> 16) & 0x7Fu;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);               /* subnormal: f * 2^-126 * 2^-7 */
    else
        mag = ldexp(1.0 + (double)f / 128.0, (int)e - 127);
    return mag;
}

/* fp32 -> bf16 by IEEE round-to-nearest, ties-to-even, from the definition:
 * the candidates are the bf16 number t obtained by dropping the low 16 bits
 * (the neighbour toward zero) and the next bf16 number a away from zero; the
 * nearer one wins and a tie goes to the one whose last kept bit is 0.  A
 * result beyond the largest finite bf16 is infinity.  NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040u);
    if (isinf(x))
        return (uint16_t)(u >> 16);
    uint32_t t = u & 0xFFFF0000u;
    uint32_t a = t + 0x00010000u;              /* carries into the exponent as needed */
    double ax = fabs((double)x);
    double dt = ax - bf16_pattern_value(t);    /* exact: same binade, 2^-149 grid */
    double da = bf16_pattern_value(a) - ax;
    uint32_t pick;
    if (dt < da)
        pick = t;
    else if (da < dt)
        pick = a;
    else
        pick = ((t >> 16) & 1u) ? a : t;
    return (uint16_t)(pick >> 16);
}

/* The same rounding applied to an array (for tests that sweep many patterns). */
void orc_f32_to_bf16_n(const float* x, uint16_t* y, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i)
        y[i] = orc_f32_to_bf16(x[i]);
}

/* ---------------------------------------------------------------- fp16 --- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h)
{
    int e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 31)
        v = f ? (double)NAN : (double)INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -24);
    else
        v = ldexp(1.0 + f / 1024.0, e - 15);
    return (float)((h & 0x8000) ? -v : v); /* every binary16 value is exact in fp32 */
}

/* fp32 -> binary16, round to nearest, ties to even, from the definition: on
 * the binary16 grid of |x|'s binade (spacing 2^(e-10) for |x| in [2^e,
 * 2^(e+1)), 2^-24 below 2^-14) take the nearer neighbour, the even multiple
 * on a tie; a result of 2^16 or more is infinity.  All steps are exact in
 * double precision (power-of-two scalings of an fp32 value). */
uint16_t orc_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    if (isinf(x))
        return (uint16_t)(sign | 0x7C00u);
    const double a = fabs((double)x);
    double ulp;
    if (a < ldexp(1.0, -14)) {
        ulp = ldexp(1.0, -24);
    } else {
        int e;
        frexp(a, &e); /* a = m * 2^e, m in [0.5, 1): the binade is [2^(e-1), 2^e) */
        ulp = ldexp(1.0, (e - 1) - 10);
    }
    const double q = a / ulp;
    const double t = floor(q);
    const double rem = q - t;
    double n;
    if (rem < 0.5)
        n = t;
    else if (rem > 0.5)
        n = t + 1.0;
    else
        n = fmod(t, 2.0) == 0.0 ? t : t + 1.0;
    const double v = n * ulp;
    if (v >= 65536.0)
        return (uint16_t)(sign | 0x7C00u);
    if (v < ldexp(1.0, -14))
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24)));
    int e;
    const double m = frexp(v, &e);
    const int biased = (e - 1) + 15;
    const uint16_t frac = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | frac);
}

void orc_f32_to_f16_n(const float* x, uint16_t* y, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i)
        y[i] = orc_f32_to_f16(x[i]);
}

/* ------------------------------------------------------- element access --- */

static size_t esize(int dtype)
{
    switch (dtype) {
    case ORC_BF16:
    case ORC_FP16:
        return 2u;
    case ORC_U8:
        return 1u;
    default:
        return 4u;
    }
}

static float load_f32(const void* buf, int dtype, uint64_t i)
{
    if (dtype == ORC_BF16)
        return orc_bf16_to_f32(((const uint16_t*)buf)[i]);
    if (dtype == ORC_FP16)
        return orc_f16_to_f32(((const uint16_t*)buf)[i]);
    return ((const float*)buf)[i];
}

static void store_f32(void* buf, int dtype, uint64_t i, float v)
{
    if (dtype == ORC_BF16)
        ((uint16_t*)buf)[i] = orc_f32_to_bf16(v);
    else if (dtype == ORC_FP16)
        ((uint16_t*)buf)[i] = orc_f32_to_f16(v);
    else
        ((float*)buf)[i] = v;
}

static void copy_elem(void* dst, uint64_t di, const void* src, uint64_t si, int dtype)
{
    size_t s = esize(dtype);
    memcpy((char*)dst + di * s, (const char*)src + si * s, s);
}

/* The reduction of one element position over R inputs: fp32, rank order. */
static float fold_ranks(int R, int dtype, const void* const* bufs, const uint64_t* idx)
{
    float acc = load_f32(bufs[0], dtype, idx[0]);
    for (int r = 1; r < R; ++r)
        acc = acc + load_f32(bufs[r], dtype, idx[r]);
    return acc;
}

/* The maximum of one element position over R inputs, in rank order: start
 * from rank 0's value and take rank r's value when it is greater.  NaN never
 * compares greater, so a NaN counts only from rank 0, and of +0 and -0 the
 * earlier rank's is kept. */
static float fold_max(int R, int dtype, const void* const* bufs, const uint64_t* idx)
{
    float acc = load_f32(bufs[0], dtype, idx[0]);
    for (int r = 1; r < R; ++r) {
        const float v = load_f32(bufs[r], dtype, idx[r]);
        if (v > acc)
            acc = v;
    }
    return acc;
}

static float fold_op(int op, int R, int dtype, const void* const* bufs, const uint64_t* idx)
{
    return op == ORC_MAX ? fold_max(R, dtype, bufs, idx) : fold_ranks(R, dtype, bufs, idx);
}

/* ------------------------------------------------ the seven collectives --- */

/* AllGather(V): rank j contributes n[j] elements; every rank r receives them
 * all, in rank order: out_r[sum_{k<j} n_k + i] = in_j[i]. */
void orc_allgather(int R, int dtype, const void* const* in, const uint64_t* n, void* const* out)
{
    for (int r = 0; r < R; ++r) {
        uint64_t base = 0;
        for (int j = 0; j < R; ++j) {
            for (uint64_t i = 0; i < n[j]; ++i)
                copy_elem(out[r], base + i, in[j], i, dtype);
            base += n[j];
        }
    }
}

/* ReduceScatter(V) with the reduction `op` (sum or max): every input is split
 * into partitions of lengths n[0..R-1] at prefix offsets o_k; rank k receives
 * y_k[i] = round(fold_r in_r[o_k + i]). */
void orc_reducescatter_op(int R, int dtype, int op, const void* const* in, const uint64_t* n, void* const* out)
{
    uint64_t idx[64];
    uint64_t o = 0;
    for (int k = 0; k < R; ++k) {
        for (uint64_t i = 0; i < n[k]; ++i) {
            for (int r = 0; r < R; ++r)
                idx[r] = o + i;
            store_f32(out[k], dtype, i, fold_op(op, R, dtype, in, idx));
        }
        o += n[k];
    }
}

/* ReduceScatter(V) with the sum (Figure 4). */
void orc_reducescatter(int R, int dtype, const void* const* in, const uint64_t* n, void* const* out)
{
    orc_reducescatter_op(R, dtype, ORC_SUM, in, n, out);
}

/* AllReduce with the reduction `op`, direct definition: out_r[i] =
 * round(fold_r' in_r'[i]) for all r. */
void orc_allreduce_op(int R, int dtype, int op, const void* const* in, uint64_t count, void* const* out)
{
    uint64_t idx[64];
    for (uint64_t i = 0; i < count; ++i) {
        for (int r = 0; r < R; ++r)
            idx[r] = i;
        const float v = fold_op(op, R, dtype, in, idx);
        for (int r = 0; r < R; ++r)
            store_f32(out[r], dtype, i, v);
    }
}

/* AllReduce with the sum. */
void orc_allreduce(int R, int dtype, const void* const* in, uint64_t count, void* const* out)
{
    orc_allreduce_op(R, dtype, ORC_SUM, in, count, out);
}

/* AllToAll(V): source r splits its input into partitions of lengths
 * nm[r*R + j] (j = destination); rank j receives partition j of every source,
 * in source order: out_j[sum_{r'<r} nm[r'*R+j] + i] = in_r[sum_{j'<j} nm[r*R+j'] + i]. */
void orc_alltoall(int R, int dtype, const void* const* in, const uint64_t* nm, void* const* out)
{
    for (int j = 0; j < R; ++j) {
        uint64_t dst_base = 0;
        for (int r = 0; r < R; ++r) {
            uint64_t src_base = 0;
            for (int jj = 0; jj < j; ++jj)
                src_base += nm[(uint64_t)r * R + jj];
            uint64_t len = nm[(uint64_t)r * R + j];
            for (uint64_t i = 0; i < len; ++i)
                copy_elem(out[j], dst_base + i, in[r], src_base + i, dtype);
            dst_base += len;
        }
    }
}

/* Ulysses sequence <-> head re-partition (Table 2, Ulysses row): rank r holds
 * [S, H, D] (S = its sequence shard); destination j gets heads
 * [j*H/R, (j+1)*H/R) of every source, stacked in source order:
 * out_j[((r*S + s)*(H/R) + h)*D + d] = in_r[(s*H + j*H/R + h)*D + d]. */
void orc_ulysses(int R, int dtype, const void* const* in, uint64_t S, uint64_t H, uint64_t D, void* const* out)
{
    uint64_t hs = H / (uint64_t)R;
    for (int j = 0; j < R; ++j)
        for (int r = 0; r < R; ++r)
            for (uint64_t s = 0; s < S; ++s)
                for (uint64_t h = 0; h < hs; ++h)
                    for (uint64_t d = 0; d < D; ++d)
                        copy_elem(out[j], (((uint64_t)r * S + s) * hs + h) * D + d,
                                  in[r], (s * H + (uint64_t)j * hs + h) * D + d, dtype);
}

/* ------------------------------------------- the layout-pair definition --- */

/* One named region of one rank's buffer: `rows` rows of `len` elements, row i
 * starting at element offset + i * row_stride.  Element j of the region (in
 * row-major order) is at offset + (j / len) * row_stride + j % len. */
typedef struct {
    uint64_t name, offset, len, rows, row_stride;
} orc_part;

static uint64_t region_elem(const orc_part* p, uint64_t j)
{
    return p->offset + (j / p->len) * p->row_stride + (j % p->len);
}

static uint64_t region_count(const orc_part* p) { return p->rows * p->len; }

/* Any collective given as (input layout, output layout, op): every output
 * region named p receives, element by element, the unique input region named
 * p (COPY) or the rank-ordered fp32 sum of the R input regions named p, one
 * per rank (SUM).  Returns 0, or 1 when the layout pair names no valid
 * collective (a name without its sources, COPY with several sources, SUM
 * without exactly one source per rank, or mismatched element counts). */
int orc_collective(int R, int op, int dtype,
                   const int* nin, const orc_part* in_parts, const void* const* in_bufs,
                   const int* nout, const orc_part* out_parts, void* const* out_bufs)
{
    if (R < 1 || R > 64)
        return 1;
    int in_first[65], out_first[65];
    in_first[0] = out_first[0] = 0;
    for (int r = 0; r < R; ++r) {
        in_first[r + 1] = in_first[r] + nin[r];
        out_first[r + 1] = out_first[r] + nout[r];
    }
    for (int d = 0; d < R; ++d) {
        for (int q = out_first[d]; q < out_first[d + 1]; ++q) {
            const orc_part* dp = &out_parts[q];
            uint64_t cnt = region_count(dp);
            const orc_part* src[64];
            int src_rank[64];
            int ns = 0;
            for (int r = 0; r < R; ++r)
                for (int s = in_first[r]; s < in_first[r + 1]; ++s)
                    if (in_parts[s].name == dp->name) {
                        if (ns == 64)
                            return 1;
                        src[ns] = &in_parts[s];
                        src_rank[ns] = r;
                        ++ns;
                    }
            if (op != ORC_COPY && dtype == ORC_U8)
                return 1; /* 1-byte elements are moved, never reduced */
            if (op == ORC_COPY) {
                if (ns != 1 || region_count(src[0]) != cnt)
                    return 1;
                for (uint64_t j = 0; j < cnt; ++j)
                    copy_elem(out_bufs[d], region_elem(dp, j), in_bufs[src_rank[0]],
                              region_elem(src[0], j), dtype);
            } else {
                if (ns != R)
                    return 1;
                for (int r = 0; r < R; ++r)
                    if (src_rank[r] != r || region_count(src[r]) != cnt)
                        return 1;
                uint64_t idx[64];
                for (uint64_t j = 0; j < cnt; ++j) {
                    for (int r = 0; r < R; ++r)
                        idx[r] = region_elem(src[r], j);
                    store_f32(out_bufs[d], dtype, region_elem(dp, j),
                              fold_op(op, R, dtype, in_bufs, idx));
                }
            }
        }
    }
    return 0;
}
