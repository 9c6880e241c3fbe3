/*
 * oracle.c -- plain, slow CPU definition of the sum collectives.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (the usual sum collectives, which point (3) of the MSCCL++
 * abstract offers as a collection of ready-made algorithms; the AllReduce use
 * case is in the project summary, "Highlighted Details"):
 *
 *   AllReduce      out[i]        = R( x_0[i] + x_1[i] + ... + x_{N-1}[i] )
 *   ReduceScatter  out_r[j]      = R( sum_p x_p[r*m + j] )
 *   AllGather      out[q*m + j]  = x_q[j]                    (bit copy)
 *
 * The pages do not fix the arithmetic, so this file takes the plainest
 * reading:
 *   - the sum runs left to right in rank order 0..N-1 and starts from x_0
 *     (not from +0.0, which would turn an all -0.0 column into +0.0);
 *   - fp32, fp16 and bf16 inputs are widened exactly to fp32 and accumulated
 *     in fp32 with IEEE round-to-nearest-even after every add, subnormals
 *     kept; R rounds the fp32 sum once to the output type (RNE);
 *   - int32 accumulates with two's-complement wraparound.
 * MAX / MIN AllReduce (orc_allreduce_op) is not on the pages, which speak of
 * sum reductions only; it follows the IEEE 754-2019 maximum / minimum
 * operations in rank order: a NaN in any rank gives the canonical quiet NaN
 * (positive, top mantissa bit set; for every N, one rank included), -0
 * orders below +0, and int32 takes the integer maximum / minimum.
 * The widening/narrowing routines below are written from the IEEE-754
 * binary16 format and from bfloat16 being the top 16 bits of binary32.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -shared -fPIC
 * (the C compiler's float additions are IEEE binary32 on x86-64 SSE and on
 * aarch64, round-to-nearest-even, no flush-to-zero).
 *
 * Parity: every function here is pinned by the CPU tests (closed forms,
 * exhaustive conversion round trips, an independent pure-Python brute force,
 * library conversion routines).  None is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* element kinds, private to the oracle (the Python wrapper maps names) */
enum { ORC_INT32 = 0, ORC_FP32 = 1, ORC_FP16 = 2, ORC_BF16 = 3 };

/* ---------------------------------------------------------------------- */
/* binary32 bit access                                                     */
/* ---------------------------------------------------------------------- */
static float bits_to_f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* ---------------------------------------------------------------------- */
/* bfloat16: sign, 8 exponent bits, 7 fraction bits -- the upper half of a */
/* binary32 word.  Widening appends 16 zero fraction bits (exact).         */
/* ---------------------------------------------------------------------- */
float orc_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* Narrowing: keep the upper 16 bits and round the 16 dropped fraction bits
 * to nearest, ties to even.  Sign-magnitude: rounding the magnitude bits
 * rounds |x|, and a carry out of the fraction moves into the exponent
 * (so the largest finite values round up to infinity as IEEE requires).
 * NaN stays NaN (quiet bit set, sign kept). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t b = f32_to_bits(f);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0)
        return (uint16_t)((b >> 16) | 0x0040u);              /* quiet NaN */
    uint32_t hi = b >> 16;
    uint32_t dropped = b & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

/* ---------------------------------------------------------------------- */
/* binary16: sign, 5 exponent bits (bias 15), 10 fraction bits.            */
/* ---------------------------------------------------------------------- */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F) {
        if (m == 0) v = INFINITY;
        else return bits_to_f32(((uint32_t)sign << 31) | 0x7FC00000u | ((uint32_t)m << 13));
    } else if (e == 0) {
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    } else {
        v = ldexp((double)(1024 + m), e - 25);     /* (1.m) * 2^(e-15) */
    }
    return (float)(sign ? -v : v);                 /* exact: fits binary32 */
}

/* Narrowing from the definition: pick the binade, scale |x| to an integer
 * count of quanta of that binade (exact in double), round that count to
 * nearest with ties to even, and re-encode.  |x| >= 65520 (the midpoint
 * between 65504, the largest finite half, and 2^16) rounds to infinity. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t b = f32_to_bits(f);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    if ((b & 0x7F800000u) == 0x7F800000u) {
        if (b & 0x007FFFFFu)
            return (uint16_t)(sign | 0x7E00u | ((b >> 13) & 0x03FFu));   /* NaN */
        return (uint16_t)(sign | 0x7C00u);                               /* inf */
    }
    double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);            /* a = frac * 2^e2, frac in [0.5, 1) */
    int e = e2 - 1;                 /* a in [2^e, 2^(e+1)) */
    if (e < -14) e = -14;           /* subnormal range shares the 2^-24 quantum */
    double q = ldexp(1.0, e - 10);  /* one unit in the last place of the binade */
    double n = a / q;               /* exact: a has 24 significant bits */
    double fl = floor(n);
    double r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    long k = (long)fl;              /* number of quanta, <= 2048 */
    if (k == 0) return sign;
    if (e == -14 && k < 1024) return (uint16_t)(sign | (uint16_t)k);   /* subnormal */
    if (k == 2048) { k = 1024; e += 1; }                  /* rounded into the next binade */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(k - 1024));
}

/* ---------------------------------------------------------------------- */
/* element access                                                          */
/* ---------------------------------------------------------------------- */
static size_t elem_size(int dtype)
{
    switch (dtype) {
    case ORC_INT32: case ORC_FP32: return 4;
    case ORC_FP16: case ORC_BF16: return 2;
    default: return 0;
    }
}

static float widen(const void* buf, size_t i, int dtype)
{
    switch (dtype) {
    case ORC_FP32: return ((const float*)buf)[i];
    case ORC_FP16: return orc_f16_to_f32(((const uint16_t*)buf)[i]);
    default:       return orc_bf16_to_f32(((const uint16_t*)buf)[i]);
    }
}

/* binary64 -> fp16 / bf16 with one round-to-nearest-even, from the IEEE-754
 * formats: p significant bits (implicit one included), exponents emin..emax,
 * subnormals down to 2^(emin - p + 1), overflow to infinity at the midpoint
 * above the largest finite value.  Used where a result is defined as a
 * binary64 value rounded once to the 16-bit output type. */
static uint16_t f64_to_half_once(double v, int dtype)
{
    const int p = dtype == ORC_FP16 ? 11 : 8, emin = dtype == ORC_FP16 ? -14 : -126,
              emax = dtype == ORC_FP16 ? 15 : 127, bias = dtype == ORC_FP16 ? 15 : 127;
    const uint16_t sign = signbit(v) ? 0x8000u : 0u, exp_all = dtype == ORC_FP16 ? 0x7C00u : 0x7F80u;
    if (isnan(v)) return (uint16_t)(sign | exp_all | (dtype == ORC_FP16 ? 0x0200u : 0x0040u));
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);             /* a in [2^(e2-1), 2^e2) */
    int e = e2 - 1;
    if (e < emin) e = emin;          /* subnormals share the smallest quantum */
    double q = ldexp(1.0, e - (p - 1));
    double n = a / q;                /* exact: a power-of-two scaling */
    double fl = floor(n);
    double r = n - fl;               /* exact */
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    long k = (long)fl;               /* quanta, <= 2^p */
    const long one = 1L << (p - 1);
    if (k == 0) return sign;
    if (e == emin && k < one) return (uint16_t)(sign | (uint16_t)k);   /* subnormal */
    if (k == 2 * one) { k = one; e += 1; }                             /* next binade */
    if (e > emax) return (uint16_t)(sign | exp_all);                   /* overflow */
    return (uint16_t)(sign | (uint16_t)((e + bias) << (p - 1)) | (uint16_t)(k - one));
}

static void narrow_store(void* buf, size_t i, float v, int dtype)
{
    switch (dtype) {
    case ORC_FP32: ((float*)buf)[i] = v; break;
    case ORC_FP16: ((uint16_t*)buf)[i] = orc_f32_to_f16(v); break;
    default:       ((uint16_t*)buf)[i] = orc_f32_to_bf16(v); break;
    }
}

/* One output element of the sum: rank order 0..n-1, starting from x_0. */
static void reduce_one(int n, const void* const* in, size_t src_i,
                       void* out, size_t dst_i, int dtype)
{
    if (dtype == ORC_INT32) {
        uint32_t acc = (uint32_t)((const int32_t*)in[0])[src_i];
        for (int p = 1; p < n; ++p)
            acc += (uint32_t)((const int32_t*)in[p])[src_i];   /* wraps mod 2^32 */
        ((int32_t*)out)[dst_i] = (int32_t)acc;                  /* two's complement */
        return;
    }
    float acc = widen(in[0], src_i, dtype);
    for (int p = 1; p < n; ++p)
        acc = acc + widen(in[p], src_i, dtype);
    narrow_store(out, dst_i, acc, dtype);
}

static int check_args(int n, const void* const* in, int dtype)
{
    if (n < 1 || in == NULL || elem_size(dtype) == 0) return -1;
    for (int p = 0; p < n; ++p) if (in[p] == NULL) return -1;
    return 0;
}

/* ---------------------------------------------------------------------- */
/* AllReduce                                                               */
/* ---------------------------------------------------------------------- */
int orc_allreduce(int n, const void* const* in, void* out, size_t count, int dtype)
{
    if (check_args(n, in, dtype) || (count && !out)) return -1;
    for (size_t i = 0; i < count; ++i) reduce_one(n, in, i, out, i, dtype);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* AllReduce with MAX or MIN: an extension the pages do not define.  Plain */
/* reading: the ranks' values combine in rank order 0..N-1 starting from   */
/* x_0 with the IEEE 754-2019 maximum / minimum operations -- a NaN        */
/* operand gives NaN, and -0 orders below +0.  16-bit inputs widen exactly */
/* to binary32 and the result is one of the inputs (or NaN), so storing it */
/* rounds nothing.  int32 takes the integer maximum / minimum.             */
/* ---------------------------------------------------------------------- */
#define ORC_OP_MAX 1
#define ORC_OP_MIN 2

static float max_ieee(float a, float b)
{
    if (isnan(a) || isnan(b)) return NAN;
    if (a == b) return signbit(a) ? b : a;   /* equal values, or +0 and -0: +0 wins */
    return a > b ? a : b;
}

static float min_ieee(float a, float b)
{
    if (isnan(a) || isnan(b)) return NAN;
    if (a == b) return signbit(a) ? a : b;   /* -0 wins */
    return a < b ? a : b;
}

int orc_allreduce_op(int n, const void* const* in, void* out, size_t count, int dtype, int op)
{
    if (check_args(n, in, dtype) || (count && !out) || (op != ORC_OP_MAX && op != ORC_OP_MIN)) return -1;
    for (size_t i = 0; i < count; ++i) {
        if (dtype == ORC_INT32) {
            int32_t acc = ((const int32_t*)in[0])[i];
            for (int p = 1; p < n; ++p) {
                const int32_t v = ((const int32_t*)in[p])[i];
                acc = op == ORC_OP_MAX ? (v > acc ? v : acc) : (v < acc ? v : acc);
            }
            ((int32_t*)out)[i] = acc;
            continue;
        }
        float acc = widen(in[0], i, dtype);
        for (int p = 1; p < n; ++p)
            acc = op == ORC_OP_MAX ? max_ieee(acc, widen(in[p], i, dtype)) : min_ieee(acc, widen(in[p], i, dtype));
        if (isnan(acc)) acc = NAN;   /* canonical at N = 1 too, where no operation ran */
        narrow_store(out, i, acc, dtype);
    }
    return 0;
}

/* The same definition at chosen indices only: out[k] = R(sum_p x_p[idx[k]]).
 * Used to check outputs of full-size runs one sampled element at a time. */
int orc_allreduce_at(int n, const void* const* in, size_t count, int dtype,
                     const int64_t* idx, size_t nidx, void* out)
{
    if (check_args(n, in, dtype) || (nidx && (!idx || !out))) return -1;
    for (size_t k = 0; k < nidx; ++k) {
        if (idx[k] < 0 || (size_t)idx[k] >= count) return -1;
        reduce_one(n, in, (size_t)idx[k], out, k, dtype);
    }
    return 0;
}

/* Threaded form for timing only: the element range is cut into contiguous
 * pieces, one per thread; every element still sums in rank order, so the
 * result is bit-identical to orc_allreduce. */
typedef struct {
    int n; const void* const* in; void* out; int dtype; size_t lo, hi;
} orc_job;

static void* allreduce_job(void* arg)
{
    orc_job* j = (orc_job*)arg;
    for (size_t i = j->lo; i < j->hi; ++i) reduce_one(j->n, j->in, i, j->out, i, j->dtype);
    return NULL;
}

int orc_allreduce_mt(int n, const void* const* in, void* out, size_t count, int dtype,
                     int nthreads)
{
    if (check_args(n, in, dtype) || (count && !out)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int joined[256];
    orc_job jobs[256];
    size_t per = (count + (size_t)nthreads - 1) / (size_t)nthreads;
    for (int t = 0; t < nthreads; ++t) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo > count) lo = count;
        if (hi > count) hi = count;
        jobs[t] = (orc_job){n, in, out, dtype, lo, hi};
        joined[t] = pthread_create(&th[t], NULL, allreduce_job, &jobs[t]) == 0;
        if (!joined[t]) allreduce_job(&jobs[t]);      /* no thread: run inline */
    }
    for (int t = 0; t < nthreads; ++t)
        if (joined[t]) pthread_join(th[t], NULL);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* ReduceScatter: rank r receives the reduced r-th block of m elements.    */
/* ---------------------------------------------------------------------- */
int orc_reduce_scatter(int n, const void* const* in, void* out, int rank,
                       size_t recv_count, int dtype)
{
    if (check_args(n, in, dtype) || rank < 0 || rank >= n || (recv_count && !out)) return -1;
    for (size_t j = 0; j < recv_count; ++j)
        reduce_one(n, in, (size_t)rank * recv_count + j, out, j, dtype);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* AllGather: every rank receives x_0 | x_1 | ... | x_{N-1}.               */
/* ---------------------------------------------------------------------- */
int orc_allgather(int n, const void* const* in, void* out, size_t send_count, int dtype)
{
    if (check_args(n, in, dtype) || (send_count && !out)) return -1;
    size_t es = elem_size(dtype);
    for (int q = 0; q < n; ++q)
        memcpy((char*)out + (size_t)q * send_count * es, in[q], send_count * es);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Ring barrier bookkeeping.  One iteration passes a token once around the */
/* ring: rank r signals rank (r+1) mod N exactly once.  After `iters`      */
/* iterations the inbound counter of rank d for signals from rank s is     */
/* iters when s = (d-1) mod N, else 0.  counts is N*N, row d, column s.    */
/* ---------------------------------------------------------------------- */
int orc_ring_barrier_counts(int n, uint64_t iters, uint64_t* counts)
{
    if (n < 1 || !counts) return -1;
    for (int d = 0; d < n; ++d)
        for (int s = 0; s < n; ++s)
            counts[d * n + s] = (s == (d + n - 1) % n) ? iters : 0;
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Row-parallel linear layer followed by the sum AllReduce (tensor-parallel */
/* decode: every rank holds a slice of the contraction dimension).          */
/*   y[i] = R( sum_p sum_k W_p[i][k] * x_p[k] ),  i < rows, k < kp          */
/* W_p is rows x kp row-major, x_p has kp elements (fp16 or bf16).  The     */
/* products of two 16-bit floats are exact in binary64 and the sum is taken */
/* in binary64 (for the small-integer inputs the tests pin it with, exactly */
/* the real sum), then rounded once to the output type.                     */
/* ---------------------------------------------------------------------- */
/* row i of the layer: sum_p sum_k W_p[i][k] * x_p[k] in binary64 */
static double layer_row(int n, const void* const* w, const void* const* x, size_t i, size_t kp, int dtype)
{
    double acc = 0.0;
    for (int p = 0; p < n; ++p)
        for (size_t k = 0; k < kp; ++k)
            acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], k, dtype);
    return acc;
}

int orc_linear_allreduce(int n, const void* const* w, const void* const* x, size_t rows, size_t kp,
                         int dtype, void* out)
{
    if (n < 1 || !w || !x || (rows && !out) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    for (int p = 0; p < n; ++p) if (!w[p] || !x[p]) return -1;
    for (size_t i = 0; i < rows; ++i) {
        const double acc = layer_row(n, w, x, i, kp, dtype);
        ((uint16_t*)out)[i] = f64_to_half_once(acc, dtype);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* The same layer for a batch of tokens (a multi-token decode step): x_p    */
/* holds tokens x kp elements, row-major, token t's slice of the            */
/* contraction dimension at x_p + t*kp, and                                 */
/*   y[t][i] = R( sum_p sum_k W_p[i][k] * x_p[t][k] ),  t < tokens,        */
/* out is tokens x rows, row-major (token t's hidden vector at out +        */
/* t*rows).  Binary64 sum of the exact products, one rounding, exactly as   */
/* for a single token.                                                      */
/* ---------------------------------------------------------------------- */
int orc_linear_allreduce_tokens(int n, const void* const* w, const void* const* x, size_t tokens,
                                size_t rows, size_t kp, int dtype, void* out)
{
    if (n < 1 || !w || !x || (tokens && rows && !out) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    for (int p = 0; p < n; ++p) if (!w[p] || !x[p]) return -1;
    for (size_t t = 0; t < tokens; ++t)
        for (size_t i = 0; i < rows; ++i) {
            double acc = 0.0;
            for (int p = 0; p < n; ++p)
                for (size_t k = 0; k < kp; ++k)
                    acc += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], t * kp + k, dtype);
            ((uint16_t*)out)[t * rows + i] = f64_to_half_once(acc, dtype);
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* The batched layer with a residual per output rank (the residual stream  */
/* of a multi-token step, h_q <- h_q + layer): res_q holds tokens x rows     */
/* elements like the output, and the residual joins the binary64 sum       */
/* before the single rounding,                                              */
/*   y_q[t][i] = R( sum_p sum_k W_p[i][k] * x_p[t][k] + res_q[t][i] ).     */
/* out holds the N outputs one after another (rank q's at out + q*tokens*rows). */
/* ---------------------------------------------------------------------- */
int orc_linear_allreduce_tokens_residual(int n, const void* const* w, const void* const* x,
                                         const void* const* res, size_t tokens, size_t rows, size_t kp,
                                         int dtype, void* out)
{
    if (n < 1 || !w || !x || !res || (tokens && rows && !out) || (dtype != ORC_FP16 && dtype != ORC_BF16))
        return -1;
    for (int p = 0; p < n; ++p) if (!w[p] || !x[p] || !res[p]) return -1;
    for (size_t t = 0; t < tokens; ++t)
        for (size_t i = 0; i < rows; ++i) {
            double dot = 0.0;
            for (int p = 0; p < n; ++p)
                for (size_t k = 0; k < kp; ++k)
                    dot += (double)widen(w[p], i * kp + k, dtype) * (double)widen(x[p], t * kp + k, dtype);
            for (int q = 0; q < n; ++q) {
                const double y = dot + (double)widen(res[q], t * rows + i, dtype);
                ((uint16_t*)out)[((size_t)q * tokens + t) * rows + i] = f64_to_half_once(y, dtype);
            }
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* The same layer with a residual added for each output rank (the          */
/* tensor-parallel residual stream: h_q <- h_q + the layer's AllReduced    */
/* output).  Reading taken: the residual joins the binary64 sum before the */
/* single rounding,                                                        */
/*   y_q[i] = R( sum_p sum_k W_p[i][k] * x_p[k] + res_q[i] ),              */
/* res_q has rows elements of the same type; out holds the N outputs one  */
/* after another (rank q's at out + q * rows).                             */
/* ---------------------------------------------------------------------- */
int orc_linear_allreduce_residual(int n, const void* const* w, const void* const* x,
                                  const void* const* res, size_t rows, size_t kp, int dtype, void* out)
{
    if (n < 1 || !w || !x || !res || (rows && !out) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    for (int p = 0; p < n; ++p) if (!w[p] || !x[p] || !res[p]) return -1;
    for (size_t i = 0; i < rows; ++i) {
        const double acc = layer_row(n, w, x, i, kp, dtype);
        for (int q = 0; q < n; ++q) {
            const double y = acc + (double)widen(res[q], i, dtype);
            ((uint16_t*)out)[(size_t)q * rows + i] = f64_to_half_once(y, dtype);
        }
    }
    return 0;
}

/* exported conversions over arrays (used by the tests' pins) */
int orc_convert_to_f32(const uint16_t* src, float* dst, size_t count, int dtype)
{
    if (dtype != ORC_FP16 && dtype != ORC_BF16) return -1;
    for (size_t i = 0; i < count; ++i)
        dst[i] = dtype == ORC_FP16 ? orc_f16_to_f32(src[i]) : orc_bf16_to_f32(src[i]);
    return 0;
}

int orc_convert_from_f32(const float* src, uint16_t* dst, size_t count, int dtype)
{
    if (dtype != ORC_FP16 && dtype != ORC_BF16) return -1;
    for (size_t i = 0; i < count; ++i)
        dst[i] = dtype == ORC_FP16 ? orc_f32_to_f16(src[i]) : orc_f32_to_bf16(src[i]);
    return 0;
}
