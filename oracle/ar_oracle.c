/*
 * ar_oracle.c -- CPU oracle for the R-way reduce and the fused
 * reduce + bias + residual + RMSNorm.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The CUDA library never links or calls it, and it
 * shares no code, header, table or helper with the CUDA library.
 *
 * Plain, slow and single-threaded on purpose: every value is computed in
 * IEEE binary64 and rounded once, directly to the output format, with
 * round-to-nearest-even.  It is written for a reader checking it by eye.
 *
 * What it computes, and where the pages define it:
 *   - or_sum: the all-reduce is a sum of the tensor-parallel ranks' partial
 *     activations ("All Reduce Plugin", class AllReducePlugin description:
 *     all-reduce (sum) after row-parallel linear layers).  out[i] =
 *     sum_r p_r[i], summed in rank order 0..R-1.
 *   - or_residual_rmsnorm: the RESIDUAL_RMS_NORM fusion
 *     ("type.d2", AllReduceFusionOp and AllReduceFusionParams: bias_buffer
 *     (the GEMM bias), residual_buffer, hidden_size, weight_buffer,
 *     float eps, intermediate_buffer; "allreduce.d2", the
 *     one_shot_all_reduce_norm_kernel -> rms_norm edge).  The pages print
 *     no formula; the reading taken here is the textbook RMSNorm with eps
 *     inside the square root and no mean subtraction:
 *         x_j   = sum_r p_r[t,j] + bias_j + residual[t,j]
 *         inv   = 1 / sqrt( (sum_j x_j^2) / H + eps )
 *         out_j = x_j * inv * weight_j,   residual_out_j = x_j
 *     bias is added once (not per rank) and may be absent; eps is the
 *     float value the caller passes, widened exactly to double.
 *   - or_rmsnorm: the row normalisation on its own ("allreduce.d2",
 *     rms_norm_kernel_launcher -> rms_norm_kernel, the second phase of the
 *     two-shot fused route and the norm after a plain all-reduce):
 *         out_j = x_j / sqrt( (sum_j x_j^2) / H + eps ) * weight_j
 *     with the same reading of the formula as above.
 *
 * Formats (the pages' PackedOn16Bytes unions in "type.d2" name float and
 * half; bfloat16 is added beside them):
 *     code 0 = IEEE binary32, 1 = IEEE binary16, 2 = bfloat16.
 * fp16 and bf16 values travel as their 16-bit patterns.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ---------------------------------------------------------------------------
 * Format description: p = significand bits (with the implicit one),
 * emin = exponent of the smallest normal number, emax = largest exponent.
 * ------------------------------------------------------------------------- */
typedef struct { int p, emin, emax; } or_format;

static or_format format_of(int dtype)
{
    or_format f;
    switch (dtype) {
    case OR_F16:  f.p = 11; f.emin = -14;  f.emax = 15;  break;
    case OR_BF16: f.p = 8;  f.emin = -126; f.emax = 127; break;
    default:      f.p = 24; f.emin = -126; f.emax = 127; break;
    }
    return f;
}

/* Round a binary64 value to the nearest value of format f, ties to even.
 * Subnormals use the quantum of the smallest normal binade; results above
 * the largest finite value become infinities. */
double or_round_value(double v, int dtype)
{
    or_format f = format_of(dtype);
    if (isnan(v) || isinf(v) || v == 0.0)
        return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);               /* a = m * 2^e with 0.5 <= m < 1 */
    int lead = e - 1;           /* exponent of a's leading bit */
    if (lead < f.emin)
        lead = f.emin;          /* subnormal range: fixed quantum */
    double q = ldexp(1.0, lead - (f.p - 1));   /* spacing of the format here */
    double r = a / q;           /* exact: division by a power of two */
    double k = floor(r);
    double frac = r - k;        /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) != 0.0))
        k += 1.0;
    double res = k * q;         /* exact */
    double max_finite = ldexp(2.0 - ldexp(1.0, 1 - f.p), f.emax);
    if (res > max_finite)
        res = INFINITY;
    return copysign(res, v);
}

/* Bit pattern of a value that is exactly representable in the format. */
static uint32_t encode_exact(double val, int dtype)
{
    if (dtype == OR_F32 || dtype == OR_BF16) {
        float fl = (float)val;  /* exact: val is representable */
        uint32_t u;
        memcpy(&u, &fl, sizeof u);
        return dtype == OR_F32 ? u : (u >> 16);
    }
    /* binary16 */
    uint32_t sign = signbit(val) ? 0x8000u : 0u;
    double a = fabs(val);
    if (isnan(val))
        return 0x7E00u;
    if (isinf(a))
        return sign | 0x7C00u;
    if (a < ldexp(1.0, -14))                     /* subnormal or zero */
        return sign | (uint32_t)(a / ldexp(1.0, -24));
    int e;
    frexp(a, &e);
    int lead = e - 1;
    uint32_t mant = (uint32_t)((a / ldexp(1.0, lead) - 1.0) * 1024.0);
    return sign | ((uint32_t)(lead + 15) << 10) | mant;
}

uint32_t or_round_bits(double v, int dtype)
{
    return encode_exact(or_round_value(v, dtype), dtype);
}

/* Exact binary64 value of a stored element. */
double or_decode_bits(uint32_t bits, int dtype)
{
    if (dtype == OR_F32) {
        float fl;
        memcpy(&fl, &bits, sizeof fl);
        return (double)fl;
    }
    if (dtype == OR_BF16) {
        uint32_t u = bits << 16;
        float fl;
        memcpy(&fl, &u, sizeof fl);
        return (double)fl;
    }
    double sign = (bits & 0x8000u) ? -1.0 : 1.0;
    uint32_t ex = (bits >> 10) & 0x1Fu;
    uint32_t mant = bits & 0x3FFu;
    if (ex == 0)
        return sign * ldexp((double)mant, -24);
    if (ex == 31)
        return mant ? NAN : sign * INFINITY;
    return sign * ldexp((double)(1024u + mant), (int)ex - 25);
}

static double load(const void* buf, size_t i, int dtype)
{
    if (dtype == OR_F32) {
        uint32_t u;
        memcpy(&u, (const char*)buf + 4 * i, 4);
        return or_decode_bits(u, dtype);
    }
    uint16_t h;
    memcpy(&h, (const char*)buf + 2 * i, 2);
    return or_decode_bits(h, dtype);
}

static void store(void* buf, size_t i, int dtype, double v)
{
    uint32_t bits = or_round_bits(v, dtype);
    if (dtype == OR_F32) {
        memcpy((char*)buf + 4 * i, &bits, 4);
    } else {
        uint16_t h = (uint16_t)bits;
        memcpy((char*)buf + 2 * i, &h, 2);
    }
}

/* out[i] = partials[0][i] + partials[1][i] + ... + partials[R-1][i], a left
 * fold in binary64 starting from the first term (so a single partial, -0
 * included, passes through unchanged), rounded once. */
void or_sum(const void* const* partials, int R, size_t n, int dtype, void* out)
{
    for (size_t i = 0; i < n; ++i) {
        double acc = load(partials[0], i, dtype);
        for (int r = 1; r < R; ++r)
            acc += load(partials[r], i, dtype);
        store(out, i, dtype, acc);
    }
}

/* Fused sum + bias + residual + RMSNorm over a row-major [tokens, hidden]
 * tensor.  bias may be NULL (then it contributes zero).  If inv_rms is not
 * NULL it receives, per row, the binary64 factor 1/sqrt(mean(x^2)+eps).
 * x is kept for one row at a time in the caller-provided scratch `xrow`
 * (hidden doubles). */
void or_residual_rmsnorm(const void* const* partials, int R, const void* bias,
                         const void* residual, const void* weight, float eps,
                         int hidden, int tokens, int dtype,
                         void* out, void* residual_out, double* inv_rms,
                         double* xrow)
{
    for (int t = 0; t < tokens; ++t) {
        size_t row = (size_t)t * (size_t)hidden;
        double sumsq = 0.0;
        for (int j = 0; j < hidden; ++j) {
            double x = load(partials[0], row + j, dtype);
            for (int r = 1; r < R; ++r)
                x += load(partials[r], row + j, dtype);
            if (bias)
                x += load(bias, (size_t)j, dtype);
            x += load(residual, row + j, dtype);
            xrow[j] = x;
            sumsq += x * x;
        }
        double mean_sq = sumsq / (double)hidden;
        double inv = 1.0 / sqrt(mean_sq + (double)eps);
        if (inv_rms)
            inv_rms[t] = inv;
        for (int j = 0; j < hidden; ++j) {
            double w = load(weight, (size_t)j, dtype);
            store(residual_out, row + j, dtype, xrow[j]);
            store(out, row + j, dtype, xrow[j] * inv * w);
        }
    }
}

/* RMSNorm of a row-major [tokens, hidden] tensor x on its own:
 * out[t,j] = x[t,j] * (1 / sqrt(mean_j x[t,j]^2 + eps)) * weight[j], the
 * factor in binary64, rounded once.  inv_rms as in or_residual_rmsnorm. */
void or_rmsnorm(const void* x, const void* weight, float eps, int hidden, int tokens,
                int dtype, void* out, double* inv_rms)
{
    for (int t = 0; t < tokens; ++t) {
        size_t row = (size_t)t * (size_t)hidden;
        double sumsq = 0.0;
        for (int j = 0; j < hidden; ++j) {
            double v = load(x, row + j, dtype);
            sumsq += v * v;
        }
        double inv = 1.0 / sqrt(sumsq / (double)hidden + (double)eps);
        if (inv_rms)
            inv_rms[t] = inv;
        for (int j = 0; j < hidden; ++j)
            store(out, row + j, dtype, load(x, row + j, dtype) * inv * load(weight, (size_t)j, dtype));
    }
}
