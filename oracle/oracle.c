/*
 * CPU oracle for the GPUOS micro-op library -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded definitions of what each micro-op computes,
 * written from "GPUOS: A GPU Operating System Primitive for Transparent
 * Operation Fusion" (§3 Q2, "Operator library": element-wise add, mul, ReLU,
 * GELU, softmax, LayerNorm; vector-matrix products; SDPA and rotary
 * embeddings; KV-cache update; small sum/max/min reductions). The page names
 * the ops but gives no formulas; each function below is the textbook
 * definition of the op, stated in its comment. Nothing here is blocked,
 * fused or reordered: loops run in index order and accumulate in double.
 *
 * Only the test-suite, the package's smoke check and the benchmark's CPU
 * baseline load this file. It shares no code, header or constant with the
 * CUDA path.
 *
 * Conventions
 *   - bf16 operands arrive as raw uint16 bit patterns and are widened exactly.
 *   - Every op writes the exact (double) result into a caller array; the
 *     caller rounds it to the output type with orc_store_* (round to nearest,
 *     ties to even), so the unrounded value stays available for tolerance
 *     checks.
 *   - dtype codes: 0 = fp32, 1 = bf16.
 *
 * Parity pins (closed forms, special cases, brute force) live in the
 * test-suite; every function here is pinned by at least one of them.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* ---- number formats -------------------------------------------------- */

/* bf16 bits -> double, exact: bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bf16 bits, one rounding to nearest, ties to even.
 * bf16 keeps 8 significant bits and binary32's exponent range: normal
 * numbers in [2^(e-1), 2^e) are quantised to 2^(e-8); below 2^-126 the
 * quantum stays 2^-133 (subnormals). Results of magnitude >= 2^128 are
 * infinite. */
uint16_t orc_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double ax = fabs(x);
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (ax == 0.0)
        return sign;
    int e;
    frexp(ax, &e); /* ax = f * 2^e, f in [0.5, 1) */
    int q = e - 8;
    if (q < -133)
        q = -133;
    double r = ldexp(nearbyint(ldexp(ax, -q)), q); /* default mode: ties-to-even */
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

static double load(int dtype, const void *p, long i)
{
    if (dtype == ORC_F32)
        return (double)((const float *)p)[i];
    return orc_bf16_to_double(((const uint16_t *)p)[i]);
}

/* Round n exact results to the output type. fp32 uses C's conversion,
 * which rounds to nearest-even under the default rounding mode. */
void orc_store(int dtype, const double *x, void *dst, long n)
{
    for (long i = 0; i < n; i++) {
        if (dtype == ORC_F32)
            ((float *)dst)[i] = (float)x[i];
        else
            ((uint16_t *)dst)[i] = orc_bf16_from_double(x[i]);
    }
}

/* ---- element-wise ------------------------------------------------------ */

/* c_i = a_i + b_i. The sum of two binary32 (or bf16) values is computed in
 * double; rounding it once to the output type gives the IEEE result of the
 * operation in that type (double has more than 2p+2 bits, so no double-
 * rounding error can occur). */
void orc_add(int dtype, const void *a, const void *b, double *out, long n)
{
    for (long i = 0; i < n; i++)
        out[i] = load(dtype, a, i) + load(dtype, b, i);
}

/* c_i = a_i * b_i (product of two binary32 values is exact in double). */
void orc_mul(int dtype, const void *a, const void *b, double *out, long n)
{
    for (long i = 0; i < n; i++)
        out[i] = load(dtype, a, i) * load(dtype, b, i);
}

/* c_i = max(a_i, 0); non-positive inputs give +0. */
void orc_relu(int dtype, const void *a, double *out, long n)
{
    for (long i = 0; i < n; i++) {
        double x = load(dtype, a, i);
        out[i] = x > 0.0 ? x : 0.0;
    }
}

/* GELU, exact form: c = x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), evaluated
 * as 0.5 x erfc(-x / sqrt 2) (the identity 1 + erf(z) = erfc(-z)), which
 * keeps full relative accuracy for x < 0, where 1 + erf cancels to 0 in
 * double below x = -8.3. */
void orc_gelu(int dtype, const void *a, double *out, long n)
{
    for (long i = 0; i < n; i++) {
        double x = load(dtype, a, i);
        out[i] = 0.5 * x * erfc(-x / sqrt(2.0));
    }
}

/* ---- row ops on x[R][H] (bf16) --------------------------------------- */

/* y_j = exp(x_j - m) / sum_k exp(x_k - m), m = max_j x_j, per row. */
void orc_softmax(const uint16_t *x, long R, long H, double *out)
{
    for (long r = 0; r < R; r++) {
        const uint16_t *row = x + r * H;
        double m = -INFINITY;
        for (long j = 0; j < H; j++) {
            double v = orc_bf16_to_double(row[j]);
            if (v > m)
                m = v;
        }
        double s = 0.0;
        for (long j = 0; j < H; j++)
            s += exp(orc_bf16_to_double(row[j]) - m);
        for (long j = 0; j < H; j++)
            out[r * H + j] = exp(orc_bf16_to_double(row[j]) - m) / s;
    }
}

/* LayerNorm with the biased variance:
 *   mu = (1/H) sum x,  var = (1/H) sum (x - mu)^2,
 *   y = (x - mu) / sqrt(var + eps) * gamma + beta. */
void orc_layernorm(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta, long R, long H,
                   double eps, double *out)
{
    for (long r = 0; r < R; r++) {
        const uint16_t *row = x + r * H;
        double mu = 0.0;
        for (long j = 0; j < H; j++)
            mu += orc_bf16_to_double(row[j]);
        mu /= (double)H;
        double var = 0.0;
        for (long j = 0; j < H; j++) {
            double d = orc_bf16_to_double(row[j]) - mu;
            var += d * d;
        }
        var /= (double)H;
        double rstd = 1.0 / sqrt(var + eps);
        for (long j = 0; j < H; j++) {
            double xn = (orc_bf16_to_double(row[j]) - mu) * rstd;
            out[r * H + j] = xn * orc_bf16_to_double(gamma[j]) + orc_bf16_to_double(beta[j]);
        }
    }
}

/* Row reductions. kind: 0 = sum, 1 = max, 2 = min. */
void orc_rowreduce(int kind, const uint16_t *x, long R, long H, double *out)
{
    for (long r = 0; r < R; r++) {
        const uint16_t *row = x + r * H;
        double acc = kind == 0 ? 0.0 : orc_bf16_to_double(row[0]);
        for (long j = (kind == 0 ? 0 : 1); j < H; j++) {
            double v = orc_bf16_to_double(row[j]);
            if (kind == 0)
                acc += v;
            else if (kind == 1)
                acc = v > acc ? v : acc;
            else
                acc = v < acc ? v : acc;
        }
        out[r] = acc;
    }
}

/* ---- attention-side ops ------------------------------------------------ */

/* Rotary position embedding, half-split pairing. For every row of q and k
 * of request b (layout [B][H][D]) and i < D/2, with p = lens[b] - 1 and
 * phi = p * theta^(-2i/D):
 *   x_i       <- x_i cos phi - x_{i+D/2} sin phi
 *   x_{i+D/2} <- x_{i+D/2} cos phi + x_i sin phi
 * Exact results go to qo / ko (same layout). Returns -1 if a position is
 * negative. */
int orc_rope(const uint16_t *q, const uint16_t *k, const int32_t *lens, long B, long H, long D,
             double theta, double *qo, double *ko)
{
    long half = D / 2;
    for (long b = 0; b < B; b++) {
        long p = (long)lens[b] - 1;
        if (p < 0)
            return -1;
        for (long h = 0; h < H; h++) {
            for (int which = 0; which < 2; which++) {
                const uint16_t *x = (which == 0 ? q : k) + (b * H + h) * D;
                double *y = (which == 0 ? qo : ko) + (b * H + h) * D;
                for (long i = 0; i < half; i++) {
                    double phi = (double)p * pow(theta, -2.0 * (double)i / (double)D);
                    double x0 = orc_bf16_to_double(x[i]);
                    double x1 = orc_bf16_to_double(x[i + half]);
                    y[i] = x0 * cos(phi) - x1 * sin(phi);
                    y[i + half] = x1 * cos(phi) + x0 * sin(phi);
                }
            }
        }
    }
    return 0;
}

/* KV-cache slot update: Kc[b][h][lens[b]-1][:] = k[b][h][:] and the same for
 * V; caches are [B][H][Lcap][D]. A plain element copy. Returns -1 if a
 * position falls outside the cache. */
int orc_kv_write(const uint16_t *k, const uint16_t *v, const int32_t *lens, long B, long H, long D,
                 long Lcap, uint16_t *Kc, uint16_t *Vc)
{
    for (long b = 0; b < B; b++) {
        long p = (long)lens[b] - 1;
        if (p < 0 || p >= Lcap)
            return -1;
        for (long h = 0; h < H; h++)
            for (long d = 0; d < D; d++) {
                Kc[((b * H + h) * Lcap + p) * D + d] = k[(b * H + h) * D + d];
                Vc[((b * H + h) * Lcap + p) * D + d] = v[(b * H + h) * D + d];
            }
    }
    return 0;
}

/* Single-query decode attention per (b, h) over the first L = lens[b] cache
 * rows: s_t = scale * (q . K_t), p = softmax(s), o = sum_t p_t V_t.
 * Returns -1 if a length is outside [1, Lcap]. */
int orc_sdpa(const uint16_t *q, const uint16_t *Kc, const uint16_t *Vc, const int32_t *lens, long B,
             long H, long D, long Lcap, double scale, double *out)
{
    for (long b = 0; b < B; b++) {
        long L = lens[b];
        if (L < 1 || L > Lcap)
            return -1;
        for (long h = 0; h < H; h++) {
            const uint16_t *qv = q + (b * H + h) * D;
            const uint16_t *K = Kc + (b * H + h) * Lcap * D;
            const uint16_t *V = Vc + (b * H + h) * Lcap * D;
            double m = -INFINITY;
            for (long t = 0; t < L; t++) {
                double s = 0.0;
                for (long d = 0; d < D; d++)
                    s += orc_bf16_to_double(qv[d]) * orc_bf16_to_double(K[t * D + d]);
                s *= scale;
                if (s > m)
                    m = s;
            }
            double den = 0.0;
            double *o = out + (b * H + h) * D;
            for (long d = 0; d < D; d++)
                o[d] = 0.0;
            for (long t = 0; t < L; t++) {
                double s = 0.0;
                for (long d = 0; d < D; d++)
                    s += orc_bf16_to_double(qv[d]) * orc_bf16_to_double(K[t * D + d]);
                double w = exp(s * scale - m);
                den += w;
                for (long d = 0; d < D; d++)
                    o[d] += w * orc_bf16_to_double(V[t * D + d]);
            }
            for (long d = 0; d < D; d++)
                o[d] /= den;
        }
    }
    return 0;
}

/* Vector-matrix product y_n = sum_k x_k W[k][n], W row-major [K][N]. */
void orc_vecmat(const uint16_t *x, const uint16_t *W, long K, long N, double *out)
{
    for (long n = 0; n < N; n++) {
        double s = 0.0;
        for (long k = 0; k < K; k++)
            s += orc_bf16_to_double(x[k]) * orc_bf16_to_double(W[k * N + n]);
        out[n] = s;
    }
}
