/*
 * qref.c -- CPU oracle for the quantized-weight matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow definition that the
 * CUDA library is checked against.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library and includes nothing from it.
 *
 * What it computes.  Sources: the page "CUDA 后端" (colibri-analysis 09),
 * section 1 "设备侧库 backend_cuda.cu": the device function `weight_at`
 * turns one stored element into its value (int4 code minus 8, int2 code minus
 * 2, the same meaning as the CPU kernel) and `quant_matmul` multiplies the
 * per-row scale; the page "第 8 章 · 02 CUDA/Metal/Vulkan 三后端", section 四,
 * header of qmatmul.comp: each output is the dot product of an input row with
 * a dequantized weight row, times that weight row's scale.  In symbols,
 *
 *     y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]
 *
 *   deq(f32, row, i) = ((float *)row)[i]
 *   deq(i8,  row, i) = row[i] read as a two's-complement byte
 *   deq(i4,  row, i) = ((row[i/2] >> 4*(i%2)) & 15) - 8     low nibble first
 *   deq(i2,  row, i) = ((row[i/4] >> 2*(i%4)) &  3) - 2     low bits first
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): nibble / bit order is low-first; a row of the host layout is
 * ceil(I*b/8) bytes and the unused high bits of its last byte are ignored; a
 * NULL scale vector means 1.0 (the CUDA tour applies the scale for quantized
 * tensors, the shader header applies it always; the two agree at scale 1).
 *
 * Every product is formed in double and summed in double in index order; the
 * result is rounded once to f32.  The error bound that goes with it is
 * bound[s,o] = |scale[o]| * sum_i |deq(W[o,i]) * x[s,i]|.
 *
 * Parallelism: OpenMP over (s, o) only; each inner sum is sequential.
 *
 * Parity: pinned.  The tests pin the code tables exhaustively, the bit order
 * by one-hot rows, the accumulation by hand-expanded worked examples and by
 * closed forms, and the scale by power-of-two invariance.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { QREF_F32 = 0, QREF_I8 = 1, QREF_I4 = 2, QREF_I2 = 3 };

/* Bytes of one row of the host layout: ceil(I * bits / 8). */
long qref_row_bytes(int fmt, long I)
{
    if (I < 0) return -1;
    switch (fmt) {
    case QREF_F32: return 4 * I;
    case QREF_I8:  return I;
    case QREF_I4:  return (I + 1) / 2;
    case QREF_I2:  return (I + 3) / 4;
    default:       return -1;
    }
}

/* The signed value a quantized code stands for; for f32 the stored float. */
double qref_weight(int fmt, const uint8_t *row, long i)
{
    switch (fmt) {
    case QREF_F32: {
        float f;
        memcpy(&f, row + 4 * i, sizeof f);
        return (double)f;
    }
    case QREF_I8: {
        int v = row[i];              /* two's complement, written out */
        if (v >= 128) v -= 256;
        return (double)v;
    }
    case QREF_I4: {
        int code = (row[i / 2] >> (4 * (i % 2))) & 0xF;
        return (double)(code - 8);
    }
    case QREF_I2: {
        int code = (row[i / 4] >> (2 * (i % 4))) & 0x3;
        return (double)(code - 2);
    }
    default:
        return NAN;
    }
}

/* Decodes one whole row into doubles (used by the exhaustive table tests). */
int qref_dequant_row(int fmt, long I, const uint8_t *row, double *out)
{
    if (qref_row_bytes(fmt, I) < 0) return -1;
    for (long i = 0; i < I; ++i) out[i] = qref_weight(fmt, row, i);
    return 0;
}

static int qref_threads = 0;   /* 0: OpenMP default */

void qref_set_threads(int n) { qref_threads = n; }

int qref_max_threads(void)
{
#ifdef _OPENMP
    return qref_threads > 0 ? qref_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * y[s*O + o]     = (float)(scale[o] * sum_i deq(W[o,i]) * x[s*I + i])
 * ydbl[s*O + o]  = the same before the final rounding (may be NULL)
 * bound[s*O + o] = |scale[o]| * sum_i |deq(W[o,i]) * x[s*I + i]| (may be NULL)
 *
 * codes: host layout, row-major [O, qref_row_bytes(fmt, I)] bytes.
 * scales: [O] floats or NULL (= 1.0).  x: [S, I] floats, row-major.
 * Returns 0, or -1 on a bad argument.
 */
int qref_matmul(int fmt, long O, long I, const uint8_t *codes, const float *scales,
                const float *x, long S, float *y, double *ydbl, double *bound)
{
    long rb = qref_row_bytes(fmt, I);
    if (rb < 0 || O < 0 || S < 0) return -1;
    if (O == 0 || S == 0) return 0;
    if (!codes || !x || !y) return -1;
    long n = S * O;
#ifdef _OPENMP
    int nt = qref_max_threads();
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (long so = 0; so < n; ++so) {
        long s = so / O, o = so % O;
        const uint8_t *row = codes + o * rb;
        const float *xs = x + s * I;
        double acc = 0.0, bnd = 0.0;
        for (long i = 0; i < I; ++i) {
            double t = qref_weight(fmt, row, i) * (double)xs[i];
            acc += t;
            bnd += fabs(t);
        }
        double sc = scales ? (double)scales[o] : 1.0;
        y[so] = (float)(sc * acc);
        if (ydbl) ydbl[so] = sc * acc;
        if (bound) bound[so] = fabs(sc) * bnd;
    }
    return 0;
}

/*
 * Group-wise scales.  The Vulkan tensor of the three-backends chapter (section
 * 三) carries a group size gs next to fmt; the pages say nothing more, so the
 * plain reading is one scale per row and group of gs consecutive columns:
 *     y[s,o] = sum_g gscales[o, g] * sum_{i in group g} deq(W[o,i]) * x[s,i]
 * groups g = 0 .. G-1, G = ceil(I / gs), the last one possibly short;
 * gscales is [O, G] row-major.  In double, one rounding at the end;
 * bound[s,o] = sum_i |gscales[o, i / gs] * deq * x|.  Returns 0 or -1.
 */
int qref_matmul_gs(int fmt, long O, long I, long gs, const uint8_t *codes, const float *gscales,
                   const float *x, long S, float *y, double *ydbl, double *bound)
{
    long rb = qref_row_bytes(fmt, I);
    if (rb < 0 || O < 0 || S < 0 || gs < 1) return -1;
    if (O == 0 || S == 0) return 0;
    if (!codes || !gscales || !x || !y) return -1;
    long G = (I + gs - 1) / gs;
    long n = S * O;
#ifdef _OPENMP
    int nt = qref_max_threads();
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (long so = 0; so < n; ++so) {
        long s = so / O, o = so % O;
        const uint8_t *wrow = codes + o * rb;
        const float *xrow = x + s * I;
        double total = 0.0, bnd = 0.0;
        for (long g = 0; g < G; ++g) {
            double acc = 0.0, gb = 0.0;
            long end = (g + 1) * gs < I ? (g + 1) * gs : I;
            for (long i = g * gs; i < end; ++i) {
                double p = qref_weight(fmt, wrow, i) * (double)xrow[i];
                acc += p;
                gb += fabs(p);
            }
            double sc = (double)gscales[o * G + g];
            total += sc * acc;
            bnd += fabs(sc) * gb;
        }
        y[so] = (float)total;
        if (ydbl) ydbl[so] = total;
        if (bound) bound[so] = bnd;
    }
    return 0;
}

/*
 * The fused gate/up pair (qmatmul_gate_up.comp in the three-backends chapter):
 * two matmuls of equal shape on the same input x.
 */
int qref_matmul_gate_up(int fmt, long O, long I,
                        const uint8_t *codes_g, const float *scales_g,
                        const uint8_t *codes_u, const float *scales_u,
                        const float *x, long S,
                        float *yg, double *bound_g, float *yu, double *bound_u)
{
    int rc = qref_matmul(fmt, O, I, codes_g, scales_g, x, S, yg, NULL, bound_g);
    if (rc) return rc;
    return qref_matmul(fmt, O, I, codes_u, scales_u, x, S, yu, NULL, bound_u);
}

/*
 * Expert glue between gate/up and down: h = silu(g) * u with the textbook
 * silu(z) = z / (1 + e^-z), in double.  The pages name the gated
 * up-projection but do not print the activation, so this is the plain reading.
 * h is returned both rounded to f32 (the input format of the next matmul) and
 * unrounded.
 */
void qref_silu_mul(const float *g, const float *u, long n, float *h, double *hdbl)
{
    for (long k = 0; k < n; ++k) {
        double z = (double)g[k];
        double v = z / (1.0 + exp(-z)) * (double)u[k];
        if (h) h[k] = (float)v;
        if (hdbl) hdbl[k] = v;
    }
}

/*
 * Layer glue kept on the device (colibri CUDA docs, "The GPU-resident
 * pipeline": rmsnorms and residual adds run on the GPU between the expert
 * loops).  The pages name the operation but do not print it; this is the
 * textbook RMSNorm, in double:
 *     h[s,d] = x[s,d] + r[s,d]           (r may be NULL: h = x)
 *     y[s,d] = h[s,d] * w[d] / sqrt(mean_d h[s,d]^2 + eps)
 * h is formed as an f32 sum (one rounding of the exact sum, which is what an
 * f32 addition gives) and normalized as stored; y is returned rounded to f32
 * and unrounded.  Returns 0, or -1 for a bad argument.
 */
int qref_rmsnorm(const float *x, const float *r, const float *w, long S, long D, double eps, float *h,
                 float *y, double *ydbl)
{
    if (S < 0 || D <= 0 || !x || !w || eps < 0) return -1;
    for (long s = 0; s < S; ++s) {
        double ss = 0.0;
        for (long d = 0; d < D; ++d) {
            float hv = r ? (float)((double)x[s * D + d] + (double)r[s * D + d]) : x[s * D + d];
            if (h) h[s * D + d] = hv;
            ss += (double)hv * (double)hv;
        }
        double inv = 1.0 / sqrt(ss / (double)D + eps);
        for (long d = 0; d < D; ++d) {
            float hv = r ? (float)((double)x[s * D + d] + (double)r[s * D + d]) : x[s * D + d];
            double v = (double)hv * (double)w[d] * inv;
            if (y) y[s * D + d] = (float)v;
            if (ydbl) ydbl[s * D + d] = v;
        }
    }
    return 0;
}

/*
 * Round an f32 to the nearest bfloat16 (8 significant bits, f32's exponent
 * range), ties to the even significand, returned as an f32.  Written from the
 * definition: take the two bf16 neighbours of v (truncation toward zero and
 * one unit further away), keep the nearer one, and on a tie the one whose last
 * kept bit is 0.  Finite inputs only.
 */
float qref_round_bf16(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    uint32_t lo_bits = u & 0xFFFF0000u;                 /* toward zero */
    uint32_t hi_bits = lo_bits + 0x00010000u;           /* next bf16 away from zero */
    float lo, hi;
    memcpy(&lo, &lo_bits, sizeof lo);
    memcpy(&hi, &hi_bits, sizeof hi);
    double dlo = fabs((double)v - (double)lo);
    double dhi = fabs((double)hi - (double)v);
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return ((lo_bits >> 16) & 1u) ? hi : lo;           /* tie: even significand */
}

/*
 * The tensor-core prefill path rounds x to bf16 before the contraction; this
 * is qref_matmul applied to the bf16-rounded x.  It is a diagnostic: the
 * contract compares the tensor-core path with the unrounded qref_matmul.
 */
int qref_matmul_bf16x(int fmt, long O, long I, const uint8_t *codes, const float *scales,
                      const float *x, long S, float *xr_scratch, float *y, double *ydbl,
                      double *bound)
{
    if (S < 0 || I < 0) return -1;
    for (long k = 0; k < S * I; ++k) xr_scratch[k] = qref_round_bf16(x[k]);
    return qref_matmul(fmt, O, I, codes, scales, xr_scratch, S, y, ydbl, bound);
}

/*
 * MLA decode attention with weight absorption (page "第 8 章 · 02
 * CUDA/Metal/Vulkan 三后端", section 四, the header of attention_absorb.comp,
 * the Vulkan twin of coli_cuda_attention_absorb).  Per new token s and head h,
 * four steps in the pages' order:
 *
 *   qabs[i]  = sum_d q_nope[s,h,d] * Wk[h,d,i]                  (absorb)
 *   score_t  = (qabs . L[t] + q_rope[s,h] . Rr[t]) * scale      t in [st0, T-S+s]
 *   p        = softmax over that window of score
 *   clat[i]  = sum_t p_t * L[t,i]                               (latent context)
 *   ctx[s,h,v] = sum_i clat[i] * Wv[h,v,i]                      (value rows)
 *
 * Wkv_b is one [H*(Dn+Dv), K] weight tensor (host layout of fmt): head h's
 * key rows are h*(Dn+Dv) + d for d < Dn, its value rows follow at
 * h*(Dn+Dv) + Dn + v.  The weight value is scale * deq(code), with per-row
 * scales [rows] as in qref_matmul (gs = 0; NULL scales mean 1.0), or
 * group-wise scales [rows, ceil(K / gs)] as in qref_matmul_gs (gs >= 1).  L is the latent cache [T, K],
 * Rr the rope cache [T, R], both f32; the S new tokens sit at positions
 * T-S .. T-1 and token s sees positions st0 .. T-S+s (causal).  q_nope is
 * [S, H, Dn], q_rope [S, H, R], ctx [S, H, Dv].  Everything is in double,
 * the softmax from its maximum; ctx is rounded once to f32.
 *
 * Error bound per output, from the f32 arithmetic of an implementation that
 * rounds each step (relative error eps per accumulated term):
 *     bound[s,h,v] = (1 + A) * sum_i |Wv[h,v,i]| * sum_t p_t |L[t,i]|
 *     A = max_t |scale| * (sum_i QA_i |L[t,i]| + sum_j |q_rope_j Rr[t,j]|),
 *     QA_i = sum_d |q_nope_d Wk[h,d,i]|
 * (a score error of eps * A moves p_t by at most 2 eps A p_t, and the value
 * step adds its own eps).  Returns 0, -1 for a bad argument (S < 1,
 * T < S, st0 < 0 or st0 > T - S: every window must hold a position), or -2
 * when host memory for the per-row scratch vectors cannot be had (the
 * outputs are then incomplete and must not be used).
 */
/* Scale of element i of weight row `row` (see qref_mla_absorb). */
static double mla_scale(const float *scales, long gs, long G, long row, long i)
{
    if (!scales) return 1.0;
    return gs ? (double)scales[row * G + i / gs] : (double)scales[row];
}

int qref_mla_absorb(int fmt, long H, long Dn, long Dv, long K, long R,
                    const uint8_t *codes, const float *scales, long gs,
                    const float *q_nope, const float *q_rope,
                    const float *lat, const float *rope,
                    long T, long st0, double scale, long S,
                    float *ctx, double *ctxdbl, double *bound)
{
    long rb = qref_row_bytes(fmt, K);
    if (rb < 0 || H < 1 || Dn < 1 || Dv < 1 || K < 1 || R < 0 || S < 1 || T < S || st0 < 0 || st0 > T - S)
        return -1;
    if (!codes || !q_nope || (R > 0 && (!q_rope || !rope)) || !lat || !ctx || gs < 0 || (gs && !scales)) return -1;
    long HS = H * S;
    long G = gs ? (K + gs - 1) / gs : 1;
    int oom = 0;                                       /* set by any row whose scratch malloc failed */
#ifdef _OPENMP
    int nt = qref_max_threads();
#pragma omp parallel for schedule(dynamic) num_threads(nt)
#endif
    for (long hs = 0; hs < HS; ++hs) {
        long s = hs / H, h = hs % H;
        long key0 = h * (Dn + Dv), val0 = key0 + Dn;
        long first = st0, last = T - S + s;            /* the window token s sees */
        long nwin = last - first + 1;
        double *qabs = (double *)malloc(sizeof(double) * (size_t)K);
        double *qa = (double *)malloc(sizeof(double) * (size_t)K);
        double *clat = (double *)malloc(sizeof(double) * (size_t)K);
        double *cabs = (double *)malloc(sizeof(double) * (size_t)K);
        double *score = (double *)malloc(sizeof(double) * (size_t)nwin);
        double *sabs = (double *)malloc(sizeof(double) * (size_t)nwin);
        if (!qabs || !qa || !clat || !cabs || !score || !sabs) {
            free(qabs); free(qa); free(clat); free(cabs); free(score); free(sabs);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            oom = 1;
            continue;
        }
        const float *qn = q_nope + (s * H + h) * Dn;
        const float *qr = R > 0 ? q_rope + (s * H + h) * R : NULL;

        /* absorb: qabs = sum over the head's key rows of q_nope[d] * row d */
        for (long i = 0; i < K; ++i) qabs[i] = qa[i] = 0.0;
        for (long d = 0; d < Dn; ++d) {
            const uint8_t *krow = codes + (key0 + d) * rb;
            for (long i = 0; i < K; ++i) {
                double kw = mla_scale(scales, gs, G, key0 + d, i) * qref_weight(fmt, krow, i);
                qabs[i] += (double)qn[d] * kw;
                qa[i] += fabs((double)qn[d] * kw);
            }
        }
        /* scores over the window, then the softmax from their maximum */
        double smax = -HUGE_VAL, amax = 0.0;
        for (long w = 0; w < nwin; ++w) {
            const float *lt = lat + (first + w) * K;
            double dot = 0.0, a = 0.0;
            for (long i = 0; i < K; ++i) {
                dot += qabs[i] * (double)lt[i];
                a += qa[i] * fabs((double)lt[i]);
            }
            for (long j = 0; j < R; ++j) {
                double t = (double)qr[j] * (double)rope[(first + w) * R + j];
                dot += t;
                a += fabs(t);
            }
            score[w] = dot * scale;
            sabs[w] = a * fabs(scale);
            if (score[w] > smax) smax = score[w];
            if (sabs[w] > amax) amax = sabs[w];
        }
        double z = 0.0;
        for (long w = 0; w < nwin; ++w) {
            score[w] = exp(score[w] - smax);
            z += score[w];
        }
        /* latent context and its magnitude */
        for (long i = 0; i < K; ++i) clat[i] = cabs[i] = 0.0;
        for (long w = 0; w < nwin; ++w) {
            double p = score[w] / z;
            const float *lt = lat + (first + w) * K;
            for (long i = 0; i < K; ++i) {
                clat[i] += p * (double)lt[i];
                cabs[i] += p * fabs((double)lt[i]);
            }
        }
        /* value rows */
        for (long v = 0; v < Dv; ++v) {
            const uint8_t *vrow = codes + (val0 + v) * rb;
            double acc = 0.0, b = 0.0;
            for (long i = 0; i < K; ++i) {
                double vw = mla_scale(scales, gs, G, val0 + v, i) * qref_weight(fmt, vrow, i);
                acc += clat[i] * vw;
                b += fabs(vw) * cabs[i];
            }
            long out = (s * H + h) * Dv + v;
            ctx[out] = (float)acc;
            if (ctxdbl) ctxdbl[out] = acc;
            if (bound) bound[out] = (1.0 + amax) * b;
        }
        free(qabs); free(qa); free(clat); free(cabs); free(score); free(sabs);
    }
    return oom ? -2 : 0;
}
