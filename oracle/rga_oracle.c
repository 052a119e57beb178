/*
 * Plain fp64 CPU oracle for the fused attention forward of the
 * TRT_Attention / TRT_QuantizedAttention custom-op schemas.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant with
 * the CUDA library.
 *
 * It is written as the plain definition, with no tiling, no online softmax
 * and no reordering: for every query row it builds the set of attendable
 * keys, the scores, the normalised probabilities and the weighted sum of V,
 * in that order, in double precision.
 *
 * Sources (page titles and sections):
 *   "TensorRT Custom Operator Schemas", TRT_Attention:
 *     - tensor format notation: padded_bhnd [B,H,N,D], packed_nhd [T,H,D];
 *     - attributes causal_kind, TRT_normalization_op ("softmax" | "none");
 *     - input attn_mask: bool true = may attend, other dtypes added to the
 *       BMM1 output;
 *     - inputs query_lengths ([B+1] cumulative), kv_lengths ([B+1]
 *       cumulative when packed, [B] per batch when padded);
 *     - output Y: same shape, form and dtype as Q.
 *   "TensorRT Custom Operator Schemas", TRT_QuantizedAttention:
 *     - normalization_quantize_to_type (fp8 default, or int8) and
 *       normalization_quantize_scale: Q/DQ between normalisation and BMM2.
 *   "TensorRT Plugins Guide", AttentionPlugin: MHA and GQA (fewer KV heads
 *     than query heads).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *   causal upper_left:  key j is allowed for query i iff j <= i.
 *   causal lower_right: iff j <= i + kv_len - q_len (per sequence).
 *   GQA: query head h reads KV head h / (Hq / Hkv).
 *   mask: rank-4 [mB, mH, mQ, mK], each dim 1 (broadcast) or full, indexed
 *     by within-sequence positions (i, j).
 *   rows with no attendable key (or whose scores are all -inf) give 0.
 *   'none': P = s on attendable pairs, 0 elsewhere.
 *   Q/DQ: x = p / s, q = saturate(round-half-even(x)), p' = q * s, with
 *     E4M3FN (bias 7, max 448, subnormals, no inf) or int8 [-128, 127].
 *   padded query rows at or beyond q_len are never written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG 1
#define ORA_ERR_LENGTHS 4

enum { ORA_PADDED = 0, ORA_PACKED = 1 };
enum { ORA_CAUSAL_NONE = 0, ORA_CAUSAL_UPPER_LEFT = 1, ORA_CAUSAL_LOWER_RIGHT = 2 };
enum { ORA_SOFTMAX = 0, ORA_NONE = 1 };
enum { ORA_Q_OFF = -1, ORA_Q_FP8 = 0, ORA_Q_INT8 = 1 };

/* ---------------------------------------------------------------------------
 * Quantisers (TRT_QuantizedAttention, normalization_quantize_to_type).
 * ------------------------------------------------------------------------- */

/* Decode one OCP E4M3FN byte: sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal; S.1111.111 is NaN; there is no infinity. */
double rga_oracle_e4m3_decode(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round x to the nearest E4M3FN value, ties to even mantissa, saturating to
 * +-448 (the largest finite E4M3FN magnitude).  NaN stays NaN. */
double rga_oracle_e4m3_round(double x)
{
    double ax, quantum, r;
    int ex;
    if (isnan(x))
        return x;
    ax = fabs(x);
    if (ax >= 448.0)
        return x < 0 ? -448.0 : 448.0;
    if (ax < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9); /* subnormal spacing: 2^-6 / 8 */
    } else {
        frexp(ax, &ex);           /* ax = f * 2^ex, f in [0.5, 1) */
        quantum = ldexp(1.0, (ex - 1) - 3);
    }
    r = nearbyint(ax / quantum) * quantum; /* default mode: half to even */
    if (r > 448.0)
        r = 448.0;
    return x < 0 ? -r : r;
}

/* Encode to the E4M3FN byte (used only by the code round-trip pin). */
int rga_oracle_e4m3_encode(double x)
{
    double r = rga_oracle_e4m3_round(x);
    int code;
    if (isnan(r))
        return 0x7f;
    for (code = 0; code < 127; ++code)
        if (rga_oracle_e4m3_decode(code) == fabs(r))
            return (r < 0 || (r == 0 && signbit(r))) ? (code | 0x80) : code;
    return -1;
}

/* FP8 KV cache ("TensorRT Plugins Guide", AttentionPlugin: kv_cache_type
 * FP8): the cache holds E4M3FN codes and one scale per tensor; the key or
 * value element is the decoded code times the scale.  out[i] for i < n. */
void rga_oracle_e4m3_dequant(const unsigned char *codes, long n, double scale, double *out)
{
    long i;
    for (i = 0; i < n; ++i)
        out[i] = rga_oracle_e4m3_decode(codes[i]) * scale;
}

/* int8 QuantizeLinear with zero-point 0: round half to even, clamp. */
double rga_oracle_int8_round(double x)
{
    double r;
    if (isnan(x))
        return x;
    r = nearbyint(x);
    if (r > 127.0)
        r = 127.0;
    if (r < -128.0)
        r = -128.0;
    return r;
}

/* Q then DQ of one probability with scale s. */
static double qdq(double p, int quant, double s)
{
    double x = p / s;
    if (quant == ORA_Q_FP8)
        return rga_oracle_e4m3_round(x) * s;
    return rga_oracle_int8_round(x) * s;
}

/* Where floating point decides a quantised code, a value x = |p / s| within
 * eps * x of a rounding midpoint may round either way in another correct
 * evaluation (another precision or order).  The window is relative to x:
 * after softmax, x is an exponential of the scores, so an error in the
 * scores moves it by a relative amount.  (Under 'none', x is the score
 * itself, and near a cancellation in the dot product the error of another
 * evaluation is larger than eps * x; such codes sit next to zero, where the
 * first midpoint lies far away.)  Returns the change of the dequantised
 * value if such a code flipped (one quantisation step times s), or 0 when
 * the decision is clear. */
static double qdq_ambiguity(double p, int quant, double s, double eps)
{
    double x = fabs(p / s), step, t;
    int ex;
    if (eps <= 0.0 || x == 0.0)
        return 0.0;
    if (quant == ORA_Q_FP8) {
        if (x >= 448.0)
            return 0.0;                   /* saturated either way */
        if (x < ldexp(1.0, -6)) {
            step = ldexp(1.0, -9);
        } else {
            frexp(x, &ex);
            step = ldexp(1.0, (ex - 1) - 3);
        }
    } else {
        if (x >= 127.5)
            return 0.0;
        step = 1.0;
    }
    t = x / step - floor(x / step);      /* position inside the step */
    if (fabs(t - 0.5) * step <= eps * x)
        return step * s;
    return 0.0;
}

/* ---------------------------------------------------------------------------
 * Problem description shared by the worker threads.
 * ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v;
    double *y;
    double *amb;                /* optional: per-element Q/DQ ambiguity bound */
    double amb_eps;
    int q_form, kv_form, B, Hq, Hkv, D, q_seq, kv_seq;
    const int32_t *query_lengths, *kv_lengths;
    const double *mask_add;     /* additive mask, or NULL */
    const uint8_t *mask_bool;   /* bool mask, or NULL */
    int64_t md[4];              /* mask dims [mB, mH, mQ, mK] */
    double scale;
    int causal, norm, quant;
    double quant_scale;
    /* per-batch resolved offsets and lengths */
    int64_t *q_off, *q_len, *kv_off, *kv_len;
    /* work distribution */
    int next_unit;
    pthread_mutex_t lock;
} ora_problem;

/* Element offset of Q[b, h, i, 0] (or of Y, same layout). */
static int64_t q_index(const ora_problem *P, int b, int h, int64_t i)
{
    if (P->q_form == ORA_PACKED)
        return ((P->q_off[b] + i) * P->Hq + h) * (int64_t)P->D;
    return (((int64_t)b * P->Hq + h) * P->q_seq + i) * (int64_t)P->D;
}

/* Element offset of K[b, g, j, 0] (or of V, same layout). */
static int64_t kv_index(const ora_problem *P, int b, int g, int64_t j)
{
    if (P->kv_form == ORA_PACKED)
        return ((P->kv_off[b] + j) * P->Hkv + g) * (int64_t)P->D;
    return (((int64_t)b * P->Hkv + g) * P->kv_seq + j) * (int64_t)P->D;
}

/* Flat index of the mask element for (b, h, i, j) under broadcast. */
static int64_t mask_index(const ora_problem *P, int b, int h, int64_t i, int64_t j)
{
    int64_t ib = P->md[0] == 1 ? 0 : b;
    int64_t ih = P->md[1] == 1 ? 0 : h;
    int64_t iq = P->md[2] == 1 ? 0 : i;
    int64_t ik = P->md[3] == 1 ? 0 : j;
    return ((ib * P->md[1] + ih) * P->md[2] + iq) * P->md[3] + ik;
}

static int causal_allows(const ora_problem *P, int b, int64_t i, int64_t j)
{
    if (P->causal == ORA_CAUSAL_UPPER_LEFT)
        return j <= i;
    if (P->causal == ORA_CAUSAL_LOWER_RIGHT)
        return j <= i + P->kv_len[b] - P->q_len[b];
    return 1;
}

/* One query row: the plain definition, written out. */
static void attend_row(const ora_problem *P, int b, int h, int64_t i,
                       double *s, unsigned char *allowed)
{
    const int G = P->Hq / P->Hkv;
    const int g = h / G;
    const int64_t L = P->kv_len[b];
    const double *qrow = P->q + q_index(P, b, h, i);
    double *yrow = P->y + q_index(P, b, h, i);
    double m = -INFINITY, l = 0.0;
    int64_t j;
    int d, any = 0;

    /* scores s_j = scale * <q_i, k_j> + additive mask, on the allowed set */
    for (j = 0; j < L; ++j) {
        const double *krow = P->k + kv_index(P, b, g, j);
        double dot = 0.0;
        allowed[j] = (unsigned char)causal_allows(P, b, i, j);
        if (P->mask_bool && !P->mask_bool[mask_index(P, b, h, i, j)])
            allowed[j] = 0;
        if (!allowed[j]) {
            s[j] = 0.0;
            continue;
        }
        for (d = 0; d < P->D; ++d)
            dot += qrow[d] * krow[d];
        s[j] = P->scale * dot;
        if (P->mask_add)
            s[j] += P->mask_add[mask_index(P, b, h, i, j)];
        any = 1;
    }

    for (d = 0; d < P->D; ++d)
        yrow[d] = 0.0;
    if (P->amb)
        for (d = 0; d < P->D; ++d)
            P->amb[q_index(P, b, h, i) + d] = 0.0;
    if (!any)
        return; /* no attendable key: the row is zero */

    if (P->norm == ORA_SOFTMAX) {
        for (j = 0; j < L; ++j)
            if (allowed[j] && s[j] > m)
                m = s[j];
        if (m == -INFINITY)
            return; /* every score is -inf: the row is zero */
        for (j = 0; j < L; ++j)
            if (allowed[j])
                l += exp(s[j] - m);
        for (j = 0; j < L; ++j)
            s[j] = allowed[j] ? exp(s[j] - m) / l : 0.0;
    } else {
        for (j = 0; j < L; ++j)
            if (!allowed[j])
                s[j] = 0.0;
    }

    if (P->quant != ORA_Q_OFF)
        for (j = 0; j < L; ++j) {
            if (!allowed[j])
                continue;
            if (P->amb) {
                double a = qdq_ambiguity(s[j], P->quant, P->quant_scale, P->amb_eps);
                if (a != 0.0) {
                    const double *vrow = P->v + kv_index(P, b, g, j);
                    double *arow = P->amb + q_index(P, b, h, i);
                    for (d = 0; d < P->D; ++d)
                        arow[d] += a * fabs(vrow[d]);
                }
            }
            s[j] = qdq(s[j], P->quant, P->quant_scale);
        }

    for (j = 0; j < L; ++j) {
        const double *vrow;
        if (!allowed[j])
            continue;
        vrow = P->v + kv_index(P, b, g, j);
        for (d = 0; d < P->D; ++d)
            yrow[d] += s[j] * vrow[d];
    }
}

static void *worker(void *arg)
{
    ora_problem *P = (ora_problem *)arg;
    int64_t maxkv = 1, i;
    int b, u;
    double *s;
    unsigned char *allowed;
    for (b = 0; b < P->B; ++b)
        if (P->kv_len[b] > maxkv)
            maxkv = P->kv_len[b];
    s = (double *)malloc(sizeof(double) * maxkv);
    allowed = (unsigned char *)malloc(maxkv);
    for (;;) {
        pthread_mutex_lock(&P->lock);
        u = P->next_unit++;
        pthread_mutex_unlock(&P->lock);
        if (u >= P->B * P->Hq)
            break;
        b = u / P->Hq;
        for (i = 0; i < P->q_len[b]; ++i)
            attend_row(P, b, u % P->Hq, i, s, allowed);
    }
    free(s);
    free(allowed);
    return NULL;
}

/* ---------------------------------------------------------------------------
 * Entry point.  All pointers are host pointers; Q/K/V/Y are doubles holding
 * the stored (fp16/bf16) input values exactly.  mask_dims gives the mask
 * right-aligned to rank 4 (missing leading dims are 1).  quant is -1 (off),
 * 0 (fp8 E4M3FN) or 1 (int8).  Returns 0, 1 (bad argument) or 4 (bad
 * lengths).  Rows that are not valid query rows are left as they were.
 * amb (optional, shaped like y): for the quantised op, the sum over the
 * row's codes that lie within relative distance amb_eps of a rounding
 * midpoint of (one quantisation step * s * |v|): how far another correct
 * evaluation order may move each output element.
 * ------------------------------------------------------------------------- */
int rga_oracle_attention(const double *q, const double *k, const double *v,
                         double *y, int q_form, int kv_form, int B, int Hq,
                         int Hkv, int D, int q_seq, int kv_seq,
                         const int32_t *query_lengths,
                         const int32_t *kv_lengths, const double *mask_add,
                         const uint8_t *mask_bool, const int64_t *mask_dims,
                         double scale, int causal, int norm, int quant,
                         double quant_scale, int nthreads, double *amb,
                         double amb_eps)
{
    ora_problem P;
    pthread_t *th;
    int b, t, rc = ORA_OK;

    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return ORA_ERR_ARG;
    if (q_form == ORA_PACKED && !query_lengths)
        return ORA_ERR_ARG;
    if (kv_form == ORA_PACKED && !kv_lengths)
        return ORA_ERR_ARG;
    if (mask_add && mask_bool)
        return ORA_ERR_ARG;

    memset(&P, 0, sizeof(P));
    P.q = q; P.k = k; P.v = v; P.y = y;
    P.q_form = q_form; P.kv_form = kv_form;
    P.B = B; P.Hq = Hq; P.Hkv = Hkv; P.D = D;
    P.q_seq = q_seq; P.kv_seq = kv_seq;
    P.query_lengths = query_lengths; P.kv_lengths = kv_lengths;
    P.mask_add = mask_add; P.mask_bool = mask_bool;
    for (t = 0; t < 4; ++t)
        P.md[t] = (mask_add || mask_bool) ? mask_dims[t] : 1;
    P.scale = scale; P.causal = causal; P.norm = norm;
    P.quant = quant; P.quant_scale = quant_scale;
    P.amb = amb; P.amb_eps = amb_eps;
    P.q_off = (int64_t *)calloc(B + 1, sizeof(int64_t));
    P.q_len = (int64_t *)calloc(B + 1, sizeof(int64_t));
    P.kv_off = (int64_t *)calloc(B + 1, sizeof(int64_t));
    P.kv_len = (int64_t *)calloc(B + 1, sizeof(int64_t));

    /* Resolve per-batch offsets and lengths from the two length inputs. */
    for (b = 0; b < B; ++b) {
        if (q_form == ORA_PACKED) {
            P.q_off[b] = query_lengths[b];
            P.q_len[b] = (int64_t)query_lengths[b + 1] - query_lengths[b];
            if (query_lengths[0] != 0 || P.q_len[b] < 0 || query_lengths[b + 1] > q_seq)
                rc = ORA_ERR_LENGTHS;
        } else {
            P.q_len[b] = query_lengths
                ? (int64_t)query_lengths[b + 1] - query_lengths[b] : q_seq;
            if (P.q_len[b] < 0 || P.q_len[b] > q_seq)
                rc = ORA_ERR_LENGTHS;
        }
        if (kv_form == ORA_PACKED) {
            P.kv_off[b] = kv_lengths[b];
            P.kv_len[b] = (int64_t)kv_lengths[b + 1] - kv_lengths[b];
            if (kv_lengths[0] != 0 || P.kv_len[b] < 0 || kv_lengths[b + 1] > kv_seq)
                rc = ORA_ERR_LENGTHS;
        } else {
            P.kv_len[b] = kv_lengths ? kv_lengths[b] : kv_seq;
            if (P.kv_len[b] < 0 || P.kv_len[b] > kv_seq)
                rc = ORA_ERR_LENGTHS;
        }
        /* a non-broadcast mask dim must cover every within-sequence index */
        if ((mask_add || mask_bool) &&
            ((P.md[2] != 1 && P.md[2] < P.q_len[b]) ||
             (P.md[3] != 1 && P.md[3] < P.kv_len[b])))
            rc = ORA_ERR_LENGTHS;
    }
    if ((mask_add || mask_bool) &&
        ((P.md[0] != 1 && P.md[0] != B) || (P.md[1] != 1 && P.md[1] != Hq)))
        rc = ORA_ERR_ARG;

    if (rc == ORA_OK) {
        if (nthreads < 1)
            nthreads = 1;
        pthread_mutex_init(&P.lock, NULL);
        th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
        for (t = 0; t < nthreads; ++t)
            pthread_create(&th[t], NULL, worker, &P);
        for (t = 0; t < nthreads; ++t)
            pthread_join(th[t], NULL);
        free(th);
        pthread_mutex_destroy(&P.lock);
    }
    free(P.q_off); free(P.q_len); free(P.kv_off); free(P.kv_len);
    return rc;
}
