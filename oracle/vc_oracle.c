/*
 * VeriCache oracle -- plain, slow CPU definitions of the attention-step
 * operations.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product path never does.  It
 * shares no code, header or table with the CUDA library.
 *
 * Sources (page titles, sections):
 *  - "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea":
 *    drafting with the compressed cache, one verification pass that yields a
 *    prediction for each drafted position plus one, and the accept rule
 *    (left-to-right compare, correction at the first mismatch, bonus token
 *    when all match), including its worked example A..H / A..E X.
 *  - "VeriCache Guide", section "The Uniform Compressor Interface" and the
 *    compressor in "Implementing VeriCache in Python and PyTorch": token
 *    eviction = gather of a sorted kept-index list shared by all heads;
 *    low-bit quantisation families (INT2/INT4 ...).
 *  - "KV Cache and Speculative Decoding", section "Autoregressive Decoding
 *    and the KV Cache": causal attention, a query attends to itself and all
 *    earlier positions.
 * The pages give no bit format for the quantised cache; the reading used
 * here is asymmetric uniform quantisation, groups of 32 consecutive channels
 * of one token, fp16 scale and fp16 zero (= group minimum), codes packed
 * little-endian.
 *
 * Precision: attention and dequantisation in fp64 (exact dequantisation);
 * quantisation in fp32 with round-to-nearest-even because it decides integer
 * codes; logits in fp32 with one fused multiply-add per term in index order
 * because they decide an argmax.  Compile with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define VCO_GROUP 32

/* ------------------------------------------------------------------------ */
/* fp16 / bf16 conversions (IEEE binary16, round to nearest even)           */
/* ------------------------------------------------------------------------ */

uint16_t vco_f32_to_f16_rn(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) /* NaN -> quiet NaN */
        return (uint16_t)(sign | 0x7E00u);
    if (ax >= 0x477FF000u) /* >= 65520 rounds to infinity */
        return (uint16_t)(sign | 0x7C00u);
    uint32_t e = ax >> 23;
    if (e < 113) { /* below 2^-14: fp16 subnormal or zero */
        if (e < 102)
            return (uint16_t)sign; /* < 2^-25: rounds to zero */
        uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t shift = 126 - e; /* value * 2^24 = m * 2^(e-126-... ) */
        uint32_t q = m >> shift;
        uint32_t rem = m & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u)))
            q++;
        return (uint16_t)(sign | q);
    }
    uint32_t m = ax & 0x7FFFFFu;
    uint32_t h = ((e - 112) << 10) | (m >> 13);
    uint32_t rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
        h++;
    return (uint16_t)(sign | h);
}

float vco_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(m | 0x400u), (int)e - 25);
    }
    uint32_t bits;
    memcpy(&bits, &v, 4);
    bits |= sign;
    memcpy(&v, &bits, 4);
    return v;
}

float vco_bf16_to_f32(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float v;
    memcpy(&v, &bits, 4);
    return v;
}

/* fp16 storage of a scale or zero: magnitudes beyond the largest finite fp16
 * value are saturated to +-65504 before rounding (reading: the pages give no
 * overflow rule; saturation keeps the decoder finite). */
static uint16_t f16_store(float f)
{
    if (f > 65504.0f)
        f = 65504.0f;
    if (f < -65504.0f)
        f = -65504.0f;
    return vco_f32_to_f16_rn(f);
}

/* ------------------------------------------------------------------------ */
/* quantisation of one group of channels                                    */
/* ------------------------------------------------------------------------ */

/*
 * Asymmetric uniform quantisation of n values with b bits:
 *   mn, mx = min, max of the group (fp32, exact for bf16 inputs)
 *   s_dot  = (mx - mn) / (2^b - 1)        fp32, each op rounded to nearest
 *   s      = fp16(s_dot), z = fp16(mn)    stored parameters
 *   c_i    = clamp(rint((x_i - z) / s), 0, 2^b - 1), or 0 when s == 0
 * Codes are computed against the stored fp16 parameters so that encoder and
 * decoder share one grid.  A minimum of -0 is stored as +0.
 */
void vco_quantize_group(const float *x, int n, int bits, uint8_t *codes,
                        uint16_t *scale, uint16_t *zero)
{
    float mn = x[0], mx = x[0];
    for (int i = 1; i < n; i++) {
        if (x[i] < mn)
            mn = x[i];
        if (x[i] > mx)
            mx = x[i];
    }
    mn = mn + 0.0f; /* -0 -> +0 */
    int qmax = (1 << bits) - 1;
    float range = mx - mn;
    float s_dot = range / (float)qmax;
    uint16_t sh = f16_store(s_dot);
    uint16_t zh = f16_store(mn);
    *scale = sh;
    *zero = zh;
    float s = vco_f16_to_f32(sh);
    float z = vco_f16_to_f32(zh);
    for (int i = 0; i < n; i++) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float t = (x[i] - z) / s;
        float r = nearbyintf(t); /* default rounding mode: nearest even */
        if (r < 0.0f)
            r = 0.0f;
        if (r > (float)qmax)
            r = (float)qmax;
        codes[i] = (uint8_t)r;
    }
}

/* one token's d channels (bf16 bits) -> codes[d], scales[d/32], zeros[d/32] */
void vco_quantize_row(const uint16_t *x_bf16, int d, int bits, uint8_t *codes,
                      uint16_t *scales, uint16_t *zeros)
{
    float g[VCO_GROUP];
    for (int j = 0; j < d / VCO_GROUP; j++) {
        for (int i = 0; i < VCO_GROUP; i++)
            g[i] = vco_bf16_to_f32(x_bf16[j * VCO_GROUP + i]);
        vco_quantize_group(g, VCO_GROUP, bits, codes + j * VCO_GROUP, scales + j, zeros + j);
    }
}

/* code i occupies bits [b*i, b*i + b) of the little-endian byte string */
void vco_pack_codes(const uint8_t *codes, int d, int bits, uint8_t *packed)
{
    memset(packed, 0, (size_t)d * bits / 8);
    for (int i = 0; i < d; i++) {
        for (int k = 0; k < bits; k++) {
            int bit = bits * i + k;
            if ((codes[i] >> k) & 1)
                packed[bit / 8] |= (uint8_t)(1u << (bit % 8));
        }
    }
}

void vco_unpack_codes(const uint8_t *packed, int d, int bits, uint8_t *codes)
{
    for (int i = 0; i < d; i++) {
        uint8_t c = 0;
        for (int k = 0; k < bits; k++) {
            int bit = bits * i + k;
            if ((packed[bit / 8] >> (bit % 8)) & 1)
                c |= (uint8_t)(1u << k);
        }
        codes[i] = c;
    }
}

/* x_hat = s * c + z, evaluated exactly in fp64 */
void vco_dequant_row(const uint8_t *codes, const uint16_t *scales, const uint16_t *zeros,
                     int d, double *out)
{
    for (int i = 0; i < d; i++) {
        double s = (double)vco_f16_to_f32(scales[i / VCO_GROUP]);
        double z = (double)vco_f16_to_f32(zeros[i / VCO_GROUP]);
        out[i] = s * (double)codes[i] + z;
    }
}

/* ------------------------------------------------------------------------ */
/* compression of one request: gather by the kept list, then quantise       */
/* ------------------------------------------------------------------------ */

/*
 * k, v: logical [n][hkv][d] bf16.  kept: n_kept positions (each < n).
 * bits in {2,3,4}: packed [n_kept][hkv][d*bits/8], scales/zeros
 *                  [n_kept][hkv][d/32] for K and for V.
 * bits == 16:      gathered [n_kept][hkv][d] bf16 in k_out16 / v_out16.
 * Returns 0, or -1 on a kept index outside [0, n).
 */
int vco_compress(const uint16_t *k, const uint16_t *v, int n, int hkv, int d,
                 const int32_t *kept, int n_kept, int bits,
                 uint8_t *k_packed, uint16_t *k_scales, uint16_t *k_zeros,
                 uint8_t *v_packed, uint16_t *v_scales, uint16_t *v_zeros,
                 uint16_t *k_out16, uint16_t *v_out16)
{
    int pb = d * bits / 8, ng = d / VCO_GROUP;
    uint8_t *codes = (uint8_t *)malloc((size_t)d);
    for (int j = 0; j < n_kept; j++) {
        int t = kept[j];
        if (t < 0 || t >= n) {
            free(codes);
            return -1;
        }
        for (int h = 0; h < hkv; h++) {
            const uint16_t *ks = k + ((size_t)t * hkv + h) * d;
            const uint16_t *vs = v + ((size_t)t * hkv + h) * d;
            size_t row = (size_t)j * hkv + h;
            if (bits == 16) {
                memcpy(k_out16 + row * d, ks, (size_t)d * 2);
                memcpy(v_out16 + row * d, vs, (size_t)d * 2);
                continue;
            }
            vco_quantize_row(ks, d, bits, codes, k_scales + row * ng, k_zeros + row * ng);
            vco_pack_codes(codes, d, bits, k_packed + row * pb);
            vco_quantize_row(vs, d, bits, codes, v_scales + row * ng, v_zeros + row * ng);
            vco_pack_codes(codes, d, bits, v_packed + row * pb);
        }
    }
    free(codes);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* attention                                                                */
/* ------------------------------------------------------------------------ */

/*
 * Single-query softmax attention in fp64 over n explicit keys/values:
 *   s_t = scale * <q, k_t>,  p_t = exp(s_t - max_s) / sum_j exp(s_j - max_s)
 *   o   = sum_t p_t v_t
 * weights (optional, length n) receives p.
 */
void vco_attend(const double *q, const double *keys, const double *vals, int n, int d,
                double scale, double *out, double *weights)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    for (int t = 0; t < n; t++) {
        double acc = 0.0;
        for (int i = 0; i < d; i++)
            acc += q[i] * keys[(size_t)t * d + i];
        s[t] = scale * acc;
        if (s[t] > m)
            m = s[t];
    }
    double l = 0.0;
    for (int t = 0; t < n; t++) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int i = 0; i < d; i++)
        out[i] = 0.0;
    for (int t = 0; t < n; t++) {
        double p = s[t] / l;
        if (weights)
            weights[t] = p;
        for (int i = 0; i < d; i++)
            out[i] += p * vals[(size_t)t * d + i];
    }
    free(s);
}

/*
 * Draft attention of one request: one query per query head over the n_comp
 * entries of its compressed cache.  Query head h reads kv head h / (hq/hkv).
 * q: [hq][d] bf16.  Cache in the logical layout written by vco_compress.
 * out: [hq][d] fp64.
 */
int vco_draft_attn(const uint16_t *q, int hq, int hkv, int d, int n_comp, int bits,
                   const uint8_t *k_packed, const uint16_t *k_scales, const uint16_t *k_zeros,
                   const uint8_t *v_packed, const uint16_t *v_scales, const uint16_t *v_zeros,
                   const uint16_t *k16, const uint16_t *v16, double scale, double *out)
{
    if (hkv <= 0 || hq % hkv)
        return -1;
    int grp = hq / hkv, pb = d * bits / 8, ng = d / VCO_GROUP;
    double *keys = (double *)malloc(sizeof(double) * (size_t)(n_comp > 0 ? n_comp : 1) * d);
    double *vals = (double *)malloc(sizeof(double) * (size_t)(n_comp > 0 ? n_comp : 1) * d);
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    uint8_t *codes = (uint8_t *)malloc((size_t)d);
    for (int g = 0; g < hkv; g++) {
        for (int t = 0; t < n_comp; t++) {
            size_t row = (size_t)t * hkv + g;
            if (bits == 16) {
                for (int i = 0; i < d; i++) {
                    keys[(size_t)t * d + i] = vco_bf16_to_f32(k16[row * d + i]);
                    vals[(size_t)t * d + i] = vco_bf16_to_f32(v16[row * d + i]);
                }
            } else {
                vco_unpack_codes(k_packed + row * pb, d, bits, codes);
                vco_dequant_row(codes, k_scales + row * ng, k_zeros + row * ng, d, keys + (size_t)t * d);
                vco_unpack_codes(v_packed + row * pb, d, bits, codes);
                vco_dequant_row(codes, v_scales + row * ng, v_zeros + row * ng, d, vals + (size_t)t * d);
            }
        }
        for (int hh = 0; hh < grp; hh++) {
            int h = g * grp + hh;
            for (int i = 0; i < d; i++)
                qd[i] = vco_bf16_to_f32(q[(size_t)h * d + i]);
            vco_attend(qd, keys, vals, n_comp, d, scale, out + (size_t)h * d, NULL);
        }
    }
    free(keys);
    free(vals);
    free(qd);
    free(codes);
    return 0;
}

/*
 * Verification attention of one request over its full cache of n_ctx tokens,
 * the last n_q of which are the block being verified.  Query i sits at
 * position p_i = n_ctx - n_q + i and attends to positions 0..p_i (causal
 * inside the block, the whole prefix before it).
 * q: [n_q][hq][d] bf16;  k, v: [n_ctx][hkv][d] bf16;  out: [n_q][hq][d] fp64.
 */
int vco_verify_attn(const uint16_t *q, int n_q, int hq, int hkv, int d, int n_ctx,
                    const uint16_t *k, const uint16_t *v, double scale, double *out)
{
    if (hkv <= 0 || hq % hkv || n_q > n_ctx)
        return -1;
    int grp = hq / hkv;
    double *keys = (double *)malloc(sizeof(double) * (size_t)(n_ctx > 0 ? n_ctx : 1) * d);
    double *vals = (double *)malloc(sizeof(double) * (size_t)(n_ctx > 0 ? n_ctx : 1) * d);
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    for (int g = 0; g < hkv; g++) {
        for (int t = 0; t < n_ctx; t++)
            for (int i = 0; i < d; i++) {
                keys[(size_t)t * d + i] = vco_bf16_to_f32(k[((size_t)t * hkv + g) * d + i]);
                vals[(size_t)t * d + i] = vco_bf16_to_f32(v[((size_t)t * hkv + g) * d + i]);
            }
        for (int i = 0; i < n_q; i++) {
            int pos = n_ctx - n_q + i;
            for (int hh = 0; hh < grp; hh++) {
                int h = g * grp + hh;
                for (int c = 0; c < d; c++)
                    qd[c] = vco_bf16_to_f32(q[((size_t)i * hq + h) * d + c]);
                vco_attend(qd, keys, vals, pos + 1, d, scale, out + ((size_t)i * hq + h) * d, NULL);
            }
        }
    }
    free(keys);
    free(vals);
    free(qd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* greedy acceptance                                                         */
/* ------------------------------------------------------------------------ */

/*
 * hidden: [n_pred][hg][dm] fp32 -- each prediction's hidden vector is the
 *         mean of hg consecutive dm-vectors (hg = 1: the vector itself);
 *         mean = (fp32 sum in index order) / hg.
 * w:      [dm][vocab] fp32 LM head.
 * logit_v = fp32 dot(h, w[:, v]) with one fused multiply-add per term, k in
 *         increasing order.  verified[i] = argmax_v logit_v, lowest v on ties.
 * drafts: [x].  a = first i < x with drafts[i] != verified[i], else x.
 * emitted: [x+1], filled with drafts[0:a] then verified[a] when a < n_pred;
 *         remaining slots -1.  Returns the number of emitted tokens.
 * If ambiguous (len n_pred) is given, ambiguous[i] = 1 when the fp64 logits
 * leave more than one id within the fp32 dot-product error bound
 * gamma_m * (sum_k |h_k w_kv| + sum_k |h_k w_kv*|), gamma_m = m u / (1 - m u),
 * u = 2^-24, m = dm + hg + 1 (report-only: the near-tie rule).
 */
int vco_accept(const float *hidden, int n_pred, int hg, const float *w, int dm, int vocab,
               const int32_t *drafts, int x, int32_t *verified, int32_t *accept_len,
               int32_t *emitted, uint8_t *ambiguous)
{
    float *h = (float *)malloc(sizeof(float) * (size_t)dm);
    double *hd = (double *)malloc(sizeof(double) * (size_t)dm);
    for (int i = 0; i < n_pred; i++) {
        for (int k = 0; k < dm; k++) {
            float s = 0.0f;
            for (int j = 0; j < hg; j++)
                s = s + hidden[((size_t)i * hg + j) * dm + k];
            h[k] = s / (float)hg;
            hd[k] = (double)h[k];
        }
        int best = 0;
        float bestv = -INFINITY;
        for (int v = 0; v < vocab; v++) {
            float acc = 0.0f;
            for (int k = 0; k < dm; k++)
                acc = fmaf(h[k], w[(size_t)k * vocab + v], acc);
            if (acc > bestv) {
                bestv = acc;
                best = v;
            }
        }
        verified[i] = best;
        if (ambiguous) {
            double u = ldexp(1.0, -24), mm = (double)(dm + hg + 1);
            double gam = mm * u / (1.0 - mm * u);
            double lb = 0.0, ab = 0.0;
            for (int k = 0; k < dm; k++) {
                double p = hd[k] * (double)w[(size_t)k * vocab + best];
                lb += p;
                ab += fabs(p);
            }
            int amb = 0;
            for (int v = 0; v < vocab && !amb; v++) {
                if (v == best)
                    continue;
                double l = 0.0, a = 0.0;
                for (int k = 0; k < dm; k++) {
                    double p = hd[k] * (double)w[(size_t)k * vocab + v];
                    l += p;
                    a += fabs(p);
                }
                if (lb - l <= gam * (ab + a))
                    amb = 1;
            }
            ambiguous[i] = (uint8_t)amb;
        }
    }
    free(h);
    free(hd);
    int a = 0;
    while (a < x && a < n_pred && drafts[a] == verified[a])
        a++;
    *accept_len = a;
    int ne = 0;
    for (int j = 0; j < a; j++)
        emitted[ne++] = drafts[j];
    if (a < n_pred)
        emitted[ne++] = verified[a];
    for (int j = ne; j < x + 1; j++)
        emitted[j] = -1;
    return ne;
}

/*
 * Token importance of the guide's compressor ("VeriCache Guide",
 * "Implementing VeriCache in Python and PyTorch", the compressor class: the
 * key norm over the head dimension, averaged over heads, ranks the tokens).
 * Reading fixed here so that a kept list is reproducible bit for bit: fp32,
 * per kv head the sum of squares with one fused multiply-add per channel in
 * increasing channel order, a correctly rounded square root, the heads'
 * norms added in increasing head order, then divided by the head count.
 * k: [n][hkv][d] bf16; score: [n].
 */
void vco_keynorm_scores(const uint16_t *k, int n, int hkv, int d, float *score)
{
    for (int t = 0; t < n; t++) {
        float tot = 0.0f;
        for (int h = 0; h < hkv; h++) {
            const uint16_t *row = k + ((size_t)t * hkv + h) * d;
            float ss = 0.0f;
            for (int c = 0; c < d; c++) {
                float x = vco_bf16_to_f32(row[c]);
                ss = fmaf(x, x, ss);
            }
            tot = tot + sqrtf(ss);
        }
        score[t] = tot / (float)hkv;
    }
}

/* (score, position) order of the selection: higher score first, equal
 * scores by lower position */
typedef struct {
    float s;
    int i;
} vco_ranked;

static int vco_rank_cmp(const void *a, const void *b)
{
    const vco_ranked *x = (const vco_ranked *)a, *y = (const vco_ranked *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

/*
 * Kept-index list of one request (the guide's compressor: the top tokens by
 * importance, then sorted by position; with the sink / recent window of the
 * workloads): positions [0, sink) and [n - recent, n) always (clamped to n),
 * plus the `keep - sink - recent` middle positions of highest score, equal
 * scores by lower position, all written in ascending position order.  The
 * middle takes max(0, min(n - sink - recent, keep - sink - recent))
 * positions.  Returns the number of indices written.
 */
int vco_select_kept(const float *score, int n, int sink, int recent, int keep, int32_t *idx)
{
    if (sink > n) sink = n;
    if (recent > n - sink) recent = n - sink;
    int m = n - sink - recent;
    int top = keep - sink - recent;
    if (top < 0) top = 0;
    if (top > m) top = m;
    uint8_t *take = (uint8_t *)calloc((size_t)n + 1, 1);
    vco_ranked *r = (vco_ranked *)malloc(sizeof(vco_ranked) * ((size_t)m + 1));
    for (int j = 0; j < m; j++) {
        r[j].s = score[sink + j];
        r[j].i = sink + j;
    }
    qsort(r, (size_t)m, sizeof(vco_ranked), vco_rank_cmp);
    for (int j = 0; j < top; j++) take[r[j].i] = 1;
    for (int t = 0; t < sink; t++) take[t] = 1;
    for (int t = n - recent; t < n; t++) take[t] = 1;
    int c = 0;
    for (int t = 0; t < n; t++)
        if (take[t]) idx[c++] = t;
    free(take);
    free(r);
    return c;
}

/*
 * Logits of hidden rows: mean of each row's hidden group (fp32, increasing
 * j), then one fused multiply-add per hidden index in increasing order --
 * the same arithmetic as vco_accept.  hidden [rows][hg][dm] -> out [rows][vocab].
 */
void vco_logits(const float *hidden, int rows, int hg, const float *w, int dm, int vocab, float *out)
{
    float *h = (float *)malloc(sizeof(float) * (size_t)dm);
    for (int i = 0; i < rows; i++) {
        for (int k = 0; k < dm; k++) {
            float s = 0.0f;
            for (int j = 0; j < hg; j++)
                s = s + hidden[((size_t)i * hg + j) * dm + k];
            h[k] = s / (float)hg;
        }
        for (int v = 0; v < vocab; v++) {
            float acc = 0.0f;
            for (int k = 0; k < dm; k++)
                acc = fmaf(h[k], w[(size_t)k * vocab + v], acc);
            out[(size_t)i * vocab + v] = acc;
        }
    }
    free(h);
}

/* softmax(logits / tau) in fp64 */
static void vco_softmax64(const float *l, int vocab, double tau, double *p)
{
    double m = -INFINITY;
    for (int v = 0; v < vocab; v++)
        if ((double)l[v] / tau > m) m = (double)l[v] / tau;
    double z = 0.0;
    for (int v = 0; v < vocab; v++) {
        p[v] = exp((double)l[v] / tau - m);
        z += p[v];
    }
    for (int v = 0; v < vocab; v++) p[v] /= z;
}

/* inverse CDF: the first id whose cumulative weight exceeds u * total;
 * *margin = distance of u * total to the nearest cumulative boundary,
 * relative to total */
static int vco_sample_cdf(const double *wgt, int vocab, double u, double *margin)
{
    double tot = 0.0;
    for (int v = 0; v < vocab; v++) tot += wgt[v];
    double thr = u * tot, cum = 0.0;
    int pick = vocab - 1;
    double best = INFINITY;
    for (int v = 0; v < vocab; v++) {
        if (wgt[v] <= 0.0) continue;
        double next = cum + wgt[v];
        double dm = fabs(next - thr);
        if (dm < best) best = dm;
        if (pick == vocab - 1 && next > thr) {
            pick = v;
        }
        cum = next;
    }
    /* ids after the last positive weight are never picked */
    if (pick == vocab - 1)
        for (int v = vocab - 1; v >= 0; v--)
            if (wgt[v] > 0.0) {
                pick = v;
                break;
            }
    *margin = tot > 0.0 ? best / tot : 0.0;
    return pick;
}

/*
 * Speculative acceptance with rejection sampling ("VeriCache Guide",
 * "Mathematical Guarantee of Lossless Correctness"): draft token d_i is kept
 * when u_i < alpha_i = min(1, p_target_i(d_i) / p_draft_i(d_i)); at the first
 * rejection a token is drawn from the residual max(0, p_target_i -
 * p_draft_i) (normalised) by inverse CDF with uniform v_i and the round
 * ends; when all x drafts are kept a bonus token is drawn from
 * p_target_x with v_x.  Distributions are softmax(logits / tau), in fp64.
 * target_logits [x+1][vocab], draft_logits [x][vocab], u [x], v [x+1].
 * emitted [x+1] (then -1); margins [x+1]: per decision taken, its distance
 * to flipping (|u - alpha| for an accept test, the inverse-CDF boundary
 * distance for a draw); returns the number of emitted tokens.
 */
int vco_accept_sampled(const float *target_logits, const float *draft_logits, int vocab, float tau,
                       const int32_t *drafts, int x, const float *u, const float *v, int32_t *accept_len,
                       int32_t *emitted, double *margins)
{
    double *pt = (double *)malloc(sizeof(double) * (size_t)vocab);
    double *pd = (double *)malloc(sizeof(double) * (size_t)vocab);
    int ne = 0, a = 0;
    for (int j = 0; j < x + 1; j++) margins[j] = INFINITY;
    for (; a < x; a++) {
        vco_softmax64(target_logits + (size_t)a * vocab, vocab, (double)tau, pt);
        vco_softmax64(draft_logits + (size_t)a * vocab, vocab, (double)tau, pd);
        const int d = drafts[a];
        const double alpha = pd[d] > 0.0 ? fmin(1.0, pt[d] / pd[d]) : 1.0;
        margins[a] = fabs((double)u[a] - alpha);
        if ((double)u[a] < alpha) {
            emitted[ne++] = d;
            continue;
        }
        for (int t = 0; t < vocab; t++) pd[t] = fmax(0.0, pt[t] - pd[t]);
        double mg;
        emitted[ne++] = vco_sample_cdf(pd, vocab, (double)v[a], &mg);
        if (mg < margins[a]) margins[a] = mg;
        break;
    }
    if (a == x) {
        vco_softmax64(target_logits + (size_t)x * vocab, vocab, (double)tau, pt);
        double mg;
        emitted[ne++] = vco_sample_cdf(pt, vocab, (double)v[x], &mg);
        margins[x] = mg;
    }
    *accept_len = a;
    for (int j = ne; j < x + 1; j++) emitted[j] = -1;
    free(pt);
    free(pd);
    return ne;
}

/* array helpers for the tests */
void vco_f32_to_f16_array(const float *x, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = vco_f32_to_f16_rn(x[i]);
}

void vco_f16_to_f32_array(const uint16_t *x, float *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = vco_f16_to_f32(x[i]);
}
