/*
 * oracle.c -- plain, slow, obviously correct CPU reference of the batched
 * Q4_K decode step.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg may call it; the library never does.
 * It shares no code with the CUDA path (or with the input generator).
 *
 * What it computes follows three blog pages on batched decode of a GQA
 * transformer ("Eight concurrent agents pull 5.6x more tokens from one RX
 * 9070 XT", "Batched swarm: the KV read does not amortize", "Q8 KV cache
 * pushes an RDNA4 swarm crossover from 5k to 10k tokens"):
 *   - one decode step advances B sequences; the weights are the same for all
 *     of them and each sequence reads its own KV cache ("The weight read is
 *     the only term that does not scale", "The two halves of a decode-step
 *     memory bill");
 *   - the KV cache is fp16 or 8-bit (Q8_0, or FP8 e4m3 as the pages' scale-free
 *     alternative), per tensor, dequantized where it is read ("Why Q8 is
 *     close to free and where the sharp edges are");
 *   - greedy sampling of the LM head output.
 * The pages leave the model's layer arithmetic open; the plain readings used
 * here are: RMSNorm (eps 1e-6 unless given), rotate-half RoPE on pairs
 * (i, i+hd/2) with inv_freq_i = theta^(-2i/hd), grouped-query attention with
 * query head h reading kv head h/(n_q/n_kv), softmax in double, SwiGLU FFN,
 * fp32 residual stream, tied embedding / LM head, argmax ties to the lowest
 * index.  The Q4_K block layout and Q8_0 rule are the ones the synthetic
 * model uses (fp16 d/dmin, 6-bit scales and mins per 32, 4-bit codes; Q8_0:
 * 32-element blocks, fp16 scale amax/127, round-half-even int8).
 *
 * Arithmetic is fp64 except where a storage precision is part of the
 * definition: dequantized Q4_K weights are fp32 values, matmul outputs and
 * the residual stream are stored as fp32, the KV cache holds fp16 or Q8_0.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------ fp16 ---- */

/* binary16 bits -> value (exact). */
float orc_half_to_float(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp((double)(1024 + m), e - 25);
    return (float)(s ? -v : v);
}

/* Round a double to the nearest binary16 (ties to even).  The value is
 * scaled by a power of two so that the kept significand becomes an integer
 * and rint() does the single rounding. */
uint16_t orc_double_to_half(double v) {
    if (isnan(v)) return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0) return sign | 0x7C00;            /* rounds to infinity */
    if (a < ldexp(1.0, -14)) {                          /* subnormal range */
        double m = rint(ldexp(a, 24));                  /* units of 2^-24 */
        return sign | (uint16_t)m;                      /* m == 1024 is the smallest normal */
    }
    int E;
    frexp(a, &E);                                       /* a = f*2^E, f in [0.5,1) */
    int e = E - 1;                                      /* a in [2^e, 2^(e+1)) */
    double m = rint(ldexp(a, 10 - e));                  /* in [1024, 2048] */
    if (m == 2048.0) { m = 1024.0; e += 1; }
    if (e > 15) return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)m - 1024));
}

/* ------------------------------------------------------------ Q4_K ---- */

/* Read one canonical 144-byte block: d, dmin (fp16), sixteen 6-bit fields
 * (bits 6i..6i+5 of the little-endian 96-bit word at bytes 4..15; fields
 * 0-7 are sub-block scales, 8-15 sub-block mins) and 256 4-bit codes (byte t:
 * element 2t low nibble, 2t+1 high nibble). */
void orc_q4k_unpack(const uint8_t *blk, float *d, float *dmin, int sc[8], int mn[8], int q[256]) {
    *d = orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    *dmin = orc_half_to_float((uint16_t)(blk[2] | (blk[3] << 8)));
    for (int i = 0; i < 16; i++) {
        int v = 0;
        for (int b = 0; b < 6; b++) {
            int bit = 6 * i + b;
            if (blk[4 + bit / 8] & (1 << (bit % 8))) v |= 1 << b;
        }
        if (i < 8) sc[i] = v; else mn[i - 8] = v;
    }
    for (int t = 0; t < 128; t++) {
        q[2 * t] = blk[16 + t] & 15;
        q[2 * t + 1] = blk[16 + t] >> 4;
    }
}

/* Dequantize one block: w_i = (d*sc_j)*q_i - (dmin*m_j), j = i/32, each
 * operation a separately rounded fp32 operation in this order. */
void orc_q4k_dequant(const uint8_t *blk, float out[256]) {
    float d, dmin;
    int sc[8], mn[8], q[256];
    orc_q4k_unpack(blk, &d, &dmin, sc, mn, q);
    for (int i = 0; i < 256; i++) {
        int j = i / 32;
        float step = d * (float)sc[j];
        float off = dmin * (float)mn[j];
        float prod = step * (float)q[i];
        out[i] = prod - off;
    }
}

/* y[n] = sum_k W[n][k] x[k], W given as canonical Q4_K rows (K/256 blocks
 * per row), summed in double. */
void orc_q4k_matvec(const uint8_t *W, int64_t N, int64_t K, const double *x, double *y) {
    int64_t nb = K / 256;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        float w[256];
        double acc = 0.0;
        for (int64_t b = 0; b < nb; b++) {
            orc_q4k_dequant(W + (n * nb + b) * 144, w);
            for (int i = 0; i < 256; i++) acc += (double)w[i] * x[b * 256 + i];
        }
        y[n] = acc;
    }
}

/* ------------------------------------------------------------ Q8_0 ---- */

/* Q8_0 block of 32 fp16 values: amax = max|x| (exact in fp32),
 * d = amax/127 (fp32 division), stored scale = fp16(d);
 * q_i = clamp(rint(x_i/d), -127, 127) with the fp32 d (not the fp16 one),
 * ties to even; an all-zero block stores scale 0 and codes 0. */
void orc_q8_0_quantize(const uint16_t x16[32], uint16_t *scale, int8_t q[32]) {
    float x[32], amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        x[i] = orc_half_to_float(x16[i]);
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        *scale = 0;
        memset(q, 0, 32);
        return;
    }
    float d = amax / 127.0f;
    *scale = orc_double_to_half((double)d);
    for (int i = 0; i < 32; i++) {
        float r = rintf(x[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

/* Value a Q8_0 code stands for: fp16 scale times the code. */
double orc_q8_0_value(uint16_t scale, int8_t q) {
    return (double)orc_half_to_float(scale) * (double)q;
}

/* ------------------------------------------------------------ FP8 ----- */

/* FP8 e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities, S.1111.111 is NaN, largest finite 448).  The cache type the
 * pages name as the scale-free alternative to Q8 ("FP8 (e4m3) KV ... native
 * Blackwell conversion, same bytes as Q8, no scale"): each fp16 value maps to
 * the nearest e4m3 value, ties to the even code, magnitudes at or beyond 448
 * to +-448 (saturating, as the hardware's satfinite conversion), NaN to NaN. */
uint8_t orc_e4m3_from_half(uint16_t h) {
    double x = (double)orc_half_to_float(h);
    uint8_t sign = (h & 0x8000u) ? 0x80u : 0x00u;
    if (x != x) return (uint8_t)(sign | 0x7Fu);
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    int e;
    frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                         /* a = (1 + m) * 2^e, m in [0, 1) */
    if (e < -6) {                   /* subnormal: a = M * 2^-9, M in 0..7 */
        double M = rint(ldexp(a, 9));   /* exact scaling; rint ties to even */
        return (uint8_t)(sign | (uint8_t)M);   /* M = 8 is the smallest normal's code */
    }
    double M = rint((ldexp(a, -e) - 1.0) * 8.0);
    if (M == 8.0) { M = 0.0; e += 1; }
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)M);
}

/* Value of an e4m3 code (NaN for S.1111.111). */
double orc_e4m3_value(uint8_t c) {
    int E = (c >> 3) & 15, M = c & 7;
    double sign = (c & 0x80u) ? -1.0 : 1.0;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) return sign * ldexp((double)M, -9);
    return sign * ldexp(1.0 + M / 8.0, E - 7);
}

/* ------------------------------------------------------- layer math ---- */

/* y = x / sqrt(mean(x^2) + eps) * g, in double. */
void orc_rmsnorm(const double *x, const float *g, int64_t n, double eps, double *y) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; i++) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; i++) y[i] = x[i] * r * (double)g[i];
}

/* Rotate-half RoPE of one head vector at position pos: pairs (i, i+hd/2),
 * angle = pos * theta^(-2i/hd). */
void orc_rope(double *v, int hd, int64_t pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; i++) {
        double inv = pow(theta, -2.0 * (double)i / (double)hd);
        double a = (double)pos * inv;
        double c = cos(a), s = sin(a);
        double x0 = v[i], x1 = v[i + half];
        v[i] = x0 * c - x1 * s;
        v[i + half] = x1 * c + x0 * s;
    }
}

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* Greedy argmax, ties to the lowest index. */
int64_t orc_argmax(const float *x, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; i++)
        if (x[i] > x[best]) best = i;
    return best;
}

/* ------------------------------------------------------ KV cache ---- */

/* One sequence's cache in canonical layout, tokens major:
 *   fp16:  k16/v16  [n_layers][max_L][n_kv][hd]          binary16 bits
 *   Q8_0:  kq/vq    [n_layers][max_L][n_kv][hd]          int8 codes
 *          ks/vs    [n_layers][max_L][n_kv][hd/32]       fp16 scales
 *   FP8:   k8/v8    [n_layers][max_L][n_kv][hd]          e4m3 codes
 * K and V may have different types (llama.cpp-style separate cache types). */
typedef struct {
    int kv_dtype;          /* 0 = fp16, 1 = Q8_0, 2 = FP8 e4m3 for both tensors; -1: k_type / v_type */
    int64_t max_L;
    uint16_t *k16, *v16;
    int8_t *kq, *vq;
    uint16_t *ks, *vs;
    uint8_t *k8, *v8;      /* e4m3 codes [n_layers][max_L][n_kv][hd] */
    int k_type, v_type;    /* per-tensor types when kv_dtype = -1 */
} orc_kv;

/* Storage type of K (which = 0) or V (which = 1). */
static inline int orc_kv_type(const orc_kv *kv, int which) {
    return kv->kv_dtype >= 0 ? kv->kv_dtype : (which ? kv->v_type : kv->k_type);
}

/* Store one head row of hd fp16 values of K (which = 0) or V at `row`. */
static void orc_kv_put_row(orc_kv *kv, int which, int hd, int64_t row, const uint16_t *x16) {
    switch (orc_kv_type(kv, which)) {
        case 0:
            memcpy((which ? kv->v16 : kv->k16) + row * hd, x16, (size_t)hd * 2);
            break;
        case 1:
            for (int b = 0; b < hd / 32; b++)
                orc_q8_0_quantize(x16 + 32 * b, (which ? kv->vs : kv->ks) + row * (hd / 32) + b,
                                  (which ? kv->vq : kv->kq) + row * hd + 32 * b);
            break;
        default:
            for (int i = 0; i < hd; i++) (which ? kv->v8 : kv->k8)[row * hd + i] = orc_e4m3_from_half(x16[i]);
            break;
    }
}

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    double rope_theta, rms_eps;
} orc_desc;

typedef struct {
    const uint8_t *embed;              /* [vocab][hidden/256] blocks; tied LM head */
    const float *final_norm;           /* [hidden] */
    const float *const *attn_norm;     /* [n_layers] -> [hidden] */
    const float *const *ffn_norm;
    const uint8_t *const *wq, *const *wk, *const *wv, *const *wo;
    const uint8_t *const *w_gate, *const *w_up, *const *w_down;
} orc_weights;

/* Store one head row (hd values, already rotated for K) at (layer, t, kvh). */
static void orc_kv_store(const orc_desc *m, orc_kv *kv, int layer, int64_t t, int kvh,
                         const double *kr, const double *vr) {
    int hd = m->head_dim;
    int64_t row = (((int64_t)layer * kv->max_L + t) * m->n_kv_heads + kvh);
    uint16_t k16[1024], v16[1024];
    for (int i = 0; i < hd; i++) {
        k16[i] = orc_double_to_half(kr[i]);
        v16[i] = orc_double_to_half(vr[i]);
    }
    orc_kv_put_row(kv, 0, hd, row, k16);
    orc_kv_put_row(kv, 1, hd, row, v16);
}

/* Element i of the stored K (which=0) or V (which=1) row at (layer, t, kvh). */
static inline double orc_kv_get(const orc_desc *m, const orc_kv *kv, int layer, int64_t t,
                                int kvh, int which, int i) {
    int hd = m->head_dim;
    int64_t row = (((int64_t)layer * kv->max_L + t) * m->n_kv_heads + kvh);
    switch (orc_kv_type(kv, which)) {
        case 0: return (double)orc_half_to_float((which ? kv->v16 : kv->k16)[row * hd + i]);
        case 1: {
            const int8_t *q = which ? kv->vq : kv->kq;
            const uint16_t *s = which ? kv->vs : kv->ks;
            return orc_q8_0_value(s[row * (hd / 32) + i / 32], q[row * hd + i]);
        }
        default: return orc_e4m3_value((which ? kv->v8 : kv->k8)[row * hd + i]);
    }
}

/* Grouped-query attention for one sequence at position pos over the stored
 * tokens 0..pos: o_h = sum_t softmax_t(q_h.k_t / sqrt(hd)) v_t, query head h
 * reading kv head h / (n_q/n_kv). */
void orc_attention(const orc_desc *m, const orc_kv *kv, int layer, int64_t pos,
                   const double *q, double *o) {
    int hd = m->head_dim, group = m->n_q_heads / m->n_kv_heads;
    double scale = 1.0 / sqrt((double)hd);
    #pragma omp parallel for schedule(static)
    for (int h = 0; h < m->n_q_heads; h++) {
        int kvh = h / group;
        double *sc = (double *)malloc((size_t)(pos + 1) * sizeof(double));
        double mx = -INFINITY;
        for (int64_t t = 0; t <= pos; t++) {
            double s = 0.0;
            for (int i = 0; i < hd; i++) s += q[h * hd + i] * orc_kv_get(m, kv, layer, t, kvh, 0, i);
            sc[t] = s * scale;
            if (sc[t] > mx) mx = sc[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t <= pos; t++) { sc[t] = exp(sc[t] - mx); den += sc[t]; }
        for (int i = 0; i < hd; i++) o[h * hd + i] = 0.0;
        for (int64_t t = 0; t <= pos; t++) {
            double p = sc[t] / den;
            for (int i = 0; i < hd; i++) o[h * hd + i] += p * orc_kv_get(m, kv, layer, t, kvh, 1, i);
        }
        free(sc);
    }
}

static void orc_round_f32(double *v, int64_t n) {
    for (int64_t i = 0; i < n; i++) v[i] = (double)(float)v[i];
}

/* One decode step of one sequence.  Appends the new token's K/V at `pos`
 * (rounded to fp16, then Q8_0-quantized when the cache is Q8_0), attends
 * over tokens 0..pos, writes fp32 logits and returns the greedy id.
 * hidden (optional) receives the fp32 residual after the embedding and after
 * each layer: [n_layers+1][hidden]. */
int64_t orc_decode_one(const orc_desc *m, const orc_weights *w, orc_kv *kv,
                       int32_t token, int64_t pos, float *logits, float *hidden) {
    int H = m->hidden, hd = m->head_dim, nq = m->n_q_heads, nkv = m->n_kv_heads;
    int F = m->ffn;
    float *x = (float *)malloc((size_t)H * sizeof(float));
    double *xd = (double *)malloc((size_t)H * sizeof(double));
    double *h = (double *)malloc((size_t)H * sizeof(double));
    double *q = (double *)malloc((size_t)nq * hd * sizeof(double));
    double *k = (double *)malloc((size_t)nkv * hd * sizeof(double));
    double *v = (double *)malloc((size_t)nkv * hd * sizeof(double));
    double *o = (double *)malloc((size_t)nq * hd * sizeof(double));
    double *y = (double *)malloc((size_t)(F > H ? F : H) * sizeof(double));
    double *g = (double *)malloc((size_t)F * sizeof(double));
    double *u = (double *)malloc((size_t)F * sizeof(double));
    double *lg = (double *)malloc((size_t)m->vocab * sizeof(double));

    /* embedding row of the tied matrix */
    for (int b = 0; b < H / 256; b++)
        orc_q4k_dequant(w->embed + ((int64_t)token * (H / 256) + b) * 144, x + 256 * b);
    if (hidden) memcpy(hidden, x, (size_t)H * sizeof(float));

    for (int l = 0; l < m->n_layers; l++) {
        for (int i = 0; i < H; i++) xd[i] = x[i];
        orc_rmsnorm(xd, w->attn_norm[l], H, m->rms_eps, h);
        orc_q4k_matvec(w->wq[l], (int64_t)nq * hd, H, h, q);
        orc_q4k_matvec(w->wk[l], (int64_t)nkv * hd, H, h, k);
        orc_q4k_matvec(w->wv[l], (int64_t)nkv * hd, H, h, v);
        orc_round_f32(q, (int64_t)nq * hd);
        orc_round_f32(k, (int64_t)nkv * hd);
        orc_round_f32(v, (int64_t)nkv * hd);
        for (int hh = 0; hh < nq; hh++) orc_rope(q + hh * hd, hd, pos, m->rope_theta);
        for (int hh = 0; hh < nkv; hh++) orc_rope(k + hh * hd, hd, pos, m->rope_theta);
        for (int hh = 0; hh < nkv; hh++) orc_kv_store(m, kv, l, pos, hh, k + hh * hd, v + hh * hd);
        orc_attention(m, kv, l, pos, q, o);
        orc_q4k_matvec(w->wo[l], H, (int64_t)nq * hd, o, y);
        for (int i = 0; i < H; i++) x[i] = (float)((double)x[i] + (double)(float)y[i]);

        for (int i = 0; i < H; i++) xd[i] = x[i];
        orc_rmsnorm(xd, w->ffn_norm[l], H, m->rms_eps, h);
        orc_q4k_matvec(w->w_gate[l], F, H, h, g);
        orc_q4k_matvec(w->w_up[l], F, H, h, u);
        for (int i = 0; i < F; i++) g[i] = orc_silu((double)(float)g[i]) * (double)(float)u[i];
        orc_q4k_matvec(w->w_down[l], H, F, g, y);
        for (int i = 0; i < H; i++) x[i] = (float)((double)x[i] + (double)(float)y[i]);
        if (hidden) memcpy(hidden + (int64_t)(l + 1) * H, x, (size_t)H * sizeof(float));
    }
    for (int i = 0; i < H; i++) xd[i] = x[i];
    orc_rmsnorm(xd, w->final_norm, H, m->rms_eps, h);
    orc_q4k_matvec(w->embed, m->vocab, H, h, lg);
    for (int64_t i = 0; i < m->vocab; i++) logits[i] = (float)lg[i];
    int64_t id = orc_argmax(logits, m->vocab);

    free(x); free(xd); free(h); free(q); free(k); free(v); free(o);
    free(y); free(g); free(u); free(lg);
    return id;
}

/* A batch of B sequences.  Each row is computed on its own, so the batch
 * result equals B independent single-sequence steps by construction. */
void orc_decode_step(const orc_desc *m, const orc_weights *w, orc_kv *kv, int B,
                     const int32_t *tokens, const int32_t *positions,
                     float *logits, int32_t *ids, float *hidden) {
    for (int b = 0; b < B; b++) {
        float *hb = hidden ? hidden + (int64_t)b * (m->n_layers + 1) * m->hidden : NULL;
        ids[b] = (int32_t)orc_decode_one(m, w, kv + b, tokens[b], positions[b],
                                         logits + (int64_t)b * m->vocab, hb);
    }
}

/* Bulk append of already-rotated fp16 K/V rows ([n_layers][n][n_kv][hd]) at
 * tokens t0..t0+n-1 of one sequence; Q8_0 tensors quantize each 32-block,
 * FP8 tensors convert each value. */
void orc_kv_append(const orc_desc *m, orc_kv *kv, int64_t t0, int64_t n,
                   const uint16_t *k16, const uint16_t *v16) {
    int hd = m->head_dim, nkv = m->n_kv_heads;
    for (int l = 0; l < m->n_layers; l++)
        for (int64_t t = 0; t < n; t++)
            for (int g = 0; g < nkv; g++) {
                int64_t src = (((int64_t)l * n + t) * nkv + g) * hd;
                int64_t row = (((int64_t)l * kv->max_L + t0 + t) * nkv + g);
                orc_kv_put_row(kv, 0, hd, row, k16 + src);
                orc_kv_put_row(kv, 1, hd, row, v16 + src);
            }
}
