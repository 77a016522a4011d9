/*
 * synth.c -- seeded synthetic inputs shared by the oracle tests and the GPU
 * path: random numbers, Gaussian draws, fp16 rounding, and the Q4_K
 * quantizer that turns Gaussian weights into canonical Q4_K blocks.
 *
 * None of the decode step's arithmetic lives here.  Weights reach the
 * library already quantized (the library only ever unpacks Q4_K), so the
 * quantizer is part of building the synthetic model, not of the hot path.
 * The KV cache quantizer (Q8_0), which the hot path does run, is NOT here.
 *
 * Counter-based generator: every value is a pure function of
 * (seed, stream, index), so any slice of any tensor can be regenerated
 * independently and in parallel.  The mixer is the splitmix64 finaliser
 * (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t syn_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* 64 random bits for element `index` of stream `stream` under `seed`. */
uint64_t synth_bits(uint64_t seed, uint64_t stream, uint64_t index) {
    uint64_t key = syn_mix(seed * SYN_GOLDEN + 0x632BE59BD9B4E019ull)
                 ^ syn_mix(stream * 0xD1B54A32D192ED03ull + SYN_GOLDEN);
    return syn_mix(key + (index + 1) * SYN_GOLDEN);
}

/* Uniform double in the open interval (0, 1). */
static inline double syn_u01(uint64_t bits) {
    return ((double)(bits >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal for element `index`: Box-Muller on the uniform pair
 * (2p, 2p+1), p = index/2; even indices take the cosine branch and odd
 * indices the sine branch. */
static inline double syn_normal(uint64_t seed, uint64_t stream, uint64_t index) {
    uint64_t p = index >> 1;
    double u1 = syn_u01(synth_bits(seed, stream, 2 * p));
    double u2 = syn_u01(synth_bits(seed, stream, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925 * u2;
    return (index & 1) ? r * sin(a) : r * cos(a);
}

/* fp32 -> IEEE binary16 bits, round to nearest, ties to even.  Overflow
 * goes to +-inf, NaN stays NaN (quiet). */
uint16_t synth_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u)                          /* inf or NaN */
        return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0u));
    if (ax >= 0x477FF000u)                          /* rounds past 65504 */
        return (uint16_t)(sign | 0x7C00u);
    int e = (int)(ax >> 23) - 127;                  /* unbiased exponent */
    uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;   /* 24-bit significand */
    if (ax < 0x00800000u) mant = ax & 0x7FFFFFu, e = -126;  /* fp32 subnormal */
    int shift;                                      /* bits dropped from mant */
    uint32_t base;
    if (e >= -14) { shift = 13; base = (uint32_t)(e + 15) << 10; mant &= 0x7FFFFFu; }
    else {
        shift = 13 + (-14 - e);                     /* half subnormal */
        base = 0;
        if (shift > 24) return (uint16_t)sign;      /* below half the smallest subnormal */
    }
    uint32_t kept = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u);
    uint32_t halfway = 1u << (shift - 1);
    uint32_t h = base + kept;
    if (rem > halfway || (rem == halfway && (kept & 1u))) h += 1;  /* carries into exponent correctly */
    return (uint16_t)(sign | h);
}

float synth_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu, x;
    if (e == 0x1F) x = sign | 0x7F800000u | (m << 13);
    else if (e != 0) x = sign | ((e + 112u) << 23) | (m << 13);
    else if (m == 0) x = sign;
    else {                                           /* subnormal: normalise */
        int s = 0;
        while (!(m & 0x400u)) { m <<= 1; s++; }
        x = sign | ((uint32_t)(113 - s) << 23) | ((m & 0x3FFu) << 13);
    }
    float f;
    memcpy(&f, &x, 4);
    return f;
}

/* n Gaussian floats N(mean, std^2), elements [offset, offset+n) of a stream. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double mean, double std, float *out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        out[i] = (float)(mean + std * syn_normal(seed, stream, offset + (uint64_t)i));
}

/* n Gaussian values N(0, std^2) rounded to fp16 (via fp32, both round to nearest even). */
void synth_normal_f16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double std, uint16_t *out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        out[i] = synth_f32_to_f16((float)(std * syn_normal(seed, stream, offset + (uint64_t)i)));
}

/* n integers uniform in [0, range). */
void synth_uniform_int(uint64_t seed, uint64_t stream, int64_t n, uint32_t range, int32_t *out) {
    for (int64_t i = 0; i < n; i++) {
        uint64_t b = synth_bits(seed, stream, (uint64_t)i) >> 32;
        out[i] = (int32_t)((b * (uint64_t)range) >> 32);
    }
}

/* ---------------------------------------------------------------- Q4_K --
 * Canonical Q4_K block, 144 bytes for 256 weights:
 *   [0:2]   d    (fp16, little endian)   super-block scale of the scales
 *   [2:4]   dmin (fp16)                  super-block scale of the mins
 *   [4:16]  16 six-bit fields: field i occupies bits 6i..6i+5 of the
 *           little-endian 96-bit word; fields 0..7 are the sub-block scales
 *           sc_0..sc_7, fields 8..15 the sub-block mins m_0..m_7
 *   [16:144] 256 four-bit codes: byte t holds element 2t in its low nibble
 *           and element 2t+1 in its high nibble
 * Element i of the block, in sub-block j = i/32, stands for
 *   w = (d*sc_j)*q_i - (dmin*m_j).
 */
static void syn_q4k_pack(uint16_t d, uint16_t dmin, const int sc[8], const int mn[8],
                         const uint8_t q[256], uint8_t *blk) {
    blk[0] = (uint8_t)(d & 0xFF); blk[1] = (uint8_t)(d >> 8);
    blk[2] = (uint8_t)(dmin & 0xFF); blk[3] = (uint8_t)(dmin >> 8);
    memset(blk + 4, 0, 12);
    for (int i = 0; i < 16; i++) {
        uint32_t v = (uint32_t)(i < 8 ? sc[i] : mn[i - 8]) & 63u;
        int bit = 6 * i;
        for (int b = 0; b < 6; b++, bit++)
            if (v & (1u << b)) blk[4 + bit / 8] |= (uint8_t)(1u << (bit % 8));
    }
    for (int t = 0; t < 128; t++)
        blk[16 + t] = (uint8_t)((q[2 * t] & 15u) | ((q[2 * t + 1] & 15u) << 4));
}

static inline int syn_clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Min/max Q4_K quantizer for one 256-weight super-block.  Per sub-block j
 * of 32: lo_j = min(0, min x), s_j = (max x - lo_j)/15, mn_j = -lo_j.
 * d = fp16(max_j s_j / 63), dmin = fp16(max_j mn_j / 63);
 * sc_j = clamp(rint(s_j/d), 0, 63), m_j = clamp(rint(mn_j/dmin), 0, 63);
 * q = clamp(rint((x + dmin*m_j)/(d*sc_j)), 0, 15), or 0 where d*sc_j == 0. */
void synth_q4k_quantize_block(const float *x, uint8_t *blk) {
    float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        s[j] = (hi - lo) / 15.0f;
        mn[j] = -lo;
        if (s[j] > smax) smax = s[j];
        if (mn[j] > mmax) mmax = mn[j];
    }
    uint16_t dh = synth_f32_to_f16(smax / 63.0f), mh = synth_f32_to_f16(mmax / 63.0f);
    float d = synth_f16_to_f32(dh), dmin = synth_f16_to_f32(mh);
    int sc[8], m[8];
    uint8_t q[256];
    for (int j = 0; j < 8; j++) {
        sc[j] = d > 0.0f ? syn_clampi((int)rintf(s[j] / d), 0, 63) : 0;
        m[j] = dmin > 0.0f ? syn_clampi((int)rintf(mn[j] / dmin), 0, 63) : 0;
        float step = d * (float)sc[j];
        float off = dmin * (float)m[j];
        for (int i = 0; i < 32; i++) {
            int v = 0;
            if (step > 0.0f) v = syn_clampi((int)rintf((x[32 * j + i] + off) / step), 0, 15);
            q[32 * j + i] = (uint8_t)v;
        }
    }
    syn_q4k_pack(dh, mh, sc, m, q, blk);
}

/* Quantize n_blocks consecutive super-blocks of x into canonical blocks. */
void synth_q4k_quantize(const float *x, int64_t n_blocks, uint8_t *out) {
    #pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n_blocks; b++)
        synth_q4k_quantize_block(x + 256 * b, out + 144 * b);
}

/* A rows x cols Gaussian N(0, std^2) matrix (row-major element index
 * r*cols + c within `stream`), quantized to canonical Q4_K blocks without
 * materialising the fp32 matrix.  cols must be a multiple of 256. */
void synth_q4k_matrix(uint64_t seed, uint64_t stream, int64_t rows, int64_t cols,
                      double std, uint8_t *out) {
    int64_t nb = cols / 256, total = rows * nb;
    #pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < total; b++) {
        float x[256];
        uint64_t base = (uint64_t)b * 256u;   /* == r*cols + sb*256 */
        for (int i = 0; i < 256; i++) {
            uint64_t idx = base + (uint64_t)i;
            x[i] = (float)(std * syn_normal(seed, stream, idx));
        }
        synth_q4k_quantize_block(x, out + 144 * b);
    }
}
