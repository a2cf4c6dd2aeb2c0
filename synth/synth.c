/*
 * Seeded synthetic inputs for the EAGLE-2 draft-tree cycle.
 *
 * This module is shared by the oracle side and the CUDA side of the tests and
 * by the benchmark. It holds no arithmetic of the method (no softmax, no
 * top-k, no tree logic): it only turns (seed, stream, counter) into numbers.
 *
 *  - Philox4x32-10, written from its published definition (Salmon, Moraes,
 *    Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11):
 *    two 32x32->64 multiplies per round with multipliers 0xD2511F53 and
 *    0xCD9E8D57, key bumped by the Weyl constants 0x9E3779B9 / 0xBB67AE85,
 *    ten rounds. Key = (seed_lo ^ stream, seed_hi).
 *  - Normal draws: Box-Muller on the first two output words, in double,
 *    u1 = (w0 + 1) 2^-32 in (0, 1], u2 = w1 2^-32.
 *  - A draw is scaled (the "sharpness" knob of the dynamic-trees tutorial
 *    page's widget), rounded to fp32 (RNE) and, for bf16 outputs, to bf16 (RNE).
 *
 * Counters (one Philox call per element; word 0..3 of the counter):
 *   logits     : (token, row, i2, i3)  stream 1 draft, 2 target
 *   q          : (element, 0, 0, 0)    stream 3
 *   k / v      : ((pos*Hkv + h)*d + e, layer, b, 0)  stream 4 / 5
 *   seq params : (b, 0, 0, 0)          stream 6
 *   uniforms   : (j, b, cycle, 0)      stream 7
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox_round(uint32_t c[4], uint32_t k0, uint32_t k1) {
    uint64_t p0 = (uint64_t)PHILOX_M0 * c[0];
    uint64_t p1 = (uint64_t)PHILOX_M1 * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k0;
    uint32_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        philox_round(c, k0, k1);
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    memcpy(out, c, sizeof c);
}

static void draw(uint64_t seed, uint32_t stream, uint32_t c0, uint32_t c1, uint32_t c2,
                 uint32_t c3, uint32_t out[4]) {
    uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t key[2] = {(uint32_t)seed ^ stream, (uint32_t)(seed >> 32)};
    synth_philox4x32_10(ctr, key, out);
}

static double box_muller(uint32_t w0, uint32_t w1) {
    const double two_m32 = 2.3283064365386962890625e-10; /* 2^-32 */
    double u1 = ((double)w0 + 1.0) * two_m32;
    double u2 = (double)w1 * two_m32;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static uint16_t f32_to_bf16(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return 0x7FC0; /* NaN */
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

static void store(void* out, int dtype, int64_t idx, double v) {
    float f = (float)v;
    if (dtype == 0)
        ((float*)out)[idx] = f;
    else
        ((uint16_t*)out)[idx] = f32_to_bf16(f);
}

/* out[i3][i2][i1][i0] = scale * N(0,1) drawn at counter (i0, i1, i2, i3).
 * scale_axis: -1 -> scale[0] for all; 2 -> scale[i2]; 3 -> scale[i3]. */
void synth_normal4(void* out, int dtype, int64_t n0, int64_t n1, int64_t n2, int64_t n3,
                   const float* scale, int scale_axis, uint64_t seed, uint32_t stream) {
    int64_t rows = n1 * n2 * n3;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t i1 = r % n1, i2 = (r / n1) % n2, i3 = r / (n1 * n2);
        double s = scale_axis == 2 ? scale[i2] : scale_axis == 3 ? scale[i3] : scale[0];
        for (int64_t i0 = 0; i0 < n0; ++i0) {
            uint32_t w[4];
            draw(seed, stream, (uint32_t)i0, (uint32_t)i1, (uint32_t)i2, (uint32_t)i3, w);
            store(out, dtype, r * n0 + i0, s * box_muller(w[0], w[1]));
        }
    }
}

/* "Planted" rows: in each row (i1, i2, i3) of an [n3][n2][n1][n0] array, the
 * token chosen by counter (0xFFFFFFFF, i1, i2, i3) gets the logit `value`.
 * Rows whose plant draw w[1] * 2^-32 >= frac are left alone. */
void synth_plant(void* out, int dtype, int64_t n0, int64_t n1, int64_t n2, int64_t n3,
                 double value, double frac, uint64_t seed, uint32_t stream) {
    int64_t rows = n1 * n2 * n3;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t i1 = r % n1, i2 = (r / n1) % n2, i3 = r / (n1 * n2);
        uint32_t w[4];
        draw(seed, stream, 0xFFFFFFFFu, (uint32_t)i1, (uint32_t)i2, (uint32_t)i3, w);
        if ((double)w[1] * 2.3283064365386962890625e-10 >= frac) continue;
        store(out, dtype, r * n0 + (int64_t)(w[0] % (uint32_t)n0), value);
    }
}

/* K or V rows of one (sequence, layer): positions [pos0, pos1) of a region
 * whose position p starts at base + p*pos_stride (elements), heads of d
 * contiguous elements each. Counter ((p*Hkv + h)*d + e, layer, b, 0). */
void synth_kv_region(void* base, int dtype, int64_t pos_stride, int hkv, int d, int pos0,
                     int pos1, uint32_t layer, uint32_t b, double scale, uint64_t seed,
                     uint32_t stream) {
#pragma omp parallel for schedule(static)
    for (int p = pos0; p < pos1; ++p) {
        for (int h = 0; h < hkv; ++h)
            for (int e = 0; e < d; ++e) {
                uint32_t w[4];
                uint32_t c0 = (uint32_t)(((int64_t)p * hkv + h) * d + e);
                draw(seed, stream, c0, layer, b, 0, w);
                store(base, dtype, (int64_t)p * pos_stride + (int64_t)h * d + e,
                      scale * box_muller(w[0], w[1]));
            }
    }
}

/* Raw 32-bit words: out[i1][i0] = word 0 at counter (i0, i1, c2, 0). */
void synth_words(uint32_t* out, int64_t n0, int64_t n1, uint32_t c2, uint64_t seed,
                 uint32_t stream) {
    for (int64_t i1 = 0; i1 < n1; ++i1)
        for (int64_t i0 = 0; i0 < n0; ++i0) {
            uint32_t w[4];
            draw(seed, stream, (uint32_t)i0, (uint32_t)i1, c2, 0, w);
            out[i1 * n0 + i0] = w[0];
        }
}

/* Per-sequence prefix length and sharpness: counter (b, 0, 0, 0), stream 6.
 * L_b = lmin + w0 mod lspan ; s_b = smin + sspan * w1 2^-32. */
void synth_seq_params(int batch, int lmin, int lspan, double smin, double sspan, uint64_t seed,
                      int32_t* len, float* sharp) {
    for (int b = 0; b < batch; ++b) {
        uint32_t w[4];
        draw(seed, 6, (uint32_t)b, 0, 0, 0, w);
        len[b] = lmin + (int32_t)(lspan > 0 ? w[0] % (uint32_t)lspan : 0);
        sharp[b] = (float)(smin + sspan * ((double)w[1] * 2.3283064365386962890625e-10));
    }
}

int synth_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Uniform words of sampled drafting, one Philox call per four elements:
 * out[(b * k + f) * V + x] = word (x & 3) of Philox4x32-10 at counter
 * (x >> 2, b * k + f, step, cycle), key (seed_lo ^ 10, seed_hi). */
void synth_gumbel_words(uint32_t* out, int B, int k, int V, uint32_t step, uint32_t cycle, uint64_t seed) {
    const int rows = B * k;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int q = 0; 4 * q < V; ++q) {
            uint32_t w[4];
            draw(seed, 10, (uint32_t)q, (uint32_t)r, step, cycle, w);
            for (int i = 0; i < 4 && 4 * q + i < V; ++i) out[(int64_t)r * V + 4 * q + i] = w[i];
        }
    }
}
