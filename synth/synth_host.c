/*
 * Seeded synthetic inputs, host side.
 *
 * This file holds only input generation: no step of the decoding method is
 * computed here.  The same generator is implemented for the device in
 * synth_dev.cu and in numpy in synth/__init__.py; all three give identical
 * bits for the same (key, index).
 *
 * Generator: element i of a tensor with 64-bit key K is the i-th output of a
 * SplitMix64 stream seeded with K (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014): state = K + (i+1)*GAMMA,
 * output = the SplitMix64 finaliser of that state.
 *
 * Approximately normal values: the four 16-bit fields of the output are
 * summed (Irwin-Hall with n = 4 over {0..65535}, exact in integers), centred
 * by subtracting 131070, converted to float (exact, |c| < 2^24) and scaled by
 * ONE IEEE-754 binary32 multiply with a caller-supplied scale.  bf16 output is
 * that float rounded to nearest-even on its upper 16 bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t sm64_at(uint64_t key, uint64_t i) {
    return sm64_mix(key + (i + 1) * SM64_GAMMA);
}

static inline float irwin_hall4(uint64_t u, float scale) {
    int64_t s = (int64_t)(u & 0xFFFF) + (int64_t)((u >> 16) & 0xFFFF) +
                (int64_t)((u >> 32) & 0xFFFF) + (int64_t)(u >> 48);
    float c = (float)(s - 131070); /* exact: |c| < 2^24 */
    return c * scale;              /* the one rounding step */
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

void synth_host_u64(uint64_t key, uint64_t start, int64_t n, uint64_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = sm64_at(key, start + (uint64_t)i);
}

void synth_host_normal_f32(uint64_t key, uint64_t start, int64_t n, float scale, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = irwin_hall4(sm64_at(key, start + (uint64_t)i), scale);
}

void synth_host_normal_bf16(uint64_t key, uint64_t start, int64_t n, float scale, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne(irwin_hall4(sm64_at(key, start + (uint64_t)i), scale));
}

/* float -> FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * largest finite value 448, subnormals m * 2^-9), rounded to nearest-even and
 * saturated to +-448.  Normal range: round the binary32 pattern at its 20th
 * bit (exact integer arithmetic) and rebias the exponent; below 2^-6 the value
 * times 512 (exact) is rounded to an integer mantissa 0..8. */
static inline uint8_t f32_to_e4m3_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    const uint32_t sign = (b >> 31) << 7;
    const uint32_t a = b & 0x7FFFFFFFu;
    uint32_t code;
    if (a >= 0x7F800000u) {
        code = 0x7Eu;
    } else if (a >= 0x3C800000u) { /* |f| >= 2^-6 */
        const uint32_t r = (a + 0x7FFFFu + ((a >> 20) & 1u)) >> 20;
        code = r - (120u << 3);
        if (code > 0x7Eu) code = 0x7Eu;
    } else {
        float m;
        memcpy(&m, &a, 4);
        code = (uint32_t)rintf(m * 512.0f);
    }
    return (uint8_t)(code | sign);
}

/* FP8 E4M3 codes of normal values: round_e4m3(irwin_hall4 * scale). */
void synth_host_e4m3(uint64_t key, uint64_t start, int64_t n, float scale, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3_rne(irwin_hall4(sm64_at(key, start + (uint64_t)i), scale));
}

/* The conversion alone, for checking it on chosen values. */
void synth_host_f32_to_e4m3(const float* in, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3_rne(in[i]);
}

/* Per-row scales (16 + (u & 15)) * 2^-16, exact in binary32. */
void synth_host_row_scales(uint64_t key, uint64_t start, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(16 + (int)(sm64_at(key, start + (uint64_t)i) & 15u)) * 0x1p-16f;
}

/* bf16 bit patterns -> float64, for handing weights to an fp64 consumer. */
void synth_host_bf16_to_f64(const uint16_t* in, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = (uint32_t)in[i] << 16;
        float f;
        memcpy(&f, &b, 4);
        out[i] = (double)f;
    }
}

int synth_host_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
