/* synth_host.c -- host twin of the seeded input generator, in plain C.
 *
 * The definition lives in ../synth.py (numpy); this file computes the same
 * bits about a hundred times faster, so that the tests and the benchmark's
 * oracle leg can regenerate whole full-size experts on the host.  It draws
 * numbers only: no part of the method.  A CPU test checks it against the
 * numpy definition stream by stream.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, OOPSLA 2014,
 * with the "Mix13" finaliser constants of Vigna's public splitmix64.c):
 *   word(key, i) = mix64(key + (i + 1) * GAMMA)
 * element i uses words 4i..4i+3: twelve 16-bit uniforms from the first three
 * (Irwin-Hall(12), exact in fp32), the fourth marks outliers (low half) and
 * exact zeros (high half).  The value fl32(z * s) is rounded to bf16 (ties to
 * even). */
#include <stdint.h>
#include <string.h>

static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint16_t f32_to_bf16_rne(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    uint64_t r = ((uint64_t)u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return (uint16_t)r;
}

/* bf16 bit patterns of elements start .. start+n-1 of the stream `key`.
 * s_norm / s_out are fl32(sigma) and fl32(sigma * outlier multiple);
 * t_out / t_zero are the 32-bit thresholds (<= 2^32) of the outlier and
 * zero marks.  Returns 0. */
int synth_values_bf16(uint64_t key, int64_t n, float s_norm, float s_out, uint64_t t_out,
                      uint64_t t_zero, int64_t start, uint16_t *out)
{
    for (int64_t e = 0; e < n; ++e) {
        const uint64_t i0 = 4u * (uint64_t)(start + e);
        uint64_t w[4];
        for (int q = 0; q < 4; ++q)
            w[q] = mix64(key + (i0 + (uint64_t)q + 1u) * GAMMA);
        int64_t acc = 0;
        for (int q = 0; q < 3; ++q)
            for (int h = 0; h < 4; ++h)
                acc += (int64_t)((w[q] >> (16 * h)) & 0xFFFFu);
        const int64_t C = 2 * acc - 12 * 65535;
        const float z = (float)C * (1.0f / 131072.0f);
        const int is_out = (w[3] & 0xFFFFFFFFull) < t_out;
        const int is_zero = (w[3] >> 32) < t_zero;
        float v = z * (is_out ? s_out : s_norm);
        if (is_zero)
            v = 0.0f;
        out[e] = f32_to_bf16_rne(v);
    }
    return 0;
}
