/*
 * Oracle initialiser: N(0, std^2) draws for the GPT-2 weight init.
 *
 * TEST INFRASTRUCTURE ONLY.  This file belongs to the CPU oracle; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * What it follows: the GPT-2 reproduction ("Let's reproduce GPT-2 (124M)",
 * §Bölümler 2, the nn.Module GPT-2) initialises the 2-D weights from a normal
 * distribution with standard deviation 0.02, scaling the two residual
 * projections by 1/sqrt(2L).  The pages give no generator, so one is written
 * down here from its published definitions and implemented independently on
 * each side:
 *
 *   sm64(x)      SplitMix64 output for generator state x
 *                (Steele, Lea & Flood, OOPSLA 2014);
 *   draw(s,t,c)  sm64(sm64(sm64(s) + t) + c)       (mod 2^64);
 *   u1           ((draw(seed, id, 2i)   >> 11) + 1) * 2^-53   in (0, 1];
 *   u2           ( draw(seed, id, 2i+1) >> 11)      * 2^-53   in [0, 1);
 *   value_i      (float)(std * sqrt(-2 ln u1) * cos(2 pi u2))  (Box-Muller,
 *                cosine branch; the product in double, one rounding to fp32).
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC init_rng.c -lm
 */
#include <math.h>
#include <stdint.h>

static uint64_t splitmix64_out(uint64_t state)
{
    uint64_t z = state + 0x9E3779B97F4A7C15ULL;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

/* SplitMix64 output for generator state x (exported for the published-value pin). */
uint64_t oracle_sm64(uint64_t x)
{
    return splitmix64_out(x);
}

/* One raw draw addressed by (seed, stream, counter). */
uint64_t oracle_draw(uint64_t seed, uint64_t stream, uint64_t counter)
{
    uint64_t key = splitmix64_out(splitmix64_out(seed) + stream);
    return splitmix64_out(key + counter);
}

/* Fill out[0..n) with fp32-rounded N(0, std^2) draws of tensor `stream`. */
void oracle_normal_fill(uint64_t seed, uint64_t stream, int64_t n, double std, float *out)
{
    const double two_pi = 6.283185307179586;   /* 2*pi rounded to double */
    const double ulp53 = 1.0 / 9007199254740992.0; /* 2^-53 */
    for (int64_t i = 0; i < n; ++i) {
        uint64_t a = oracle_draw(seed, stream, 2 * (uint64_t)i);
        uint64_t b = oracle_draw(seed, stream, 2 * (uint64_t)i + 1);
        double u1 = ((double)(a >> 11) + 1.0) * ulp53;
        double u2 = (double)(b >> 11) * ulp53;
        double radius = sqrt(-2.0 * log(u1));
        double angle = two_pi * u2;
        double z = radius * cos(angle);
        out[i] = (float)(std * z);
    }
}
