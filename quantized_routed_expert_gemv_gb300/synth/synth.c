/*
 * synth.c -- seeded synthetic inputs for the MoE FFN layer.
 *
 * This file only DRAWS data (codes, bf16 scales and biases, bf16 hidden
 * states) and lays it out in the library's record format.  It holds none of
 * the layer's arithmetic (no dequantisation, routing, FFN or combine), so
 * the CUDA library and the fp64 oracle can both be fed from it.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used counter-style: the i-th draw of a
 * stream with key K is mix(K + (i+1)*0x9E3779B97F4A7C15), where mix is the
 * SplitMix64 output function.  Every value therefore depends only on
 * (key, index), so any expert of any layer can be regenerated on its own.
 *
 *   uniform in [0,1):   (draw >> 11) * 2^-53
 *   normal N(mu, sd):   Box-Muller, cosine branch, from draws 2i and 2i+1:
 *                       mu + sd * sqrt(-2 ln(1 - u1)) * cos(2 pi u2)
 *   to bf16:            round-to-nearest-even from double to 8 significant
 *                       bits, done with exact double operations
 *   code bytes:         the little-endian bytes of successive draws, so every
 *                       4-bit (or 8-bit) code is uniform over its range
 *
 * Keys: key(seed, tag, a, b, c) chains mix() over the five words.  Tags name
 * the tensor (expert codes, expert scales, expert biases, router codes, ...);
 * a/b/c carry layer, expert, token or attempt numbers.
 *
 * Record format (the library's; re-derived here, not shared):
 *   [gate codes F x H/2][up codes F x H/2][down codes H x F/2]
 *   [gate sb F x H/64][up sb F x H/64][down sb H x F/64], stride rounded
 *   up to 4096 bytes, sb word = bf16 scale | (bf16 bias << 16).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ull

static uint64_t mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t k = mix(seed + GAMMA);
    k = mix(k ^ (tag + GAMMA));
    k = mix(k ^ (a + 2 * GAMMA));
    k = mix(k ^ (b + 3 * GAMMA));
    k = mix(k ^ (c + 4 * GAMMA));
    return k;
}

uint64_t synth_draw(uint64_t key, uint64_t i) { return mix(key + (i + 1) * GAMMA); }

static double uni(uint64_t key, uint64_t i)
{
    return (double)(synth_draw(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

static double normal(uint64_t key, uint64_t i)
{
    double u1 = uni(key, 2 * i), u2 = uni(key, 2 * i + 1);
    return sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586 * u2);
}

uint16_t synth_bf16_from_double(double v)
{
    if (v == 0.0 || v != v)
        return (v != v) ? 0x7FC0 : (signbit(v) ? 0x8000 : 0x0000);
    int e;
    double m = frexp(fabs(v), &e);     /* |v| = m 2^e, m in [0.5, 1) */
    double t = nearbyint(ldexp(m, 8)); /* 8 significant bits, ties to even */
    double r = ldexp(t, e - 8);
    float f = (float)(v < 0 ? -r : r); /* exact: 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(bits >> 16);
}

void synth_fill_bytes(uint64_t key, uint8_t *out, size_t n)
{
    size_t words = n / 8;
    for (size_t i = 0; i < words; ++i) {
        uint64_t v = synth_draw(key, i);
        for (int b = 0; b < 8; ++b)
            out[8 * i + b] = (uint8_t)(v >> (8 * b));
    }
    if (n % 8) {
        uint64_t v = synth_draw(key, words);
        for (size_t b = 0; b < n % 8; ++b)
            out[8 * words + b] = (uint8_t)(v >> (8 * b));
    }
}

void synth_fill_bf16_uniform(uint64_t key, uint16_t *out, size_t n, double lo, double hi)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = synth_bf16_from_double(lo + (hi - lo) * uni(key, i));
}

void synth_fill_bf16_normal(uint64_t key, uint16_t *out, size_t n, double mu, double sd)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = synth_bf16_from_double(mu + sd * normal(key, i));
}

void synth_fill_f64_uniform(uint64_t key, double *out, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = uni(key, i);
}

void synth_fill_f64_normal(uint64_t key, double *out, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = normal(key, i);
}

/* sb words: scale ~ U[slo, shi] -> bf16, bias ~ N(0, bsd) -> bf16 */
static void fill_sb(uint64_t kscale, uint64_t kbias, uint32_t *out, size_t n, double slo,
                    double shi, double bsd)
{
    for (size_t i = 0; i < n; ++i) {
        uint16_t s = synth_bf16_from_double(slo + (shi - slo) * uni(kscale, i));
        uint16_t b = synth_bf16_from_double(bsd * normal(kbias, i));
        out[i] = (uint32_t)s | ((uint32_t)b << 16);
    }
}

enum { TAG_CODES = 1, TAG_SCALE = 2, TAG_BIAS = 3, TAG_RCODES = 4, TAG_RSCALE = 5,
       TAG_RBIAS = 6 };

uint64_t synth_record_stride(int H, int F)
{
    uint64_t h = (uint64_t)H, f = (uint64_t)F;
    uint64_t bytes = 3 * (f * h / 2) + 3 * (f * h / 64) * 4;
    return (bytes + 4095u) / 4096u * 4096u;
}

/* One expert record (expert index e; the shared expert uses e = E) of
 * layer `layer` drawn from `seed`: codes uniform 0..15, scale U[slo,shi],
 * bias N(0,bsd), all rounded to bf16.  rec must hold synth_record_stride
 * bytes; the padding is zeroed. */
void synth_expert_record(uint64_t seed, int layer, int e, int H, int F, double slo,
                         double shi, double bsd, uint8_t *rec)
{
    uint64_t h = (uint64_t)H, f = (uint64_t)F;
    uint64_t codes = 3 * (f * h / 2);
    uint64_t nsb = 3 * (f * h / 64);
    uint64_t stride = synth_record_stride(H, F);
    synth_fill_bytes(synth_key(seed, TAG_CODES, (uint64_t)layer, (uint64_t)e, 0), rec, codes);
    fill_sb(synth_key(seed, TAG_SCALE, (uint64_t)layer, (uint64_t)e, 0),
            synth_key(seed, TAG_BIAS, (uint64_t)layer, (uint64_t)e, 0),
            (uint32_t *)(rec + codes), nsb, slo, shi, bsd);
    memset(rec + codes + nsb * 4, 0, stride - codes - nsb * 4);
}

/* Router of layer `layer`: codes uniform 0..255 [E][H], sb [E][H/64]. */
void synth_router(uint64_t seed, int layer, int E, int H, double slo, double shi,
                  double bsd, uint8_t *codes, uint32_t *sb)
{
    synth_fill_bytes(synth_key(seed, TAG_RCODES, (uint64_t)layer, 0, 0), codes,
                     (size_t)E * (size_t)H);
    fill_sb(synth_key(seed, TAG_RSCALE, (uint64_t)layer, 0, 0),
            synth_key(seed, TAG_RBIAS, (uint64_t)layer, 0, 0), sb,
            (size_t)E * (size_t)(H / 64), slo, shi, bsd);
}
