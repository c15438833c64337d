/*
 * kvq_synth_host.c -- host build of the seeded synthetic-input generator
 * (definitions in kvq_synth.h).  Plain C, no FMA contraction, so its binary32
 * multiplies round exactly like the device build's __fmul_rn.
 */
#include <stddef.h>
#include <stdint.h>

#include "kvq_synth.h"

/* out[i] = sample at global index index0 + i; an element is an outlier when
 * mask[(index0 + i) % period] is non-zero (mask may be NULL) */
void kvq_synth_fill_f16(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream, int64_t index0,
                        float sigma, const uint8_t *mask, int64_t period, float outlier_mult)
{
    uint64_t key = kvq_synth_key(seed, stream);
    for (int64_t i = 0; i < n; i++) {
        int64_t g = index0 + i;
        float mult = (mask && mask[g % period]) ? outlier_mult : 1.0f;
        out[i] = kvq_synth_normal_f16(key, (uint64_t)g, sigma, mult);
    }
}

/* exactly `count` outlier channels per head: a partial Fisher-Yates shuffle of
 * the D channels of each head; mask is [H][D] */
void kvq_synth_outliers_per_head(uint8_t *mask, int32_t H, int32_t D, int32_t count, uint64_t seed,
                                 uint64_t stream)
{
    uint64_t key = kvq_synth_key(seed, stream);
    int32_t perm[4096];
    for (int32_t h = 0; h < H; h++) {
        for (int32_t d = 0; d < D; d++) { perm[d] = d; mask[(int64_t)h * D + d] = 0; }
        for (int32_t i = 0; i < count && i < D; i++) {
            uint64_t r = kvq_synth_u64(key, (uint64_t)h * 4096u + (uint64_t)i);
            int32_t j = i + (int32_t)(r % (uint64_t)(D - i));
            int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
            mask[(int64_t)h * D + perm[i]] = 1;
        }
    }
}

/* every (head, channel) independently an outlier when its hash falls below
 * threshold (= p * 2^32, computed by the caller) */
void kvq_synth_outliers_bernoulli(uint8_t *mask, int32_t H, int32_t D, uint32_t threshold,
                                  uint64_t seed, uint64_t stream)
{
    uint64_t key = kvq_synth_key(seed, stream);
    for (int64_t i = 0; i < (int64_t)H * D; i++)
        mask[i] = (uint32_t)(kvq_synth_u64(key, (uint64_t)i) >> 32) < threshold ? 1 : 0;
}

/* a Fisher-Yates permutation of [0, n) */
void kvq_synth_permutation(int32_t *out, int64_t n, uint64_t seed, uint64_t stream)
{
    uint64_t key = kvq_synth_key(seed, stream);
    for (int64_t i = 0; i < n; i++) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; i--) {
        int64_t j = (int64_t)(kvq_synth_u64(key, (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}

/* out[i] uniform integer in [lo, hi] */
void kvq_synth_uniform_int(int32_t *out, int64_t n, int32_t lo, int32_t hi, uint64_t seed,
                           uint64_t stream)
{
    uint64_t key = kvq_synth_key(seed, stream);
    uint64_t span = (uint64_t)((int64_t)hi - lo + 1);
    for (int64_t i = 0; i < n; i++) out[i] = lo + (int32_t)(kvq_synth_u64(key, (uint64_t)i) % span);
}

/* the binary16 rounding used by the generator, exported for its own tests */
uint16_t kvq_synth_f32_to_f16_export(float f) { return kvq_synth_f32_to_f16(f); }
