/*
 * kvq_synth.h -- seeded, counter-based synthetic inputs for the KV-cache
 * workloads (keys, values, queries, block tables, sequence lengths).
 *
 * This module is the one piece shared by the CUDA path and the CPU oracle's
 * tests: it makes inputs and holds none of the quantization or attention
 * arithmetic.  Every value is a pure function of (seed, stream, index), built
 * from integer operations and a fixed sequence of IEEE binary32 multiplies, so
 * the host build (C) and the device build (CUDA) produce identical bits and
 * any sub-range of a tensor can be regenerated on its own.
 *
 * Normal deviates: the sum S of twelve uniform 16-bit integers (Irwin-Hall)
 * centred as (2 S - 12 * 65535) * 2^-17, which has mean 0 and variance
 * 1 - 2^-32 and is bounded by about 6; times sigma, optionally times an
 * outlier multiplier, then rounded to binary16 (round to nearest even).
 * Hash: the splitmix64 output function (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) over a Weyl-sequence counter.
 */
#ifndef KVQ_SYNTH_H
#define KVQ_SYNTH_H

#include <stdint.h>

#ifdef __CUDACC__
#define KVQ_SYNTH_FN __host__ __device__ __forceinline__
#else
#define KVQ_SYNTH_FN static inline
#endif

#define KVQ_SYNTH_GOLDEN 0x9E3779B97F4A7C15ull

KVQ_SYNTH_FN uint64_t kvq_synth_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* key of one stream of one seed */
KVQ_SYNTH_FN uint64_t kvq_synth_key(uint64_t seed, uint64_t stream)
{
    return kvq_synth_mix(kvq_synth_mix(seed + KVQ_SYNTH_GOLDEN) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* the 64-bit hash number i of a stream */
KVQ_SYNTH_FN uint64_t kvq_synth_u64(uint64_t key, uint64_t i)
{
    return kvq_synth_mix(key + (i + 1) * KVQ_SYNTH_GOLDEN);
}

/* centred Irwin-Hall sum of 12 uniform 16-bit integers: an even integer in
 * [-786420, 786420] whose value * 2^-17 is approximately N(0, 1) */
KVQ_SYNTH_FN int32_t kvq_synth_ih12(uint64_t key, uint64_t index)
{
    int32_t s = 0;
    for (int i = 0; i < 3; i++) {
        uint64_t h = kvq_synth_u64(key, 3 * index + (uint64_t)i);
        s += (int32_t)(h & 0xffff) + (int32_t)((h >> 16) & 0xffff) + (int32_t)((h >> 32) & 0xffff) +
             (int32_t)(h >> 48);
    }
    return 2 * s - 12 * 65535;
}

typedef union {
    float f;
    uint32_t u;
} kvq_synth_fu;

/* binary32 -> binary16, round to nearest even, overflow to infinity */
KVQ_SYNTH_FN uint16_t kvq_synth_f32_to_f16(float f)
{
    kvq_synth_fu c;
    c.f = f;
    uint32_t x = c.u;
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);   /* >= 65520 rounds to infinity */
    if (ax <= 0x33000000u) return (uint16_t)sign;               /* <= 2^-25 rounds to zero */
    uint32_t e = ax >> 23;
    uint32_t m = ax & 0x7fffffu;
    if (e < 113u) {                                            /* binary16 subnormal */
        m |= 0x800000u;
        uint32_t shift = 126u - e;                             /* 14 .. 24 */
        uint32_t r = m >> shift;
        uint32_t rem = m & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (r & 1u))) r++;
        return (uint16_t)(sign | r);
    }
    uint32_t r = ((e - 112u) << 10) | (m >> 13);
    uint32_t rem = m & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r++;     /* a carry may reach infinity: correct */
    return (uint16_t)(sign | r);
}

#ifdef __CUDA_ARCH__
#define KVQ_SYNTH_MUL(a, b) __fmul_rn((a), (b))
#else
#define KVQ_SYNTH_MUL(a, b) ((a) * (b))
#endif

/* one fp16 sample: ((ih12 * 2^-17) * sigma) * mult, each product rounded to binary32 */
KVQ_SYNTH_FN uint16_t kvq_synth_normal_f16(uint64_t key, uint64_t index, float sigma, float mult)
{
    float v = KVQ_SYNTH_MUL((float)kvq_synth_ih12(key, index), 7.62939453125e-06f); /* 2^-17, exact */
    v = KVQ_SYNTH_MUL(v, sigma);
    if (mult != 1.0f) v = KVQ_SYNTH_MUL(v, mult);
    return kvq_synth_f32_to_f16(v);
}

#endif /* KVQ_SYNTH_H */
