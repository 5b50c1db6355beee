/*
 * Seeded, counter-based synthetic inputs, shared by the CPU oracle's tests and
 * the CUDA path's tests and benchmark.  Nothing here is part of the optimizer
 * step: this header only turns (key, element index) into an input value.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the finaliser constants are the published
 * ones).  Output word j of element n under key k is
 *     mix64(k + GAMMA * (3 n + j + 1))        j = 0, 1, 2,
 * i.e. the (3n+j+1)-th state of a SplitMix64 stream seeded at k, so any
 * element can be regenerated alone, on the host or on the device.
 *
 * Approximate normal: the Irwin-Hall sum of twelve uniforms minus six (the
 * classical "sum of 12 uniforms" generator; mean 0, variance 1, support
 * [-6, 6]).  The twelve uniforms are the 16-bit quarters of the three words,
 * each taken at the centre of its cell, (k + 1/2) / 2^16.  Every step up to
 * the final scale is exact in double, so host and device agree bit for bit:
 *     z = (sum_of_quarters + 6) / 65536 - 6          (exact)
 *     x = fl64(z * sigma)                             (one IEEE rounding)
 *     f = fl32(x)  (round to nearest even)            [bf16: fl_bf16(f), RNE]
 * Outliers: a second key selects elements with probability thr / 2^24
 * (top 24 bits of one SplitMix64 word below thr); those use sigma_out.
 */
#ifndef SYNTH_GEN_H
#define SYNTH_GEN_H

#include <stdint.h>

#ifdef __CUDACC__
#define SYN_FN __host__ __device__ __forceinline__ static
#else
#define SYN_FN static inline
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

SYN_FN uint64_t syn_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

SYN_FN uint64_t syn_word(uint64_t key, uint64_t n, uint64_t j) {
    return syn_mix64(key + SYN_GAMMA * (3ULL * n + j + 1ULL));
}

/* Irwin-Hall(12) - 6, exact in double. */
SYN_FN double syn_normal(uint64_t key, uint64_t n) {
    uint64_t s = 0;
    for (uint64_t j = 0; j < 3; ++j) {
        uint64_t w = syn_word(key, n, j);
        s += (w & 0xFFFFULL) + ((w >> 16) & 0xFFFFULL) + ((w >> 32) & 0xFFFFULL) + (w >> 48);
    }
    return ((double)s + 6.0) * (1.0 / 65536.0) - 6.0;
}

/* 1 when element n is an outlier under key_out (probability thr / 2^24). */
SYN_FN int syn_is_outlier(uint64_t key_out, uint64_t n, uint32_t thr) {
    if (thr == 0) return 0;
    uint64_t w = syn_mix64(key_out + SYN_GAMMA * (n + 1ULL));
    return (uint32_t)(w >> 40) < thr;
}

typedef struct {
    uint64_t key;       /* stream key of the normal draw            */
    uint64_t key_out;   /* stream key of the outlier selection      */
    uint32_t thr;       /* outlier threshold out of 2^24 (0 = none) */
    uint32_t pad_;
    double sigma;       /* scale of ordinary elements               */
    double sigma_out;   /* scale of outlier elements                */
} syn_stream_t;

SYN_FN double syn_value(const syn_stream_t* st, uint64_t n) {
    double z = syn_normal(st->key, n);
    double s = syn_is_outlier(st->key_out, n, st->thr) ? st->sigma_out : st->sigma;
    return z * s;
}

/* fp32 bits -> bf16 bits, round to nearest even (inputs here are finite). */
SYN_FN uint16_t syn_f32bits_to_bf16(uint32_t b) {
    uint32_t r = b + 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(r >> 16);
}

/* fp32 bits -> IEEE half bits, round to nearest even, with subnormal
 * results, overflow to infinity at 65520 and NaN kept quiet. */
SYN_FN uint16_t syn_f32bits_to_f16(uint32_t b) {
    const uint32_t sign = (b >> 16) & 0x8000u;
    const uint32_t a = b & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) return (uint16_t)(sign | (a > 0x7F800000u ? 0x7E00u : 0x7C00u));
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);   /* >= 65520: infinity */
    if (a < 0x38800000u) {                                      /* below 2^-14 */
        if (a < 0x33000000u) return (uint16_t)sign;             /* below 2^-25: zero */
        const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
        const uint32_t shift = 126u - (a >> 23);                /* 14 .. 24 */
        uint32_t q = mant >> shift;
        const uint32_t rem = mant & ((1u << shift) - 1u);
        const uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (q & 1u))) ++q;
        return (uint16_t)(sign | q);
    }
    uint32_t r = a - (112u << 23);                              /* rebias 127 -> 15 */
    r = (r + 0xFFFu + ((r >> 13) & 1u)) >> 13;
    return (uint16_t)(sign | r);
}

#endif /* SYNTH_GEN_H */
