// Device-side noise generator: a counter-based murmur3 fmix32 hash evaluated
// inline, never materialised (the generator family of "RandOpt Speedrun",
// section "What was slow, and the fix"), mapped to Rademacher signs or to
// Gaussians by Box-Muller on two hash words. The exact definition is spelled
// out in include/dust.h.
//
// Fast path structure. fmix32's first step is h ^= h >> 16. With
// h = key ^ n that step distributes over the xor:
//     (key ^ n) ^ ((key ^ n) >> 16) = (key ^ (key >> 16)) ^ (n ^ (n >> 16)),
// so callers pre-fold the per-draw key once (kf) and the per-element counter
// once (nf) and each element-draw starts at the first multiplication.
#pragma once
#include <cstdint>

namespace dust {

constexpr uint32_t kMix1 = 0x85ebca6bu;  // MurmurHash3 fmix32 multipliers
constexpr uint32_t kMix2 = 0xc2b2ae35u;
constexpr uint32_t kWeyl = 0x9E3779B9u;  // floor(2^32 / golden ratio)

__host__ __device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= kMix1;
    h ^= h >> 13;
    h *= kMix2;
    h ^= h >> 16;
    return h;
}

__host__ __device__ __forceinline__ uint32_t fold16(uint32_t x) { return x ^ (x >> 16); }

__host__ __device__ __forceinline__ uint32_t seed_key(uint64_t seed) {
    return fmix32(static_cast<uint32_t>(seed) ^ fmix32(static_cast<uint32_t>(seed >> 32) + kWeyl));
}

// Key of draw i (absolute index), word stream s.
__host__ __device__ __forceinline__ uint32_t draw_key(uint32_t skey, int64_t i, uint32_t s) {
    uint32_t m = static_cast<uint32_t>(2 * i) + s;
    return fmix32(skey ^ (m * kWeyl));
}

// Base draw and sign of draw i under the antithetic mapping.
__host__ __device__ __forceinline__ int64_t base_draw(int64_t i, bool anti) {
    return anti ? (i >> 1) : i;
}

// Full word from a pre-folded key kf and pre-folded counter nf.
__device__ __forceinline__ uint32_t word_ff(uint32_t kf, uint32_t nf) {
    uint32_t h = (kf ^ nf) * kMix1;
    h = (h ^ (h >> 13)) * kMix2;
    return h ^ (h >> 16);
}

// Top bit of the word only: fmix32's last xor-shift leaves bit 31 unchanged.
__device__ __forceinline__ uint32_t sign_ff(uint32_t kf, uint32_t nf) {
    uint32_t h = (kf ^ nf) * kMix1;
    h = (h ^ (h >> 13)) * kMix2;
    return h & 0x80000000u;
}

// Bits 9..31 of the final word, as the mantissa of a float in [1, 2):
// (h ^ (h >> 16)) >> 9 == (h >> 9) ^ (h >> 25).
__device__ __forceinline__ float unit_ff(uint32_t kf, uint32_t nf) {
    uint32_t h = (kf ^ nf) * kMix1;
    h = (h ^ (h >> 13)) * kMix2;
    return __uint_as_float(0x3F800000u | ((h >> 9) ^ (h >> 25)));
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Box-Muller radius with its sign folded in: returns -rho, rho =
// sqrt(-2 ln u1), from f0 = 1 + v, v = (w0 >> 9) 2^-23, u1 = 1 - v (exact).
// -2 ln(1 - v) is taken from the hardware log2 where u1 <= 1 - 2^-11 and from
// the first two terms of the Mercator series below that, 2v + v^2 =
// f0^2 - 1 (one fused multiply-add, a single rounding): there the hardware
// log2's absolute error (about 2^-22) would dominate the small result, while
// the series' truncation is below v^2/3 <= 2^-22/3 relative. Above the
// threshold rho >= 1/32, so a 2^-22 log2 error moves rho by at most
// 2 ln2 2^-22 / (2/32) ~ 5.3e-6.
__device__ __forceinline__ float neg_radius(float f0) {
    const float u1 = 2.0f - f0;
    const float q_log = -1.38629436111989061f * lg2_approx(u1);  // -2 ln 2 * log2(u1)
    const float q_ser = fmaf(f0, f0, -1.0f);
    const float q = (f0 < 1.00048828125f) ? q_ser : q_log;  // v < 2^-11
    return -sqrt_approx(q);
}

// Centred Box-Muller angle 2 pi (u2 - 1/2) in [-pi, pi) from f1 = 1 + u2, in
// one fused multiply-add; cos/sin of the shifted angle are the negatives of
// cos/sin(2 pi u2), which neg_radius' sign undoes.
__device__ __forceinline__ float centred_angle(float f1) {
    return fmaf(f1, 6.28318530717958648f, -9.42477796076937972f);
}

// Box-Muller pair for channel pair p: a[p] = rho cos(2 pi u2), a[p+1] = rho
// sin(2 pi u2), evaluated where the hardware sine/cosine are most accurate.
__device__ __forceinline__ void gauss_pair(float f0, float f1, float& a_even, float& a_odd) {
    const float nr = neg_radius(f0);
    float s, c;
    __sincosf(centred_angle(f1), &s, &c);
    a_even = nr * c;
    a_odd = nr * s;
}

// Packed Rademacher: 32 signs per word. Bit j of the word at the counter of a
// 32-channel group's first channel is channel (first + j)'s sign, as the
// float sign bit (0: +1).
__device__ __forceinline__ uint32_t packed_sign_bit(uint32_t w, int j) {
    return (w << (31 - j)) & 0x80000000u;
}

// Scalar reference path on the device: value of a_t^(i)[c] (absolute draw i).
// Used by the materialising kernels (noise, jitter) where speed is secondary.
__device__ __forceinline__ float noise_value(int kind, uint32_t skey, int64_t i, uint32_t n,
                                             uint32_t n_pair, bool odd, bool anti) {
    float sgn = 1.0f;
    if (anti) {
        sgn = (i & 1) ? -1.0f : 1.0f;
        i >>= 1;
    }
    if (kind == 0) {
        const uint32_t kf = fold16(draw_key(skey, i, 0));
        const uint32_t sb = sign_ff(kf, fold16(n));
        return sgn * __uint_as_float(0x3F800000u | sb);
    }
    const uint32_t nf = fold16(n_pair);
    const float f0 = unit_ff(fold16(draw_key(skey, i, 0)), nf);
    const float f1 = unit_ff(fold16(draw_key(skey, i, 1)), nf);
    float ae, ao;
    gauss_pair(f0, f1, ae, ao);
    return sgn * (odd ? ao : ae);
}

}  // namespace dust
