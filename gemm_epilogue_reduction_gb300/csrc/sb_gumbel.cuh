// sb_gumbel.cuh -- standard Gumbel noise from a 24-bit uniform, for the Gumbel-max surface.
//
// g = -ln(-ln u) with u = b * 2^-24, b the top 24 bits of a SplitMix64 draw.  The
// inner t = -ln u needs a small *relative* error (g = -ln t turns it into an absolute error
// of g), so it is evaluated without cancellation on both halves of (0, 1):
//   u < 1/2  (b < 2^23):  t = ln2 * (24 - log2 b), where 24 - log2 b >= 1;
//   u >= 1/2:             with x = 1 - u = (2^24 - b) * 2^-24 exactly in (0, 1/2],
//                         t = -ln(1 - x) = 2 atanh(s), s = x / (2 - x) in (0, 1/3], summed as
//                         the classical odd series 2 (s + s^3/3 + s^5/5 + ... + s^17/17),
//                         whose truncation error is below 2e-10 relative for s <= 1/3.
// The outer logarithm only needs a small absolute error and uses the hardware log2
// approximation.  b = 0 (u = 0) gives g = -infinity, a key that never wins.
#pragma once
#include <cstdint>

namespace sb {

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float gumbel_from_bits(uint32_t b) {
    constexpr float kLn2 = 0.6931471805599453f;
    const float t_lo = kLn2 * (24.0f - lg2_approx(static_cast<float>(b)));
    const float x = static_cast<float>(16777216u - b) * 5.9604644775390625e-8f;
    const float s = __fdividef(x, 2.0f - x);
    const float s2 = s * s;
    float poly = 1.0f / 17.0f;
    poly = fmaf(poly, s2, 1.0f / 15.0f);
    poly = fmaf(poly, s2, 1.0f / 13.0f);
    poly = fmaf(poly, s2, 1.0f / 11.0f);
    poly = fmaf(poly, s2, 1.0f / 9.0f);
    poly = fmaf(poly, s2, 1.0f / 7.0f);
    poly = fmaf(poly, s2, 1.0f / 5.0f);
    poly = fmaf(poly, s2, 1.0f / 3.0f);
    poly = fmaf(poly, s2, 1.0f);
    const float t_hi = 2.0f * s * poly;
    const float t = (b < (1u << 23)) ? t_lo : t_hi;
    const float g = -kLn2 * lg2_approx(t);
    return b == 0u ? -INFINITY : g;
}

}  // namespace sb
