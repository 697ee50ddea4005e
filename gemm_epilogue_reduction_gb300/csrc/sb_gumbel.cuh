// sb_gumbel.cuh -- standard Gumbel noise from a 24-bit uniform, for the Gumbel-max surface.
//
// g = -ln(-ln u) with u = b * 2^-24, b the top 24 bits of a SplitMix64 draw.  The
// inner t = -ln u needs a small *relative* error (g = -ln t turns it into an absolute error
// of g), so it is evaluated without cancellation on both sides of u = 7/8:
//   u <= 7/8:  t = -ln2 * log2(u) with the hardware log2 (absolute error about 2^-22.6 in
//              log2 u), and t >= 0.1335, so the relative error of t stays below 1e-6;
//   u >  7/8:  with x = 1 - u = (2^24 - b) * 2^-24 exactly in (0, 1/8), the series
//              -ln(1 - x) = x + x^2/2 + ... + x^7/7, whose truncation error is below
//              x^8/8 / (1 - x) <= x^8/7, i.e. below x^7/7 < 7e-8 relative.
// The outer logarithm only needs a small absolute error and uses the hardware log2 as well.
// b = 0 (u = 0) gives g = -infinity, a key that never wins.
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
    const float u = static_cast<float>(b) * 5.9604644775390625e-8f;  // exact
    const float t_lg = -kLn2 * lg2_approx(u);
    // x = 1 - u is exact wherever it is used (u > 7/8: Sterbenz), so it needs no second
    // integer-to-float conversion
    const float x = 1.0f - u;
    float poly = 1.0f / 7.0f;
    poly = fmaf(poly, x, 1.0f / 6.0f);
    poly = fmaf(poly, x, 1.0f / 5.0f);
    poly = fmaf(poly, x, 1.0f / 4.0f);
    poly = fmaf(poly, x, 1.0f / 3.0f);
    poly = fmaf(poly, x, 1.0f / 2.0f);
    poly = fmaf(poly, x, 1.0f);
    const float t = b > 14680064u ? x * poly : t_lg;  // 14680064 = 7/8 * 2^24
    // b = 0: log2(0) = -inf, so t = +inf and g = -inf with no special case
    return -kLn2 * lg2_approx(t);
}

}  // namespace sb
