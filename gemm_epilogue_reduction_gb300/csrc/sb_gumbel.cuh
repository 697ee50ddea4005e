// sb_gumbel.cuh -- standard Gumbel noise from a 24-bit uniform, for the Gumbel-max surface.
//
// g = -ln(-ln u) with u = b * 2^-24, b the top 24 bits of a SplitMix64 draw.  It is evaluated
// in base 2: with t2 = -log2 u = (-ln u) / ln 2,
//     g = -ln(ln 2 * t2) = c0 - ln 2 * log2(t2),   c0 = -ln(ln 2),
// so a key y + g is one fused multiply-add on log2(t2) once the constant c0 is set aside; the
// epilogues compare keys less c0 and add c0 back once per record.
// The inner t2 needs a small *relative* error (the outer logarithm turns it into an absolute
// error of g), so it is evaluated without cancellation on both sides of u = 7/8:
//   u <= 7/8:  t2 = -log2 u with the hardware log2 (absolute error about 2^-22.6), and
//              |log2 u| >= 0.1926, so the relative error of t2 stays below 1e-6;
//   u >  7/8:  with x = 1 - u = (2^24 - b) * 2^-24 exactly in (0, 1/8), the series
//              -ln(1 - x) = x + x^2/2 + ... + x^7/7 times log2(e), whose truncation error is
//              below x^8/8 / (1 - x) <= x^8/7, i.e. below x^7/7 < 7e-8 relative.
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

constexpr float kGumbelC0 = 0.36651292058166435f;  // -ln(ln 2)

// y + g - c0 for the 24-bit uniform b: the key less the constant c0.
__device__ __forceinline__ float gumbel_key_less_c0(float y, uint32_t b) {
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kL2e = 1.4426950408889634f;
    const float uf = static_cast<float>(b);                  // exact (b < 2^24)
    const float L = lg2_approx(uf * 5.9604644775390625e-8f);  // log2 u, u = b 2^-24 exact
    const float x = fmaf(uf, -5.9604644775390625e-8f, 1.0f);  // 1 - u, exact where used
    // -t2 = -log2(e) (x + x^2/2 + ... + x^7/7) by Horner (negated coefficients)
    float q = -kL2e / 7.0f;
    q = fmaf(q, x, -kL2e / 6.0f);
    q = fmaf(q, x, -kL2e / 5.0f);
    q = fmaf(q, x, -kL2e / 4.0f);
    q = fmaf(q, x, -kL2e / 3.0f);
    q = fmaf(q, x, -kL2e / 2.0f);
    q = fmaf(q, x, -kL2e);
    const float t2n = b > 14680064u ? x * q : L;  // -t2 <= 0; 14680064 = 7/8 * 2^24
    // b = 0: log2(0) = -inf, so t2 = +inf and the key is -inf with no special case
    return fmaf(-kLn2, lg2_approx(fabsf(t2n)), y);
}

// The standard Gumbel noise g itself (c0 folded into the same fused multiply-add).
__device__ __forceinline__ float gumbel_from_bits(uint32_t b) {
    return gumbel_key_less_c0(kGumbelC0, b);
}

}  // namespace sb
