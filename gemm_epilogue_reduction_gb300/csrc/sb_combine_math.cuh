// sb_combine_math.cuh -- the arithmetic of the record merge, with every rounding point
// written out (no contraction into fused multiply-adds), so the merge's output bits follow
// from its input bits by the fixed sequence of fp32 operations below.  Shared by the
// combine kernels and the test hook that exposes their exp and log to a host replica.
#pragma once
#include <climits>
#include <cmath>

namespace sb {

// e^x for x <= 0: the hardware base-2 exponential (flush-to-zero) of x * log2(e), the
// product rounded to fp32 first.
__device__ __forceinline__ float exp_nonpos(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(x, 1.4426950408889634f)));
    return y;
}

// Natural log of the merged exp-sum (CUDA's logf).
__device__ __forceinline__ float log_sum(float s) { return logf(s); }

// A record (m, i, s) of a column set: max, lowest column attaining it, sum of exp(y - m).
struct Rec {
    float m;
    int i;
    float s;
};
// A Gumbel record: best key, its column, the logit there.
struct GRec {
    float k;
    int i;
    float z;
};

// Larger max wins, the lower column on an equal max; both sums are rescaled to the new max
// (a side at -inf contributes 0) and added.  Commutative bit for bit.
__device__ __forceinline__ Rec merge(const Rec &a, const Rec &b) {
    Rec r;
    r.m = fmaxf(a.m, b.m);
    r.i = (a.m > b.m) ? a.i : ((b.m > a.m) ? b.i : min(a.i, b.i));
    const float sa = (a.m == -INFINITY) ? 0.f : __fmul_rn(a.s, exp_nonpos(__fsub_rn(a.m, r.m)));
    const float sb = (b.m == -INFINITY) ? 0.f : __fmul_rn(b.s, exp_nonpos(__fsub_rn(b.m, r.m)));
    r.s = __fadd_rn(sa, sb);
    return r;
}

__device__ __forceinline__ GRec gmerge(const GRec &a, const GRec &b) {
    return (a.k > b.k || (a.k == b.k && a.i < b.i)) ? a : b;
}

// The row's outputs from its merged record: lse = m + log s; the chosen token's log-prob is
// -log s for the argmax (its logit is m), y/T - lse for a Gumbel choice with logit y.
__device__ __forceinline__ float row_lse(const Rec &acc) {
    return __fadd_rn(acc.m, log_sum(acc.s));
}
__device__ __forceinline__ float tempered_minus(float z, float inv_t, float lse) {
    return __fsub_rn(__fmul_rn(z, inv_t), lse);
}

}  // namespace sb
