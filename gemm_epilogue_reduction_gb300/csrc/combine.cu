// combine.cu -- the record combine: shard-local completion, then the cross-shard merge.
//
// "SemBridge: Compiling Consumer Observations into Cross-Stack Communication Plans",
// Section 5.2 and Figure 1: full-logit transfer rebuilds the complete logits with an
// AllGather and then applies argmax; source projection applies argmax per TP lane
// ("argmax x k") and ships int32 IDs.  Here the k lane shards are on one device, and the
// step that replaces "AllGather, then argmax" merges compact records instead of logits.
//
// A record (m, i, s) of a column set C holds m = max_C y, i = the lowest column attaining
// m, s = sum_C exp(y - m).  The merge of two records keeps the larger max, the lower index
// on an equal max, and rescales both sums to the new max.  It is commutative bit for bit;
// its associativity holds only up to rounding, so the order is fixed:
//   per (row, shard): lane l of one warp folds tiles l, l+32, ... in ascending order, then
//                     an xor butterfly (16, 8, 4, 2, 1) merges the 32 lane results;
//   per row:          the k shard results merge in ascending shard order.
// The output bits are therefore a function of the record bits alone (any grid, any run).
#include <climits>

#include "sb_internal.h"

namespace sb {
namespace {

struct Rec {
    float m;
    int i;
    float s;
};
struct GRec {
    float k;
    int i;
    float z;
};

__device__ __forceinline__ Rec merge(const Rec &a, const Rec &b) {
    Rec r;
    r.m = fmaxf(a.m, b.m);
    r.i = (a.m > b.m) ? a.i : ((b.m > a.m) ? b.i : min(a.i, b.i));
    const float sa = (a.m == -INFINITY) ? 0.f : a.s * expf(a.m - r.m);
    const float sb = (b.m == -INFINITY) ? 0.f : b.s * expf(b.m - r.m);
    r.s = sa + sb;
    return r;
}

__device__ __forceinline__ GRec gmerge(const GRec &a, const GRec &b) {
    return (a.k > b.k || (a.k == b.k && a.i < b.i)) ? a : b;
}

template <bool GUMBEL>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= p.M) return;
    Rec acc{-INFINITY, INT_MAX, 0.f};
    GRec gacc{-INFINITY, INT_MAX, 0.f};
    for (int sh = 0; sh < p.k; ++sh) {
        Rec r{-INFINITY, INT_MAX, 0.f};
        GRec g{-INFINITY, INT_MAX, 0.f};
        const size_t base = (static_cast<size_t>(row) * p.k + sh) * p.T;
        for (int t = lane; t < p.T; t += 32) {
            const Rec x{__ldg(p.ws.m + base + t), __ldg(p.ws.idx + base + t),
                        __ldg(p.ws.s + base + t)};
            r = merge(r, x);
            if (GUMBEL) {
                const GRec y{__ldg(p.ws.gk + base + t), __ldg(p.ws.gi + base + t),
                             __ldg(p.ws.gz + base + t)};
                g = gmerge(g, y);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const Rec o{__shfl_xor_sync(0xFFFFFFFFu, r.m, off),
                        __shfl_xor_sync(0xFFFFFFFFu, r.i, off),
                        __shfl_xor_sync(0xFFFFFFFFu, r.s, off)};
            r = merge(r, o);
            if (GUMBEL) {
                const GRec go{__shfl_xor_sync(0xFFFFFFFFu, g.k, off),
                              __shfl_xor_sync(0xFFFFFFFFu, g.i, off),
                              __shfl_xor_sync(0xFFFFFFFFu, g.z, off)};
                g = gmerge(g, go);
            }
        }
        acc = merge(acc, r);
        if (GUMBEL) gacc = gmerge(gacc, g);
    }
    if (lane == 0) {
        const float lse = acc.m + logf(acc.s);
        p.token[row] = GUMBEL ? gacc.i : acc.i;
        if (p.lse) p.lse[row] = lse;
        if (p.token_logprob) p.token_logprob[row] = GUMBEL ? gacc.z * p.inv_t - lse : -logf(acc.s);
        if (p.target_logprob) {
            const float tz = p.ws.tz[row];
            p.target_logprob[row] = (GUMBEL ? tz * p.inv_t : tz) - lse;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
    constexpr int kRowsPerBlock = 8;
    const int grid = (p.M + kRowsPerBlock - 1) / kRowsPerBlock;
    if (p.flags & kFlagGumbel)
        combine_kernel<true><<<grid, 32 * kRowsPerBlock, 0, stream>>>(p);
    else
        combine_kernel<false><<<grid, 32 * kRowsPerBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sb
