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
//   per (row, shard): lane l of one warp takes tiles l, l+32, ..., l+480 of each batch of 512
//                     and folds them as a balanced pairwise tree (adjacent pairs, four
//                     levels), folds the batch results in ascending order, then an xor
//                     butterfly (16, 8, 4, 2, 1) merges the 32 lane results;
//   per row:          the k shard results merge in ascending shard order.
// One block serves one row; its warps take the shards round-robin.
// The output bits are therefore a function of the record bits alone (any grid, any run).
#include <climits>

#include "sb_combine_math.cuh"
#include "sb_internal.h"

namespace sb {
namespace {

constexpr int kMaxWarps = 8;
constexpr int kBatch = 16;  // records each lane loads before folding them

// Pairwise tree over x[0 .. N): adjacent pairs first, the result in x[0].
template <int N, typename R, typename F>
__device__ __forceinline__ void tree_fold(R (&x)[N], F f) {
#pragma unroll
    for (int w = 1; w < N; w *= 2)
#pragma unroll
        for (int u = 0; u + w < N; u += 2 * w) x[u] = f(x[u], x[u + w]);
}

// Shard-local completion of (row, shard) by one warp in the fixed order above; every lane
// returns the shard record (and the Gumbel record).  on_rec(t, rec) sees each of the lane's
// records (t < T) as it is loaded, in ascending tile order.
template <bool GUMBEL, typename OnRec>
__device__ __forceinline__ void shard_fold(const Workspace &ws, size_t base, int T, int lane,
                                           Rec &r, GRec &g, OnRec on_rec) {
    r = Rec{-INFINITY, INT_MAX, 0.f};
    g = GRec{-INFINITY, INT_MAX, 0.f};
    for (int t0 = lane; t0 < T; t0 += 32 * kBatch) {
        Rec x[kBatch];
        GRec y[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int t = t0 + 32 * u;
            if (t < T) {
                x[u] = Rec{__ldg(ws.m + base + t), __ldg(ws.idx + base + t),
                           __ldg(ws.s + base + t)};
                if (GUMBEL)
                    y[u] = GRec{__ldg(ws.gk + base + t), __ldg(ws.gi + base + t),
                                __ldg(ws.gz + base + t)};
            } else {
                x[u] = Rec{-INFINITY, INT_MAX, 0.f};
                if (GUMBEL) y[u] = GRec{-INFINITY, INT_MAX, 0.f};
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (t0 + 32 * u < T) on_rec(t0 + 32 * u, x[u]);
        tree_fold(x, [](const Rec &a, const Rec &b) { return merge(a, b); });
        r = merge(r, x[0]);
        if (GUMBEL) {
            tree_fold(y, [](const GRec &a, const GRec &b) { return gmerge(a, b); });
            g = gmerge(g, y[0]);
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
}

// One block per row; warp w completes shards w, w + 8, ... (shard_fold), writes the shard
// record to shared memory, and thread 0 merges the k shard records in ascending order.
template <bool GUMBEL>
__global__ void __launch_bounds__(32 * kMaxWarps) combine_kernel(const CombineParams p) {
    extern __shared__ float sh[];  // k records: m, i, s [, gk, gi, gz]
    float *sm = sh;
    int *si = reinterpret_cast<int *>(sh + p.k);
    float *ss = sh + 2 * p.k;
    float *sgk = sh + 3 * p.k;
    int *sgi = reinterpret_cast<int *>(sh + 4 * p.k);
    float *sgz = sh + 5 * p.k;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    // Launched as a programmatic dependent of the GEMM: wait until that grid has completed
    // and its record writes are visible.
    // let the next kernel in the stream (a dependent launch) start its setup early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int sh_i = warp; sh_i < p.k; sh_i += nwarps) {
        Rec r;
        GRec g;
        shard_fold<GUMBEL>(p.ws, (static_cast<size_t>(row) * p.k + sh_i) * p.T, p.T, lane, r, g,
                           [](int, const Rec &) {});
        if (lane == 0) {
            sm[sh_i] = r.m;
            si[sh_i] = r.i;
            ss[sh_i] = r.s;
            if (GUMBEL) {
                sgk[sh_i] = g.k;
                sgi[sh_i] = g.i;
                sgz[sh_i] = g.z;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    Rec acc{-INFINITY, INT_MAX, 0.f};
    GRec gacc{-INFINITY, INT_MAX, 0.f};
    for (int s2 = 0; s2 < p.k; ++s2) {
        acc = merge(acc, Rec{sm[s2], si[s2], ss[s2]});
        if (GUMBEL) gacc = gmerge(gacc, GRec{sgk[s2], sgi[s2], sgz[s2]});
    }
    const float lse = row_lse(acc);
    const int tok = GUMBEL ? gacc.i : acc.i;
    const float tlp = GUMBEL ? tempered_minus(gacc.z, p.inv_t, lse) : -log_sum(acc.s);
    p.token[row] = tok;
    if (p.lse) p.lse[row] = lse;
    if (p.token_logprob) p.token_logprob[row] = tlp;
    if (p.token_host) p.token_host[row] = tok;
    if (p.token_logprob_host) p.token_logprob_host[row] = tlp;
    if (p.target_logprob) {
        const float tz = p.ws.tz[row];
        p.target_logprob[row] = GUMBEL ? tempered_minus(tz, p.inv_t, lse) : __fsub_rn(tz, lse);
    }
}

// ------------------------------------------------------------------ shard payloads
// The record a vocabulary lane would send to the others: its shard-local completion, with
// columns made global by `col_offset`.  Payload layout: lane-major, record (s, r) at
// index s * M + r; 12 bytes (m, idx, s), plus (gkey, gidx, gz) for the Gumbel surface.
struct PayloadParams {
    int M, k, T;
    int gumbel;
    long long col_offset;
    Workspace ws;
    unsigned char *payload;
};

template <bool GUMBEL>
__global__ void __launch_bounds__(32 * kMaxWarps) pack_kernel(const PayloadParams p) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    // let the next kernel in the stream (a dependent launch) start its setup early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int sh_i = warp; sh_i < p.k; sh_i += nwarps) {
        Rec r;
        GRec g;
        shard_fold<GUMBEL>(p.ws, (static_cast<size_t>(row) * p.k + sh_i) * p.T, p.T, lane, r, g,
                           [](int, const Rec &) {});
        if (lane == 0) {
            const size_t rec = static_cast<size_t>(sh_i) * p.M + row;
            float *f = reinterpret_cast<float *>(p.payload + rec * (GUMBEL ? 24 : 12));
            int *i = reinterpret_cast<int *>(f);
            f[0] = r.m;
            i[1] = r.i == INT_MAX ? INT_MAX : static_cast<int>(r.i + p.col_offset);
            f[2] = r.s;
            if (GUMBEL) {
                f[3] = g.k;
                i[4] = g.i == INT_MAX ? INT_MAX : static_cast<int>(g.i + p.col_offset);
                f[5] = g.z;
            }
        }
    }
}

template <bool GUMBEL>
__global__ void merge_payload_kernel(const CombineParams c, const unsigned char *payload) {
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    // let the next kernel in the stream (a dependent launch) start its setup early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row >= c.M) return;
    Rec acc{-INFINITY, INT_MAX, 0.f};
    GRec gacc{-INFINITY, INT_MAX, 0.f};
    for (int s2 = 0; s2 < c.k; ++s2) {
        const size_t rec = static_cast<size_t>(s2) * c.M + row;
        const float *f = reinterpret_cast<const float *>(payload + rec * (GUMBEL ? 24 : 12));
        const int *i = reinterpret_cast<const int *>(f);
        acc = merge(acc, Rec{f[0], i[1], f[2]});
        if (GUMBEL) gacc = gmerge(gacc, GRec{f[3], i[4], f[5]});
    }
    const float lse = row_lse(acc);
    c.token[row] = GUMBEL ? gacc.i : acc.i;
    if (c.lse) c.lse[row] = lse;
    if (c.token_logprob)
        c.token_logprob[row] = GUMBEL ? tempered_minus(gacc.z, c.inv_t, lse) : -log_sum(acc.s);
}

// ------------------------------------------------------------------ top-K helpers
__device__ __forceinline__ uint32_t ord_f(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// K rounds of warp max over the lanes' sorted lists (tv, ti) of KL entries; lane 0
// writes the winners to (ov, oi).  Lanes with nothing hold (-inf, INT_MAX) heads.
template <int KL>
__device__ __forceinline__ void warp_select(const float (&tv)[KL], const int (&ti)[KL],
                                            int K, float *ov, int *oi) {
    const int lane = threadIdx.x & 31;
    int hp = 0;
    for (int q = 0; q < K; ++q) {
        float hv = -INFINITY;
        int hi = INT_MAX;
#pragma unroll
        for (int e = 0; e < KL; ++e)
            if (e == hp) {
                hv = tv[e];
                hi = ti[e];
            }
        const uint32_t oh = ord_f(hv);
        const uint32_t om = __reduce_max_sync(0xFFFFFFFFu, oh);
        const int wi = __reduce_min_sync(0xFFFFFFFFu, oh == om ? hi : INT_MAX);
        if (oh == om && hi == wi && hp < KL) ++hp;
        if (lane == 0) {
            ov[q] = unord_f(om);
            oi[q] = wi;
        }
    }
}

template <int KL>
__device__ __forceinline__ void list_insert(float (&tv)[KL], int (&ti)[KL], float x,
                                            int xi) {
    float cv = x;
    int ci = xi;
    bool ins = false;
#pragma unroll
    for (int q = 0; q < KL; ++q) {
        if (ins || cv > tv[q]) {
            const float a = tv[q];
            const int b = ti[q];
            tv[q] = cv;
            ti[q] = ci;
            cv = a;
            ci = b;
            ins = true;
        }
    }
}

// Block-wide top-K of the threads' sorted lists: each warp picks its K best, then warp 0
// picks the K best of the warps' lists into (ov, oi) in shared memory.
template <int KL>
__device__ __forceinline__ void block_select(const float (&tv)[KL], const int (&ti)[KL],
                                             int K, float *wlv, int *wli, float *ov, int *oi) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    warp_select(tv, ti, K, wlv + warp * K, wli + warp * K);
    __syncthreads();
    if (warp == 0) {
        float lv[KL];
        int li[KL];
#pragma unroll
        for (int q = 0; q < KL; ++q) {
            const bool have = lane < nwarps && q < K;
            lv[q] = have ? wlv[lane * K + q] : -INFINITY;
            li[q] = have ? wli[lane * K + q] : INT_MAX;
        }
        warp_select(lv, li, K, ov, oi);
    }
    __syncthreads();
}

// Rank-aware insertion for entries that arrive in no particular column order: (x, xi) goes
// before the first entry it ranks above (larger value, or an equal value at a lower column).
template <int KL>
__device__ __forceinline__ void list_insert_ranked(float (&tv)[KL], int (&ti)[KL],
                                                   float x, int xi) {
    float cv = x;
    int ci = xi;
    bool ins = false;
#pragma unroll
    for (int q = 0; q < KL; ++q) {
        if (ins || cv > tv[q] || (cv == tv[q] && ci < ti[q])) {
            const float a = tv[q];
            const int b = ti[q];
            tv[q] = cv;
            ti[q] = ci;
            cv = a;
            ci = b;
            ins = true;
        }
    }
}

// Top-K combine, one block per row.
//  1. lse and token: exactly the fixed tree of the plain combine (so they equal the token
//     surface's bits): warps over shards, lanes over tiles, xor butterfly, shards ascending.
//     The same loads feed each lane's list of its best tile maxima, keyed by record number
//     (records are numbered in ascending column order, so the lower record number is the
//     lower column on an equal maximum).
//  2. The block selects the K records with the best maxima.  Every entry of the row's top K
//     lies in one of them: an entry of any other record has K distinct entries (those K
//     maxima) ranking above it.
//  3. One warp reads those K records' sorted lists (K x K entries) and selects the K best.
// Selection compares (value, column) only, so the result does not depend on how the work is
// split.
template <int KL>
__global__ void __launch_bounds__(32 * kMaxWarps) combine_topk_kernel(const CombineParams p) {
    extern __shared__ float sh[];  // k x (m, i, s); 8 x K warp lists; 2 x K block lists
    const int K = p.topk;
    float *sm = sh;
    int *si = reinterpret_cast<int *>(sh + p.k);
    float *ss = sh + 2 * p.k;
    float *wlv = sh + 3 * p.k;
    int *wli = reinterpret_cast<int *>(wlv + kMaxWarps * K);
    float *blv = reinterpret_cast<float *>(wli + kMaxWarps * K);
    int *bli = reinterpret_cast<int *>(blv + K);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int nrec = p.k * p.T;
    const size_t rbase = static_cast<size_t>(row) * nrec;
    // let the next kernel in the stream (a dependent launch) start its setup early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // 1. shard records (the plain combine's tree) and the lanes' best maxima
    float tv[KL];
    int ti[KL];
#pragma unroll
    for (int q = 0; q < KL; ++q) {
        tv[q] = -INFINITY;
        ti[q] = INT_MAX;
    }
    for (int sh_i = warp; sh_i < p.k; sh_i += nwarps) {
        Rec r;
        GRec g;
        const int fbase = sh_i * p.T;
        shard_fold<false>(p.ws, rbase + fbase, p.T, lane, r, g, [&](int t, const Rec &x) {
            if (x.m > tv[KL - 1]) list_insert(tv, ti, x.m, fbase + t);
        });
        if (lane == 0) {
            sm[sh_i] = r.m;
            si[sh_i] = r.i;
            ss[sh_i] = r.s;
        }
    }

    // 2. the K records with the best maxima (record numbers in bli; INT_MAX past the row's
    //    records when it has fewer than K)
    block_select(tv, ti, K, wlv, wli, blv, bli);
    if (warp != 0) return;

    // 3. the K best of those records' lists
#pragma unroll
    for (int q = 0; q < KL; ++q) {
        tv[q] = -INFINITY;
        ti[q] = INT_MAX;
    }
    constexpr int kPer = (KL * KL + 31) / 32;  // entries per lane at the largest K
    float xv[kPer];
    int xi[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int j = lane + 32 * u;
        const int f = j < K * K ? bli[min(j / K, K - 1)] : INT_MAX;
        const bool have = f < nrec;
        const size_t o = have ? (rbase + f) * K + j % K : 0;
        xv[u] = have ? __ldg(p.ws.tkv + o) : -INFINITY;
        xi[u] = have ? __ldg(p.ws.tki + o) : INT_MAX;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u)
        if (xv[u] != -INFINITY) list_insert_ranked(tv, ti, xv[u], xi[u]);
    __syncwarp();
    warp_select(tv, ti, K, wlv, wli);  // warp 0's slot of the warp lists is free again
    __syncwarp();

    Rec acc{-INFINITY, INT_MAX, 0.f};
    for (int s2 = 0; s2 < p.k; ++s2) acc = merge(acc, Rec{sm[s2], si[s2], ss[s2]});
    const float lse = row_lse(acc);
    if (lane < K) {
        p.topk_ids[static_cast<size_t>(row) * K + lane] = wli[lane];
        p.topk_logprob[static_cast<size_t>(row) * K + lane] = wlv[lane] - lse;
    }
    if (lane != 0) return;
    p.token[row] = acc.i;
    if (p.lse) p.lse[row] = lse;
    if (p.token_logprob) p.token_logprob[row] = -log_sum(acc.s);
    if (p.token_host) p.token_host[row] = acc.i;
    if (p.token_logprob_host) p.token_logprob_host[row] = -log_sum(acc.s);
    if (p.target_logprob) p.target_logprob[row] = __fsub_rn(p.ws.tz[row], lse);
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
    const int warps = p.k < kMaxWarps ? p.k : kMaxWarps;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.M);
    cfg.blockDim = dim3(32 * warps);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.k) * ((p.flags & kFlagGumbel) ? 24 : 12);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.flags & kFlagTopk) {
        cfg.blockDim = dim3(32 * kMaxWarps);
        cfg.dynamicSmemBytes = static_cast<size_t>(p.k) * 12 +
                               static_cast<size_t>(kMaxWarps + 1) * 8 * p.topk;
        // lists sized to the smallest of 4, 8, 16 entries that holds K
        if (p.topk <= 4) return cudaLaunchKernelEx(&cfg, combine_topk_kernel<4>, p);
        if (p.topk <= 8) return cudaLaunchKernelEx(&cfg, combine_topk_kernel<8>, p);
        return cudaLaunchKernelEx(&cfg, combine_topk_kernel<kMaxTopK>, p);
    }
    if (p.flags & kFlagGumbel) return cudaLaunchKernelEx(&cfg, combine_kernel<true>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<false>, p);
}

}  // namespace sb

namespace sb {

cudaError_t launch_pack(const Workspace &ws, int M, int k, int T, bool gumbel,
                        long long col_offset, void *payload, cudaStream_t stream) {
    PayloadParams p{};
    p.M = M;
    p.k = k;
    p.T = T;
    p.gumbel = gumbel;
    p.col_offset = col_offset;
    p.ws = ws;
    p.payload = static_cast<unsigned char *>(payload);
    const int warps = k < kMaxWarps ? k : kMaxWarps;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(32 * warps);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (gumbel) return cudaLaunchKernelEx(&cfg, pack_kernel<true>, p);
    return cudaLaunchKernelEx(&cfg, pack_kernel<false>, p);
}

cudaError_t launch_merge_payload(const CombineParams &c, const void *payload,
                                 cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((c.M + 127) / 128);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const unsigned char *pl = static_cast<const unsigned char *>(payload);
    if (c.flags & kFlagGumbel) return cudaLaunchKernelEx(&cfg, merge_payload_kernel<true>, c, pl);
    return cudaLaunchKernelEx(&cfg, merge_payload_kernel<false>, c, pl);
}

}  // namespace sb

namespace sb {
namespace {

// Host-to-device copy by the SMs: src is host memory the device can address (pinned and
// mapped), read in 16-byte words.  Triggers its dependents at entry (the GEMM's setup
// overlaps the copy) and writes dst only after the previous kernel in the stream has ended
// (that kernel may still be reading dst).
__global__ void copy16_kernel(uint4 *dst, const uint4 *src, size_t n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += stride)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy16(void *dst, const void *src, size_t n16, int num_sms,
                          cudaStream_t stream) {
    if (n16 == 0) return cudaSuccess;
    constexpr int kThreadsCopy = 256;
    size_t blocks = (n16 + kThreadsCopy - 1) / kThreadsCopy;
    if (blocks > static_cast<size_t>(num_sms) * 4) blocks = static_cast<size_t>(num_sms) * 4;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreadsCopy);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<uint4 *>(dst),
                              static_cast<const uint4 *>(src), n16);
}

}  // namespace sb
