// partial.cu -- row-parallel partial completion: lane partials of a split reduction and the
// deterministic sum that completes them.
//
// "SemBridge: Compiling Consumer Observations into Cross-Stack Communication Plans",
// Section 6.4 and Table 3: a row-parallel MLP down projection gives each tensor-parallel
// lane a slice of the reduction dimension; every lane produces an incomplete full-width
// output, and the partials must be summed (the completion obligation, Section 3.5) before
// any consumer observes the value.  Here the lanes are on one GPU:
//   Y[m][n] = sum over lanes l of P_l[m][n],  P_l = X[:, lane l] · W[:, lane l]^T.
//
// Work split.  The work is the sequence of (128-feature tile, 64-column K block) pairs, tile
// by tile and K block by K block within a tile; CTA i of G takes a contiguous run of q or
// q + 1 of them (q = work / G), so every CTA streams the same number of W bytes to within
// one K block.  Each lane's slice of a tile (a "chunk") is covered by consecutive CTAs, and
// a CTA's share of one chunk (a "piece") is accumulated in TMEM and stored as an fp32 slab
// [M][128] at slot (chunk, CTA - first CTA of the chunk).
//
// Completion.  `complete_kernel`, launched as a programmatic dependent of `partial_kernel`
// (it waits for that grid before reading), gives every thread four features of one row of
// Y: it sums the tile's slabs in ascending K order -- lane 0's first -- and writes Y.  The
// summation order is fixed, so the result bits never depend on scheduling.
//
// partial_kernel: persistent, 192 threads.  Warp 0 issues the TMA loads of one ring of
// joint stages, each holding one K block of W (128 rows, the UMMA A operand) and of X (all M
// rows, the B operand), so the MMA warp waits once and commits once per K block; warp 1 owns
// TMEM (two accumulators) and issues tcgen05.mma; warps 2-5 read the accumulator (warp w
// reads TMEM lanes 32*(w%4)..) and store the slab.  All waits are time-bounded
// (sb_pipe.cuh).
#include <cuda_bf16.h>

#include <atomic>
#include <climits>

#include "sb.h"
#include "sb_internal.h"
#include "sb_pipe.cuh"
#include "sb_ptx.cuh"

namespace sb {
namespace {

constexpr int kPThreads = 192;
constexpr uint32_t kPStageW = kTileA * kBlockK * 2;  // 16 KB of W per stage
constexpr int kPMaxStages = 16;
constexpr int kPMaxGrid = 1024;

struct PartialParams {
    int M, N, nb, kb_tile, lanes, lane_kb, n_tiles, grid, pieces, stages_w, stages_x;
    uint32_t q, r;                   // CTA i owns q + 1 K blocks if i < r, else q
    float *partials;                 // [n_tiles * lanes][pieces][M][128]
    float *yf;                       // Y as fp32, or
    uint16_t *yb;                    // Y as bf16 bits
    uint32_t *epoch_word;
    unsigned long long *status;
    uint32_t epoch;
    unsigned long long timeout_ns;
};

__host__ __device__ inline uint32_t p_smem_bytes(int nb, int stages_w, int stages_x) {
    return stages_w * kPStageW + stages_x * nb * 128 + (4 * kPMaxStages + 8) * 8 + 16 + 1024;
}

// First work index of CTA i, and the CTA that owns work index x (all 32-bit: the work
// count is checked against 2^31 on the host).
__host__ __device__ inline uint32_t cta_begin(uint32_t q, uint32_t r, uint32_t i) {
    return i * q + (i < r ? i : r);
}
__host__ __device__ inline uint32_t cta_of(uint32_t q, uint32_t r, uint32_t x) {
    const uint32_t big = r * (q + 1);
    return x < big ? x / (q + 1) : r + (x - big) / q;
}

__device__ __forceinline__ bool p_vote_any(bool pred) {  // over the 128 epilogue threads
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kPThreads, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const PartialParams p, const uint32_t tmem_cols) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t x_bytes = static_cast<uint32_t>(p.nb) * 128u;
    uint8_t *sW = smem;
    uint8_t *sX = smem + p.stages_w * kPStageW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sX + p.stages_x * x_bytes);
    uint64_t *full = bars;                 // joint stage landed (W and X bytes)
    uint64_t *empty = bars + kPMaxStages;  // joint stage consumed (one MMA commit)
    uint64_t *tfull = bars + 4 * kPMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4 * kPMaxStages + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const WaitCtx wc{p.status, p.epoch, p.timeout_ns, abort_flag};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t x_begin = cta_begin(p.q, p.r, blockIdx.x);
    const uint32_t x_end = x_begin + p.q + (blockIdx.x < p.r ? 1u : 0u);
    const uint32_t first_cut = (x_begin / p.lane_kb + 1) * p.lane_kb;  // next lane boundary

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages_w; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The setup above touches no global memory, so it overlaps the previous kernel in the
    // stream (this kernel is a programmatic dependent launch).  W is a weight that kernel
    // does not write, so the first stages' W halves are loaded before the wait (the W stream
    // starts while the previous kernel finishes; the expect covers the whole stage); X and
    // the workspace may belong to that kernel, so everything else waits for it.
    uint32_t w_pre = 0;
    if (warp == 0 && lane == 0) {
        const uint32_t n = x_end - x_begin;
        w_pre = n < static_cast<uint32_t>(p.stages_w) ? n : static_cast<uint32_t>(p.stages_w);
        int tile = static_cast<int>(x_begin / p.kb_tile);
        int kb = static_cast<int>(x_begin) - tile * p.kb_tile;
        const uint64_t pol = policy_evict_first();
        for (uint32_t i = 0; i < w_pre; ++i) {
            mbar_arrive_expect_tx(&full[i], kPStageW + x_bytes);
            tma_load_2d(sW + i * kPStageW, &tmW, &full[i], kb * kBlockK, tile * kTileA, pol);
            if (++kb == p.kb_tile) {
                kb = 0;
                ++tile;
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.epoch_word = p.epoch;
    // let the completion (a programmatic dependent launch) get scheduled early; it waits for
    // this whole grid before it reads any slab
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {  // TMA producer: the CTA's K blocks in order, W and X per stage
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            int tile = static_cast<int>(x_begin / p.kb_tile);
            int kb = static_cast<int>(x_begin) - tile * p.kb_tile;
            for (uint32_t x = x_begin; x < x_end; ++x) {
                const bool w_done = issued < w_pre;  // W issued (and expected) before the wait
                if (!w_done) {
                    if (!bwait(&empty[stage], phase ^ 1u, wc)) break;
                    mbar_arrive_expect_tx(&full[stage], kPStageW + x_bytes);
                    tma_load_2d(sW + stage * kPStageW, &tmW, &full[stage], kb * kBlockK,
                                tile * kTileA, pol_w);
                }
                tma_load_2d(sX + stage * x_bytes, &tmX, &full[stage], kb * kBlockK, 0, pol_x);
                ++issued;
                if (++stage == p.stages_w) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++kb == p.kb_tile) {
                    kb = 0;
                    ++tile;
                }
            }
            const uint32_t n = issued < static_cast<uint32_t>(p.stages_w) ? issued : p.stages_w;
            for (uint32_t i = issued - n; i < issued; ++i)
                bwait_drain(&full[i % p.stages_w], (i / p.stages_w) & 1u, wc);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer: one accumulation per piece
            const uint32_t idesc = idesc_bf16_f32(kTileA, p.nb);
            int st = 0, j = 0;
            uint32_t ph = 0;
            bool ok = true, any = false;
            uint32_t cut = first_cut;
            for (uint32_t x = x_begin; ok && x < x_end; ++j, cut += p.lane_kb) {
                const uint32_t e = cut < x_end ? cut : x_end;
                const int b = j & 1;
                if (!bwait(&tempty[b], ((j >> 1) & 1) ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.nb);
                for (uint32_t xx = x; xx < e; ++xx) {
                    if (!bwait(&full[st], ph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sW + st * kPStageW));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sX + st * x_bytes));
#pragma unroll
                    for (int ks = 0; ks < kBlockK / 16; ++ks)
                        umma_bf16(d_tmem, adesc + 2u * ks, bdesc + 2u * ks, idesc,
                                  (xx != x || ks != 0) ? 1u : 0u);
                    umma_commit(&empty[st]);  // one commit frees the joint stage
                    any = true;
                    if (++st == p.stages_w) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) umma_commit(&tfull[b]);
                x = e;
            }
            if (any) {
                umma_commit(drain);
                bwait_drain(drain, 0, wc);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // epilogue: thread = output feature of the tile, TMEM columns = rows m
        const int q = warp & 3;
        const int nl = 32 * q + lane;
        int j = 0;
        uint32_t cut = first_cut;
        for (uint32_t x = x_begin; x < x_end; ++j, cut += p.lane_kb) {
            const uint32_t e = cut < x_end ? cut : x_end;
            const uint32_t chunk = x / p.lane_kb;
            const uint32_t piece = blockIdx.x - cta_of(p.q, p.r, chunk * p.lane_kb);
            const int b = j & 1;
            const bool ok = bwait(&tfull[b], (j >> 1) & 1, wc);
            if (p_vote_any(!ok)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(b * p.nb);
            float *dst = p.partials +
                         (static_cast<size_t>(chunk) * p.pieces + piece) * p.M * kTileA + nl;
            for (int c0 = 0; c0 < p.nb; c0 += 32) {
                uint32_t raw[32];
                const int cw = min(32, p.nb - c0);
                if (cw == 32)
                    tmem_ld32x32b_x32(taddr + c0, raw);
                else
                    tmem_ld32x32b_x16(taddr + c0, raw);
                if (c0 + 32 >= p.nb) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[b]);
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (jj < cw && c0 + jj < p.M)
                        dst[static_cast<size_t>(c0 + jj) * kTileA] = __uint_as_float(raw[jj]);
            }
            x = e;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

// Y[m][n] = the left fold over the tile's slabs, in ascending K order, of slab[m][n % 128];
// one thread per four features of one row.  Slabs are read in batches of kBatch, all loads
// of a batch issued before its adds.
__global__ void __launch_bounds__(256)
    complete_kernel(const PartialParams p) {
    constexpr int kBatch = 8;
    // let the next kernel in the stream (a dependent launch) start its setup early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t items = static_cast<size_t>(p.n_tiles) * p.M * (kTileA / 4);
    for (size_t it = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
         it += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int f4 = static_cast<int>(it % (kTileA / 4));
        const int m = static_cast<int>((it / (kTileA / 4)) % p.M);
        const int tile = static_cast<int>(it / (static_cast<size_t>(kTileA / 4) * p.M));
        const int n0 = tile * kTileA + 4 * f4;
        if (n0 >= p.N) continue;
        const float *base = p.partials + static_cast<size_t>(m) * kTileA + 4 * f4;
        const size_t slab = static_cast<size_t>(p.M) * kTileA;
        // walk (lane l, CTA i) over the tile's chunks: slot = chunk * pieces + (i - a)
        int l = 0;
        uint32_t c = static_cast<uint32_t>(tile * p.lanes);
        uint32_t a = cta_of(p.q, p.r, c * p.lane_kb);
        uint32_t b = cta_of(p.q, p.r, c * p.lane_kb + p.lane_kb - 1);
        uint32_t i = a;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        while (l < p.lanes) {
            float4 v[kBatch];
            bool ok[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                ok[k] = l < p.lanes;
                if (ok[k]) {
                    v[k] = __ldg(reinterpret_cast<const float4 *>(
                        base + (static_cast<size_t>(c) * p.pieces + (i - a)) * slab));
                    if (++i > b) {
                        if (++l < p.lanes) {
                            ++c;
                            a = cta_of(p.q, p.r, c * p.lane_kb);
                            b = cta_of(p.q, p.r, c * p.lane_kb + p.lane_kb - 1);
                            i = a;
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (ok[k]) {
                    acc.x += v[k].x;
                    acc.y += v[k].y;
                    acc.z += v[k].z;
                    acc.w += v[k].w;
                }
            }
        }
        const float r4[4] = {acc.x, acc.y, acc.z, acc.w};
        const size_t o = static_cast<size_t>(m) * p.N + n0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (n0 + u >= p.N) break;
            if (p.yb)
                p.yb[o + u] = __bfloat16_as_ushort(__float2bfloat16_rn(r4[u]));
            else
                p.yf[o + u] = r4[u];
        }
    }
}

struct PartialPlan {
    int grid, pieces, n_tiles, kb_tile, lane_kb;
    uint32_t q, r;
    size_t slab_off, bytes;
};

bool partial_shape_ok(int64_t M, int64_t N, int64_t K, int32_t lanes) {
    return M >= 1 && M <= kMaxVocabModeRows * 2 && N >= 1 && N < (int64_t(1) << 31) &&
           lanes >= 1 && K >= kBlockK && K < (int64_t(1) << 31) &&
           K % (static_cast<int64_t>(lanes) * kBlockK) == 0;
}

// The split for the current device: one CTA per SM (at most one per K block), the most
// pieces any chunk has, and the workspace layout (header, then the slabs).
int32_t make_plan(int64_t M, int64_t N, int64_t K, int32_t lanes, PartialPlan *pl) {
    if (!partial_shape_ok(M, N, K, lanes)) return SB_ERR_INVALID_ARG;
    int sms = 0, cc = 0;
    if (int32_t e = device_sms_cc(&sms, &cc)) return e;
    const int64_t n_tiles = (N + kTileA - 1) / kTileA;
    const int64_t work = n_tiles * (K / kBlockK);
    if (work >= (int64_t(1) << 31)) return SB_ERR_UNSUPPORTED;
    pl->n_tiles = static_cast<int>(n_tiles);
    pl->kb_tile = static_cast<int>(K / kBlockK);
    pl->lane_kb = pl->kb_tile / lanes;
    int64_t g = sms < kPMaxGrid ? sms : kPMaxGrid;
    if (g > work) g = work;
    pl->grid = static_cast<int>(g);
    pl->q = static_cast<uint32_t>(work / g);
    pl->r = static_cast<uint32_t>(work % g);
    const uint32_t lk = static_cast<uint32_t>(pl->lane_kb);
    uint32_t pieces = 1;
    const int64_t chunks = n_tiles * lanes;
    for (int64_t c = 0; c < chunks; ++c) {
        const uint32_t c0 = static_cast<uint32_t>(c) * lk;
        const uint32_t n = cta_of(pl->q, pl->r, c0 + lk - 1) - cta_of(pl->q, pl->r, c0) + 1;
        pieces = n > pieces ? n : pieces;
    }
    pl->pieces = static_cast<int>(pieces);
    pl->slab_off = 256;
    pl->bytes = pl->slab_off + static_cast<size_t>(chunks) * pieces * M * kTileA * 4;
    return SB_OK;
}

}  // namespace
}  // namespace sb

extern "C" {

size_t sb_partial_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t lanes) {
    sb::PartialPlan pl;
    return sb::make_plan(M, N, K, lanes, &pl) == SB_OK ? pl.bytes : 0;
}

int32_t sb_partial_completion(const void *X, const void *W, int64_t M, int64_t N, int64_t K,
                              int32_t lanes, void *Y, int32_t y_bf16, void *workspace,
                              size_t workspace_bytes, void *stream) {
    using namespace sb;
    if (!X || !W || !Y || !workspace || !partial_shape_ok(M, N, K, lanes))
        return SB_ERR_INVALID_ARG;
    if (!(reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0 &&
          reinterpret_cast<uintptr_t>(workspace) % 256 == 0 &&
          reinterpret_cast<uintptr_t>(Y) % (y_bf16 ? 2 : 4) == 0))
        return SB_ERR_ALIGNMENT;
    PartialPlan pl;
    if (int32_t e = make_plan(M, N, K, lanes, &pl)) return e;
    if (workspace_bytes < pl.bytes) return SB_ERR_WORKSPACE_TOO_SMALL;

    PartialParams p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.nb = static_cast<int>((M + 15) / 16 * 16);
    p.kb_tile = pl.kb_tile;
    p.lanes = lanes;
    p.lane_kb = pl.lane_kb;
    p.n_tiles = pl.n_tiles;
    p.grid = pl.grid;
    p.pieces = pl.pieces;
    p.q = pl.q;
    p.r = pl.r;
    // joint stages (one K block of W and of X each), as many as fit
    p.stages_w = kPMaxStages;
    while (p.stages_w > 2 && p_smem_bytes(p.nb, p.stages_w, p.stages_w) > kSmemLimit)
        --p.stages_w;
    p.stages_x = p.stages_w;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.epoch_word = reinterpret_cast<uint32_t *>(ws);
    p.status = reinterpret_cast<unsigned long long *>(ws + 8);
    p.partials = reinterpret_cast<float *>(ws + pl.slab_off);
    p.yf = y_bf16 ? nullptr : static_cast<float *>(Y);
    p.yb = y_bf16 ? static_cast<uint16_t *>(Y) : nullptr;
    p.epoch = next_epoch();
    p.timeout_ns = wait_limit_ns();

    CUtensorMap tmW, tmX;
    if (!encode_bf16_map(&tmW, W, N, K, kTileA) || !encode_bf16_map(&tmX, X, M, K, p.nb))
        return SB_ERR_CUDA;
    const size_t smem = p_smem_bytes(p.nb, p.stages_w, p.stages_x);
    static std::atomic<uint64_t> opted_in{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SB_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(opted_in.load() & bit)) {
        if (cudaFuncSetAttribute(partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit)) != cudaSuccess)
            return SB_ERR_CUDA;
        opted_in.fetch_or(bit);
    }
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * p.nb)) cols <<= 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    {
        // a programmatic dependent of the previous kernel in the stream (see the kernel)
        cudaLaunchConfig_t pc{};
        pc.gridDim = dim3(static_cast<unsigned>(p.grid));
        pc.blockDim = dim3(kPThreads);
        pc.dynamicSmemBytes = smem;
        pc.stream = st;
        cudaLaunchAttribute pa[1];
        pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pa[0].val.programmaticStreamSerializationAllowed = 1;
        pc.attrs = pa;
        pc.numAttrs = 1;
        if (cudaLaunchKernelEx(&pc, partial_kernel, tmW, tmX, p, cols) != cudaSuccess)
            return SB_ERR_CUDA;
    }

    int sms = 0, cc = 0;
    if (int32_t e = device_sms_cc(&sms, &cc)) return e;
    const size_t items = static_cast<size_t>(p.n_tiles) * p.M * (kTileA / 4);
    const size_t blocks = (items + 255) / 256;
    const size_t cap = static_cast<size_t>(sms) * 8;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, complete_kernel, p) != cudaSuccess) return SB_ERR_CUDA;
    return SB_OK;
}

}  // extern "C"
