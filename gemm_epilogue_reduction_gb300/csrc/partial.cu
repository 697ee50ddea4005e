// partial.cu -- row-parallel partial completion: lane partials of a split reduction and the
// deterministic sum that completes them.
//
// "SemBridge: Compiling Consumer Observations into Cross-Stack Communication Plans",
// Section 6.4 and Table 3: a row-parallel MLP down projection gives each tensor-parallel
// lane a slice of the reduction dimension; every lane produces an incomplete full-width
// output, and the partials must be summed (the completion obligation, Section 3.5) before
// any consumer observes the value.  Here the lanes are on one GPU:
//   Y[m][n] = sum over lanes l of P_l[m][n],  P_l = X[:, lane l] · W[:, lane l]^T.
// Each lane's slice is cut into equal chunks of 64-column K blocks so the work fills the
// GPU; `partial_kernel` writes one fp32 partial per (chunk, 128-feature tile) from a
// tcgen05 accumulator, and `complete_kernel` sums the chunks in ascending order -- lane 0's
// chunks first -- so the result bits never depend on scheduling.
//
// partial_kernel: persistent, 192 threads.  Warp 0 issues TMA loads of W (128 rows, the
// UMMA A operand) and X (all M rows, the B operand) into one ring; warp 1 owns TMEM (two
// accumulators) and issues tcgen05.mma; warps 2-5 read the accumulator (warp w reads TMEM
// lanes 32*(w%4)..) and store the partial tile.  All waits are time-bounded (sb_pipe.cuh).
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
constexpr uint32_t kPStageA = kTileA * kBlockK * 2;  // 16 KB of W per stage
constexpr int kPMaxStages = 16;
constexpr int kMinUnits = 1300;                      // chunking target (many short units)

struct PartialParams {
    int M, N, K, nb, kb_per_chunk, chunks, n_tiles, num_units, stages;
    float *partials;  // [chunks][M][N]
    uint32_t *epoch_word;
    unsigned long long *status;
    uint32_t epoch;
    unsigned long long timeout_ns;
};

__host__ __device__ inline uint32_t p_smem_bytes(int nb, int stages) {
    return stages * (kPStageA + nb * 128) + (2 * kPMaxStages + 8) * 8 + 16 + 1024;
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
    const uint32_t b_bytes = static_cast<uint32_t>(p.nb) * 128u;
    uint8_t *sA = smem;
    uint8_t *sB = smem + p.stages * kPStageA;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + p.stages * b_bytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + kPMaxStages;
    uint64_t *tfull = bars + 2 * kPMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kPMaxStages + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const WaitCtx wc{p.status, p.epoch, p.timeout_ns, abort_flag};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
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
        if (blockIdx.x == 0) *p.epoch_word = p.epoch;
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const int chunk = u / p.n_tiles, nt = u - chunk * p.n_tiles;
                const int kb0 = chunk * p.kb_per_chunk;
                for (int kb = kb0; kb < kb0 + p.kb_per_chunk; ++kb) {
                    if (!bwait(&empty[stage], phase ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kPStageA + b_bytes);
                    tma_load_2d(sA + stage * kPStageA, &tmW, &full[stage], kb * kBlockK,
                                nt * kTileA, pol_w);
                    tma_load_2d(sB + stage * b_bytes, &tmX, &full[stage], kb * kBlockK, 0, pol_x);
                    ++issued;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const uint32_t n = issued < static_cast<uint32_t>(p.stages) ? issued : p.stages;
            for (uint32_t i = issued - n; i < issued; ++i)
                bwait_drain(&full[i % p.stages], (i / p.stages) & 1u, wc);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = idesc_bf16_f32(kTileA, p.nb);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
                const int b = it & 1;
                if (!bwait(&tempty[b], ((it >> 1) & 1) ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.nb);
                for (int kb = 0; kb < p.kb_per_chunk; ++kb) {
                    if (!bwait(&full[stage], phase, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * kPStageA));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + stage * b_bytes));
#pragma unroll
                    for (int ks = 0; ks < kBlockK / 16; ++ks)
                        umma_bf16(d_tmem, adesc + 2u * ks, bdesc + 2u * ks, idesc,
                                  (kb | ks) != 0 ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    any = true;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(&tfull[b]);
            }
            if (any) {
                umma_commit(drain);
                bwait_drain(drain, 0, wc);
            }
        }
    } else {  // epilogue: thread = output feature n, TMEM columns = rows m
        const int q = warp & 3;
        int it = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
            const int b = it & 1;
            const bool ok = bwait(&tfull[b], (it >> 1) & 1, wc);
            if (p_vote_any(!ok)) break;
            tc_fence_after();
            const int chunk = u / p.n_tiles, nt = u - chunk * p.n_tiles;
            const int n = nt * kTileA + 32 * q + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(b * p.nb);
            float *dst = p.partials + static_cast<size_t>(chunk) * p.M * p.N + n;
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
                if (n < p.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < cw && c0 + j < p.M)
                            dst[static_cast<size_t>(c0 + j) * p.N] = __uint_as_float(raw[j]);
                }
            }
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

// Y[i] = sum over chunks c (ascending) of partials[c][i]; fp32 or bf16 (round to nearest).
__global__ void complete_kernel(const float *__restrict__ partials, int chunks, size_t mn,
                                float *yf, uint16_t *yb) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < mn;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float acc = 0.f;
        for (int c = 0; c < chunks; ++c) acc += __ldg(partials + c * mn + i);
        if (yb)
            yb[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        else
            yf[i] = acc;
    }
}

// Chunks per lane: the smallest divisor of the lane's K blocks giving at least kMinUnits
// work units, but no more than keep the fp32 partials' round trip (write + read,
// 8*lanes*chunks*M*N bytes) within about an eighth of W's bytes (2*N*K).  Chosen from the
// shape alone, so the workspace size does not depend on the device.  (Measured on the
// 5120 x 17408 down projection: 8 chunks per lane best at 64 tokens, 17 at 8 tokens.)
int chunks_per_lane(int64_t M, int64_t N, int64_t K, int32_t lanes) {
    const int64_t kb_lane = K / kBlockK / lanes;
    const int64_t n_tiles = (N + kTileA - 1) / kTileA;
    const int64_t cap = K / (16 * lanes * M);
    int64_t best = 1;
    for (int64_t c = 1; c <= kb_lane; ++c) {
        if (kb_lane % c) continue;
        if (c > cap && c > 1) break;
        best = c;
        if (n_tiles * lanes * c >= kMinUnits) break;
    }
    return static_cast<int>(best);
}

bool partial_shape_ok(int64_t M, int64_t N, int64_t K, int32_t lanes) {
    return M >= 1 && M <= kMaxVocabModeRows * 2 && N >= 1 && N < (int64_t(1) << 31) &&
           lanes >= 1 && K >= kBlockK && K < (int64_t(1) << 31) &&
           K % (static_cast<int64_t>(lanes) * kBlockK) == 0;
}

}  // namespace
}  // namespace sb

extern "C" {

size_t sb_partial_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t lanes) {
    using namespace sb;
    if (!partial_shape_ok(M, N, K, lanes)) return 0;
    const int64_t chunks = static_cast<int64_t>(lanes) * chunks_per_lane(M, N, K, lanes);
    return 256 + static_cast<size_t>(chunks) * M * N * 4;
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
    const size_t need = sb_partial_workspace_bytes(M, N, K, lanes);
    if (workspace_bytes < need) return SB_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0, cc = 0;
    if (int32_t e = device_sms_cc(&sms, &cc)) return e;

    PartialParams p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nb = static_cast<int>((M + 15) / 16 * 16);
    const int cpl = chunks_per_lane(M, N, K, lanes);
    p.kb_per_chunk = static_cast<int>(K / kBlockK / lanes / cpl);
    p.chunks = lanes * cpl;
    p.n_tiles = static_cast<int>((N + kTileA - 1) / kTileA);
    p.num_units = p.chunks * p.n_tiles;
    p.stages = kPMaxStages;
    while (p.stages > 2 && p_smem_bytes(p.nb, p.stages) > kSmemLimit) --p.stages;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.epoch_word = reinterpret_cast<uint32_t *>(ws);
    p.status = reinterpret_cast<unsigned long long *>(ws + 8);
    p.partials = reinterpret_cast<float *>(ws + 256);
    p.epoch = next_epoch();
    p.timeout_ns = wait_limit_ns();

    CUtensorMap tmW, tmX;
    if (!encode_bf16_map(&tmW, W, N, K, kTileA) || !encode_bf16_map(&tmX, X, M, K, p.nb))
        return SB_ERR_CUDA;
    const size_t smem = p_smem_bytes(p.nb, p.stages);
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
    const int grid = p.num_units < sms ? p.num_units : sms;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    partial_kernel<<<grid, kPThreads, smem, st>>>(tmW, tmX, p, cols);
    if (cudaGetLastError() != cudaSuccess) return SB_ERR_CUDA;

    const size_t mn = static_cast<size_t>(M) * N;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(256);
    const size_t blocks = (mn + 255) / 256;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks < 4096 ? blocks : 4096));
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    float *yf = y_bf16 ? nullptr : static_cast<float *>(Y);
    uint16_t *yb = y_bf16 ? static_cast<uint16_t *>(Y) : nullptr;
    if (cudaLaunchKernelEx(&cfg, complete_kernel, static_cast<const float *>(p.partials),
                           p.chunks, mn, yf, yb) != cudaSuccess)
        return SB_ERR_CUDA;
    return SB_OK;
}

}  // extern "C"
