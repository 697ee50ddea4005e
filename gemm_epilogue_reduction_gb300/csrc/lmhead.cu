// lmhead.cu -- the fused output-head GEMM + projection-record epilogue for sm_103a.
//
// One persistent, warp-specialised kernel computes z = H·Wᵀ tile by tile on the
// 5th-generation tensor cores and reduces each tile straight out of TMEM into compact
// per-(row, lane shard, tile) records (max, lowest argmax, sum of exp), so the token
// surface never writes logits to HBM ("SemBridge: Compiling Consumer Observations into
// Cross-Stack Communication Plans", Section 5.2 and Figure 1: source projection applies
// the deterministic argmax where the logits are produced).  The full-logit surface
// additionally writes bf16 logits in shard-to-full (global column) layout.
//
// Structure (the warp roles and TMEM epilogue of the "01 · 通算融合" note on Blackwell
// SM100 GEMMs, sections 2 and 5.1: TMA producer, MMA issuer, epilogue warps; full-K
// accumulation before any epilogue work):
//   warp 0      the TMA producer (one lane) of 64-wide K slices (128-byte swizzle): one ring
//               of joint stages, each holding one K block of both operands (vocab mode: 128
//               W rows and all M rows of H; rows mode: 128 H rows and this CTA's half of the
//               W tile), so the MMA waits on one barrier and commits once per K block (each
//               commit costs the tensor pipe time); warp 2 has no role;
//   warp 1      owns the TMEM allocation; one lane issues tcgen05.mma (M = 128, or
//               M = 256 over a CTA pair in rows mode; bf16 x bf16 -> fp32) into one of two
//               TMEM accumulators and commits stage releases and "accumulator full" to
//               mbarriers;
//   warps 3-10  the epilogue, two warps per TMEM lane quadrant: tcgen05.ld of the finished
//               accumulator (warp w reads TMEM lanes 32*(w%4) .. +31), mask columns outside
//               the tile's shard, fold the projection records, release the accumulator.
// Two tile orientations share the pipeline:
//   vocab mode (M <= 128, decode): A = 128 rows of W (vocabulary), B = all
//               M rows of H (UMMA N = M rounded up to 16).  TMEM lane = vocabulary
//               column; the epilogue reduces across lanes with warp reductions.
//   rows mode  (M > 128, sampling batches and prefill scoring): A = 128 rows of H, B = 256
//               rows of W (half of them staged by each CTA of a pair).  TMEM lane = row of
//               H; each epilogue thread folds half of its row's 256 columns serially.
// Every record covers 128 vocabulary columns (one vocab-mode tile, half a rows-mode tile).
// Vocabulary tiles never cross a lane-shard boundary: tile t of shard s starts at
// s*S + t*TV and is masked at (s+1)*S, so each record belongs to one shard.
//
// Every mbarrier wait is bounded (a time limit read from %globaltimer); a wait that runs
// out records SB_ERR_DEVICE_TIMEOUT in the workspace status word, raises a CTA-wide abort
// flag, and every role then drains its own in-flight TMA copies and MMAs before the TMEM
// is freed and the CTA exits.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "sb_gumbel.cuh"
#include "sb_internal.h"
#include "sb_pipe.cuh"
#include "sb_ptx.cuh"

namespace sb {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kStageBytesA = kTileA * kBlockK * 2;  // 16 KB

struct SmemLayout {
    uint32_t a_off, b_off, bar_off, misc_off, tgt_off, scratch_off, total;
};

// Shared memory: the A halves of the stages (stages_a x atoms x 16 KB), the B halves
// (stages_b x atoms x nb*128 B, half of that per CTA in rows mode), mbarriers, TMEM address
// + abort flag, vocab-mode target ids and cross-quadrant scratch.  With a joint ring
// stages_a == stages_b and stage s is the pair (A half s, B half s); with split rings the
// two halves are independent rings of their own depths.
__host__ __device__ inline SmemLayout make_layout(int nb, int stages_a, int stages_b, bool vocab,
                                                  int flags, int topk, int atoms) {
    SmemLayout L;
    uint32_t off = 0;
    L.a_off = off;
    off += stages_a * kStageBytesA * (vocab ? 1 : atoms);
    L.b_off = off;
    // rows mode (CTA pairs): each CTA stages only its half of the W tile
    off += stages_b * (vocab ? nb : nb / 2) * 128 * (vocab ? 1 : atoms);
    L.bar_off = off;
    off += (4 * kMaxStages + 8) * 8;
    L.misc_off = off;
    off += 16;
    L.tgt_off = off;
    off += vocab ? kMaxVocabModeRows * 4 : 0;
    L.scratch_off = off;
    off += vocab ? 4 * nb * ((flags & kFlagGumbel) ? 24 : 12) : 0;
    // top-K: the tile's logits, nb rows of 128 fp32 (16-byte aligned: everything before it
    // is a multiple of 16 bytes)
    off += (vocab && (flags & kFlagTopk)) ? nb * kVocabTileV * 4 : 0;
    (void)topk;
    L.total = off + 1024;  // slack to align the base to 1024 bytes
    return L;
}

struct TileCoord {
    int s, t, v0, v_end, m0, a_row, b_row;
};

// Work unit `tile` of a CTA with cluster rank `rank`.  Vocab mode: one 128-column vocabulary
// tile.  Rows mode: one 256-column vocabulary tile times a pair of consecutive M tiles, CTA
// `rank` of the pair taking M tile 2*group + rank and staging W rows [v0 + 128*rank, +128)
// of the tile (its half of the pair MMA's B operand).
template <bool VOCAB>
__device__ __forceinline__ TileCoord tile_coord(const GemmParams &p, int tile, int rank) {
    constexpr int CS = VOCAB ? 1 : kRowsCluster;
    TileCoord c;
    const int vt = VOCAB ? tile : tile / p.m_groups;
    const int mt = VOCAB ? 0 : (tile % p.m_groups) * CS + rank;
    c.s = vt / p.Tt;
    c.t = vt - c.s * p.Tt;
    c.v0 = c.s * p.S + c.t * p.tv;
    c.v_end = min(c.v0 + p.tv, (c.s + 1) * p.S);
    c.m0 = mt * kTileA;
    c.a_row = VOCAB ? c.v0 : c.m0;
    c.b_row = VOCAB ? 0 : c.v0 + rank * (kRowsTileN / CS);
    return c;
}

__device__ __forceinline__ WaitCtx wait_ctx(const GemmParams &p, volatile int *abort_flag) {
    return WaitCtx{p.ws.status, p.epoch, p.timeout_ns, abort_flag};
}
__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                      const GemmParams &p) {
    return bwait(bar, parity, wait_ctx(p, abort_flag));
}
__device__ __forceinline__ bool bwait_drain(uint64_t *bar, uint32_t parity,
                                            volatile int *abort_flag, const GemmParams &p) {
    return bwait_drain(bar, parity, wait_ctx(p, abort_flag));
}
// For barriers armed from the other CTA of a pair (cluster-scope acquire).
__device__ __forceinline__ bool bwait_cl(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         const GemmParams &p) {
    return bwait_cluster(bar, parity, wait_ctx(p, abort_flag));
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Named-barrier vote over the 256 epilogue threads: true if any thread passes true.
__device__ __forceinline__ bool epi_vote_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// Counter-based uniform: SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) at stream index n
// of the stream seeded with `seed`: the state is seed + (n + 1) * golden-ratio increment,
// then the finaliser; the top 24 bits b give u = b * 2^-24 in [0, 1).
constexpr unsigned long long kGolden = 0x9E3779B97F4A7C15ull;
__device__ __forceinline__ unsigned long long splitmix_state(unsigned long long seed,
                                                             unsigned long long n) {
    return seed + (n + 1ull) * kGolden;
}
// The finaliser ends with x ^= x >> 31; its top 24 bits are those of x itself (x >> 31
// contributes nothing above bit 32), so that last step is left out.
__device__ __forceinline__ uint32_t bits24_from_state(unsigned long long x) {
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return static_cast<uint32_t>(x >> 40);
}

__device__ __forceinline__ uint32_t select_u32(bool pred, uint32_t a, uint32_t b) {
    uint32_t r;
    asm("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tselp.b32 %0, %2, %3, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float z) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(z));
}

// Compare-exchange for a descending sort of (key, position) pairs: after it, (ka, ea) ranks
// at or above (kb, eb), i.e. the larger key, or the lower position on an equal key.
__device__ __forceinline__ void cas_desc(uint32_t &ka, int &ea, uint32_t &kb, int &eb) {
    const bool swap = kb > ka || (kb == ka && eb < ea);
    const uint32_t k = swap ? kb : ka;
    const int e = swap ? eb : ea;
    kb = swap ? ka : kb;
    eb = swap ? ea : eb;
    ka = k;
    ea = e;
}

// Sums of 8 rows over a warp: a[j] is this lane's term of row j.  Three exchange steps
// (xor 16, 8, 4) each send half of the rows still held and add the other half's partner
// terms, so the lane keeps one row, (lane >> 2) & 7; two butterfly steps (xor 2, 1) finish
// it.  Every lane of a group of four holds the same bits (the adds are commutative).
__device__ __forceinline__ float transposed_row_sum8(const float (&a)[8], int lane) {
    const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
    float b[4], c[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? a[i] : a[i + 4];
        const float keep = b4 ? a[i + 4] : a[i];
        b[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? b[i] : b[i + 2];
        const float keep = b3 ? b[i + 2] : b[i];
        c[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    const float send = b2 ? c[0] : c[1];
    const float keep = b2 ? c[1] : c[0];
    float d = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
    d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
    d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
    return d;
}

// ------------------------------------------------------------------ epilogue, vocab mode
// Thread (warp quadrant q, lane) holds vocabulary column v = v0 + 32q + lane for every row
// (TMEM columns).  The two warps of a quadrant take alternate 8-row chunks (half h takes
// chunks h, h+2, ...), so at M <= 16 each walks at most 8 rows.  Per row: warp max, lowest
// argmax and sum of exp with warp reductions; then the four quadrants' partial records
// merge in quadrant order through shared memory.
template <int EPI>
__device__ __forceinline__ void epilogue_vocab(const GemmParams &p, const TileCoord &c,
                                               uint32_t taddr, uint64_t *tempty_b, int q,
                                               int h, int lane, const int32_t *tgt_s,
                                               float *scratch) {
    constexpr bool GUMBEL = EPI == kEpiGumbel;
    constexpr bool FULL = EPI == kEpiFull;
    constexpr bool TOPK = EPI == kEpiTopk;
    const int nb = p.nb;
    const int K = p.topk;
    const int col0 = c.v0 + 32 * q;  // column of lane 0: lanes hold ascending columns
    const int v = col0 + lane;
    const bool valid = v < c.v_end;
    const bool has_t = (p.flags & kFlagTargets) != 0;
    float *sc_m = scratch;
    int *sc_i = reinterpret_cast<int *>(scratch + 4 * nb);
    float *sc_s = scratch + 8 * nb;
    float *sc_gk = scratch + 12 * nb;
    int *sc_gi = reinterpret_cast<int *>(scratch + 16 * nb);
    float *sc_gz = scratch + 20 * nb;
    float *zs = scratch + 12 * nb;  // top-K: the tile's logits, [row][128]

    // nb is a multiple of 16, so every chunk is 8 whole accumulator columns.  The chunk's
    // rows are independent, so each step is issued for all 8 rows before the next step (the
    // warp reductions of different rows overlap); rows past M (zero rows of H) go through
    // the reductions and are not stored.
    for (int c0 = 8 * h; c0 < nb; c0 += 16) {
        constexpr int cw = 8;
        uint32_t raw[cw];
        tmem_ld32x32b_x8(taddr + c0, raw);
        float y[cw];
        uint32_t oy[cw], om[cw];
#pragma unroll
        for (int j = 0; j < cw; ++j) {
            const float z = __uint_as_float(raw[j]);
            y[j] = valid ? (GUMBEL ? z * p.inv_t : z) : -INFINITY;
            oy[j] = float_to_ordered(y[j]);
        }
#pragma unroll
        for (int j = 0; j < cw; ++j) om[j] = __reduce_max_sync(0xFFFFFFFFu, oy[j]);
        int wi[cw];
        float ws[cw];
#pragma unroll
        for (int j = 0; j < cw; ++j) {
            wi[j] = __reduce_min_sync(0xFFFFFFFFu, (valid && oy[j] == om[j]) ? v : INT_MAX);
            const float wm = ordered_to_float(om[j]);
            ws[j] = valid ? ex2_approx(fmaf(y[j], kLog2e, -wm * kLog2e)) : 0.f;
        }
        // The 8 rows' sums over the 32 lanes in one transposed reduction: each xor step hands
        // half of the rows a lane still holds to its partner (16: rows 4-7 / 0-3, 8, 4), then
        // two plain steps; row j ends in lanes 4j .. 4j+3 (identical bits in all four).
        const int jr = lane >> 2;  // the row this lane ends up holding
        const float my_s = transposed_row_sum8(ws, lane);
        float my_m = -INFINITY, my_gk = -INFINITY, my_gz = 0.f;
        int my_i = INT_MAX, my_gi = INT_MAX;
#pragma unroll
        for (int j = 0; j < cw; ++j)
            if (jr == j) {
                my_m = ordered_to_float(om[j]);
                my_i = wi[j];
            }
        if (GUMBEL) {
            // stream index of (row c0 + j, column v) is (c0 + j) V + v: the state advances by
            // V golden-ratio increments per row
            unsigned long long st = splitmix_state(
                p.seed, static_cast<unsigned long long>(c0) * static_cast<unsigned>(p.V) +
                            static_cast<unsigned>(v));
            uint32_t ok[cw], okm[cw];
#pragma unroll
            for (int j = 0; j < cw; ++j) {
                // keys are compared less the constant -ln(ln 2), added back per record
                const float kj = gumbel_key_less_c0(y[j], bits24_from_state(st));
                st += static_cast<unsigned long long>(static_cast<unsigned>(p.V)) * kGolden;
                ok[j] = float_to_ordered(valid ? kj : -INFINITY);
            }
#pragma unroll
            for (int j = 0; j < cw; ++j) okm[j] = __reduce_max_sync(0xFFFFFFFFu, ok[j]);
#pragma unroll
            for (int j = 0; j < cw; ++j) {
                const int gi =
                    __reduce_min_sync(0xFFFFFFFFu, (valid && ok[j] == okm[j]) ? v : INT_MAX);
                const int src = (gi == INT_MAX) ? 0 : (gi - col0);
                const float gz = __shfl_sync(0xFFFFFFFFu, __uint_as_float(raw[j]), src & 31);
                if (jr == j) {
                    my_gk = ordered_to_float(okm[j]);
                    my_gi = gi;
                    my_gz = gz;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < cw; ++j) {
            const int row = c0 + j;
            if (row >= p.M || !valid) continue;
            const float z = __uint_as_float(raw[j]);
            if (FULL) p.logits[static_cast<size_t>(row) * p.V + v] = bf16_bits_rn(z);
            if (has_t && tgt_s[row] == v) p.ws.tz[row] = z;
            if (TOPK) zs[row * kVocabTileV + 32 * q + lane] = z;
        }
        if ((lane & 3) == 0 && c0 + jr < p.M) {
            const int o = q * nb + c0 + jr;
            sc_m[o] = my_m;
            sc_i[o] = my_i;
            sc_s[o] = my_s;
            if (GUMBEL) {
                sc_gk[o] = my_gk;
                sc_gi[o] = my_gi;
                sc_gz[o] = my_gz;
            }
        }
    }
    // this warp's TMEM reads of the tile are done: hand its share of the accumulator back
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tempty_b);
    epi_bar_sync();
    const int te = threadIdx.x - 32 * kFirstEpiWarp;
    for (int row = te; row < p.M; row += 32 * kEpiWarps) {
        float m = -INFINITY;
        int idx = INT_MAX;
        for (int w = 0; w < 4; ++w) {
            const float mw = sc_m[w * nb + row];
            const int iw = sc_i[w * nb + row];
            if (mw > m || (mw == m && iw < idx)) {
                m = mw;
                idx = iw;
            }
        }
        float s = 0.f;
        for (int w = 0; w < 4; ++w) {
            const float mw = sc_m[w * nb + row];
            if (mw != -INFINITY) s += sc_s[w * nb + row] * ex2_approx((mw - m) * kLog2e);
        }
        const size_t ri = (static_cast<size_t>(row) * p.k + c.s) * p.T + c.t;
        p.ws.m[ri] = m;
        p.ws.idx[ri] = idx;
        p.ws.s[ri] = s;
        if (GUMBEL) {
            float gk = -INFINITY, gz = 0.f;
            int gi = INT_MAX;
            for (int w = 0; w < 4; ++w) {
                const float kw = sc_gk[w * nb + row];
                const int iw = sc_gi[w * nb + row];
                if (kw > gk || (kw == gk && iw < gi)) {
                    gk = kw;
                    gi = iw;
                    gz = sc_gz[w * nb + row];
                }
            }
            p.ws.gk[ri] = gk + kGumbelC0;
            p.ws.gi[ri] = gi;
            p.ws.gz[ri] = gz;
        }
    }
    if (TOPK) {
        // the record's K largest per row over the whole 128-column tile.  Warp e of the
        // epilogue takes rows e, e + 8, ... two at a time; lane l holds columns 4l .. 4l + 3,
        // sorted (larger first, lower column on ties).  Each round the warp max of the lanes'
        // heads wins; the lowest lane holding it has the lowest column, writes the entry to
        // shared memory (over the row's logits, already in registers) and drops its head.
        // Key 0 (below every ordered float) marks an empty slot; an entry no round fills
        // stays (-inf, INT_MAX).  The lists leave in one coalesced store per row.
        const int nvalid = c.v_end - c.v0;
        const int ew = (threadIdx.x >> 5) - kFirstEpiWarp;
        const uint32_t lt = lanemask_lt();
        const int c4 = 4 * lane;
        for (int r0 = ew; r0 < p.M; r0 += 2 * kEpiWarps) {
            uint32_t k0[2], k1[2], k2[2], k3[2];
            int e0[2], e1[2], e2[2], e3[2];
            float *lv[2];
            int *li[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int row = r0 + u * kEpiWarps;
                const bool have = row < p.M;
                float *zr = zs + (have ? row : r0) * kVocabTileV;
                const float4 x = *reinterpret_cast<const float4 *>(zr + c4);
                k0[u] = have && c4 + 0 < nvalid ? float_to_ordered(x.x) : 0u;
                k1[u] = have && c4 + 1 < nvalid ? float_to_ordered(x.y) : 0u;
                k2[u] = have && c4 + 2 < nvalid ? float_to_ordered(x.z) : 0u;
                k3[u] = have && c4 + 3 < nvalid ? float_to_ordered(x.w) : 0u;
                e0[u] = 0;
                e1[u] = 1;
                e2[u] = 2;
                e3[u] = 3;
                cas_desc(k0[u], e0[u], k1[u], e1[u]);
                cas_desc(k2[u], e2[u], k3[u], e3[u]);
                cas_desc(k0[u], e0[u], k2[u], e2[u]);
                cas_desc(k1[u], e1[u], k3[u], e3[u]);
                cas_desc(k1[u], e1[u], k2[u], e2[u]);
                // the list goes over the row's first 2K logits (a missing second row reuses
                // the first row's slots at offset 64: it is never read back)
                lv[u] = zr + (have ? 0 : 64);
                li[u] = reinterpret_cast<int *>(lv[u] + kMaxTopK);
            }
            __syncwarp();  // every lane has read its logits before the lists overwrite them
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (lane < K) {
                    lv[u][lane] = -INFINITY;
                    li[u][lane] = INT_MAX;
                }
            __syncwarp();
#pragma unroll
            for (int r = 0; r < kMaxTopK; ++r) {
                if (r >= K) break;
                uint32_t m[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) m[u] = __reduce_max_sync(0xFFFFFFFFu, k0[u]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const bool cand = m[u] != 0u && k0[u] == m[u];
                    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, cand);
                    const bool pop = cand && (hit & lt) == 0u;
                    if (pop) {
                        lv[u][r] = ordered_to_float(m[u]);
                        li[u][r] = c.v0 + c4 + e0[u];
                    }
                    k0[u] = pop ? k1[u] : k0[u];
                    e0[u] = pop ? e1[u] : e0[u];
                    k1[u] = pop ? k2[u] : k1[u];
                    e1[u] = pop ? e2[u] : e1[u];
                    k2[u] = pop ? k3[u] : k2[u];
                    e2[u] = pop ? e3[u] : e2[u];
                    k3[u] = pop ? 0u : k3[u];
                }
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int row = r0 + u * kEpiWarps;
                if (lane < K && row < p.M) {
                    const size_t o = ((static_cast<size_t>(row) * p.k + c.s) * p.T + c.t) * K;
                    p.ws.tkv[o + lane] = lv[u][lane];
                    p.ws.tki[o + lane] = li[u][lane];
                }
            }
        }
    }
    epi_bar_sync();
}

// ------------------------------------------------------------------ epilogue, rows mode
// Thread (quadrant q, half h, lane) owns row m0 + 32q + lane and the 128 columns
// [v0 + 128h, v0 + 128h + 128) of the 256-column tile, i.e. record tile 2t + h.  It walks
// them in chunks of 32: chunk max and first argmax, online rescale of the running sum, then
// the sum of exp against the running max.
// tempty_remote: the cluster address of the pair leader's accumulator-empty barrier when this
// CTA is the peer of a CTA pair (0: arrive on tempty_b in this CTA).
template <int EPI>
__device__ __forceinline__ void epilogue_rows(const GemmParams &p, const TileCoord &c,
                                              uint32_t taddr, uint64_t *tempty_b, int q, int h,
                                              int lane, uint32_t tempty_remote) {
    constexpr bool GUMBEL = EPI == kEpiGumbel;
    constexpr bool FULL = EPI == kEpiFull;
    constexpr bool TOPK = EPI == kEpiTopk || EPI == kEpiTopk8 || EPI == kEpiTopk4;
    constexpr int KL = EPI == kEpiTopk4 ? 4 : (EPI == kEpiTopk8 ? 8 : kMaxTopK);
    const int row = c.m0 + 32 * q + lane;
    const bool rv = row < p.M;
    const int rt = 2 * c.t + h;                 // record tile within the shard
    const int cbase0 = c.v0 + kRecordCols * h;  // first column of this half
    const int tgt = ((p.flags & kFlagTargets) && rv) ? __ldg(p.targets + row) : -1;
    float rm = -INFINITY, rs = 0.f, gk = -INFINITY, gz = 0.f;
    int ri = INT_MAX, gi = INT_MAX;
    // top-K: a sorted list (largest first) of the KL largest keys seen (KL >= K); only the
    // first K are written.  A key is the logit's order-preserving 32-bit image with its low
    // 7 bits replaced by 127 - (column offset in the record): one unsigned compare orders
    // by value, equal values by ascending column, and an insertion is one max and one min
    // per entry.  The value read back (tag bits cleared) is within 127 units in the last
    // place of the logit (8e-6 relative); values closer than that may order by column.
    // Key 0 = empty.
    uint32_t tk[TOPK ? KL : 1];
    if (TOPK) {
#pragma unroll
        for (int r = 0; r < KL; ++r) tk[r] = 0u;
    }
    constexpr int kChunks = kRecordCols / 32;
#pragma unroll 1
    for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t raw[32];
        tmem_ld32x32b_x32(taddr + kRecordCols * h + ch * 32, raw);
        if (ch == kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (tempty_remote)
                    mbar_arrive_remote(tempty_remote);
                else
                    mbar_arrive(tempty_b);
            }
        }
        const int cb = cbase0 + ch * 32;
        const int nval = min(32, c.v_end - cb);
        if (nval <= 0) continue;
        float y[32];
        if (nval == 32) {  // a whole chunk (every one but a shard's last): no column mask
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float z = __uint_as_float(raw[j]);
                y[j] = GUMBEL ? z * p.inv_t : z;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float z = __uint_as_float(raw[j]);
                y[j] = (j < nval) ? (GUMBEL ? z * p.inv_t : z) : -INFINITY;
            }
        }
        float cm = -INFINITY;
        int cj = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (y[j] > cm) {
                cm = y[j];
                cj = j;
            }
        if (cm > rm) {
            rs *= ex2_approx((rm - cm) * kLog2e);
            rm = cm;
            ri = cb + cj;
        }
        const float mb = rm * kLog2e;
#pragma unroll
        for (int j = 0; j < 32; ++j) rs += ex2_approx(fmaf(y[j], kLog2e, -mb));
        if (GUMBEL && rv) {
            // consecutive columns are consecutive stream indices: the state advances by one
            // golden-ratio increment per column
            unsigned long long st = splitmix_state(
                p.seed, static_cast<unsigned long long>(row) * static_cast<unsigned>(p.V) +
                            static_cast<unsigned>(cb));
            // columns past the shard end have y = -inf, so their key is -inf and never wins;
            // keys are compared less the constant -ln(ln 2), added back per record
#pragma unroll
            for (int j = 0; j < 32; ++j, st += kGolden) {
                const float key = gumbel_key_less_c0(y[j], bits24_from_state(st));
                if (key > gk) {
                    gk = key;
                    gi = cb + j;
                    gz = __uint_as_float(raw[j]);
                }
            }
        }
        if (TOPK) {
            // insertion without branches: the key passes down the list, each entry keeping
            // the larger of itself and the passing key (invalid columns, past the shard end,
            // carry key 0 and change nothing)
            const uint32_t tag0 = 127u - static_cast<uint32_t>(ch * 32);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                uint32_t x = (float_to_ordered(y[j]) & 0xFFFFFF80u) | (tag0 - j);
                if (nval != 32) x = j < nval ? x : 0u;
#pragma unroll
                for (int r = 0; r < KL; ++r) {
                    const uint32_t hi = max(tk[r], x);
                    x = min(tk[r], x);
                    tk[r] = hi;
                }
            }
        }
        if (tgt >= cb && tgt < cb + nval) {
            // an explicit select chain: written as "pick raw[tgt - cb]" the compiler moves
            // raw[] to local memory to index it
            uint32_t tzv = 0u;
            const int off = tgt - cb;
#pragma unroll
            for (int j = 0; j < 32; ++j) tzv = select_u32(j == off, raw[j], tzv);
            p.ws.tz[row] = __uint_as_float(tzv);
        }
        if (FULL && rv) {
            uint16_t *dst = p.logits + static_cast<size_t>(row) * p.V + cb;
            const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(dst)) & 31u;
            if (nval == 32 && (mis & 15u) == 0) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    pk[j] = static_cast<uint32_t>(bf16_bits_rn(__uint_as_float(raw[2 * j]))) |
                            (static_cast<uint32_t>(bf16_bits_rn(__uint_as_float(raw[2 * j + 1])))
                             << 16);
                if (mis == 0) {
                    // the chunk's 64 bytes are two whole sectors: one 32-byte store each, so
                    // no sector reaches L2 in two halves
                    st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
                    st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14],
                                 pk[15]);
                } else {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d4[j] =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nval) dst[j] = bf16_bits_rn(__uint_as_float(raw[j]));
            }
        }
    }
    if (rv && rt < p.T) {
        const size_t o = (static_cast<size_t>(row) * p.k + c.s) * p.T + rt;
        p.ws.m[o] = rm;
        p.ws.idx[o] = ri;
        p.ws.s[o] = rs;
        if (GUMBEL) {
            p.ws.gk[o] = gk + kGumbelC0;
            p.ws.gi[o] = gi;
            p.ws.gz[o] = gz;
        }
        if (TOPK) {
#pragma unroll
            for (int r = 0; r < KL; ++r) {
                if (r >= p.topk) break;
                const uint32_t key = tk[r];
                // the value without the column tag: equal logits of different records read
                // back identical, so the combine's column tie-break orders them
                p.ws.tkv[o * p.topk + r] = key ? ordered_to_float(key & 0xFFFFFF80u) : -INFINITY;
                p.ws.tki[o * p.topk + r] =
                    key ? cbase0 + 127 - static_cast<int>(key & 0x7Fu) : INT_MAX;
            }
        }
    }
}

// ------------------------------------------------------------------ the kernel
// One K block (the 64 columns from k0) of the 128 W rows from `row` (a tile of shard c.s):
// from the row-major W through a 2-D map, or from the packed copy (sb_pack_weights: each
// such box 16 KB contiguous in memory) through a 4-D map (element, row in the tile, K
// block, tile of the packed layout).
__device__ __forceinline__ int packed_tile(const GemmParams &p, const TileCoord &c, int row) {
    return c.s * p.t128 + (row - c.s * p.S) / kTileA;
}
__device__ __forceinline__ void load_w_block(void *dst, const CUtensorMap *tm, uint64_t *bar,
                                             const GemmParams &p, const TileCoord &c, int k0,
                                             int row, uint64_t policy) {
    if (p.packed)
        tma_load_4d(dst, tm, bar, 0, 0, k0 / kBlockK, packed_tile(p, c, row), policy);
    else
        tma_load_2d(dst, tm, bar, k0, row, policy);
}
__device__ __forceinline__ void load_w_block_pair(void *dst, const CUtensorMap *tm,
                                                  uint32_t bar_cluster, const GemmParams &p,
                                                  const TileCoord &c, int k0, int row,
                                                  uint64_t policy) {
    if (p.packed)
        tma_load_4d_pair(dst, tm, bar_cluster, 0, 0, k0 / kBlockK, packed_tile(p, c, row),
                         policy);
    else
        tma_load_2d_pair(dst, tm, bar_cluster, k0, row, policy);
}

// Vocab mode with 16-row H blocks: one producer per operand ring, so that H (re-read from
// L2, 2 KB per stage) takes 4 stages and W (streamed from HBM) every other stage that fits:
// decode at 16 rows is bound by the W bytes in flight.
__device__ __forceinline__ void produce_ring(const GemmParams &p, const CUtensorMap *tm,
                                             uint8_t *ring, uint32_t stage_bytes, int stages,
                                             uint64_t *full, uint64_t *empty, bool is_a,
                                             uint64_t policy, int unit0, int unit_stride,
                                             volatile int *abort_flag, uint32_t pre) {
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < p.num_tiles; tile += unit_stride) {
        const TileCoord c = tile_coord<true>(p, tile, 0);
        const int row = is_a ? c.a_row : c.b_row;
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (issued < pre) {  // already issued before the wait on the previous kernel
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                continue;
            }
            if (!bwait(&empty[stage], phase ^ 1u, abort_flag, p)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&full[stage], stage_bytes);
            if (is_a)
                load_w_block(ring + stage * stage_bytes, tm, &full[stage], p, c, kb * kBlockK,
                             row, policy);
            else
                tma_load_2d(ring + stage * stage_bytes, tm, &full[stage], kb * kBlockK, row,
                            policy);
            ++issued;
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // Drain: the last `stages` issues may still be landing (only possible after an abort;
    // on the normal path the MMA warp consumed every one of them).
    const uint32_t n = issued < static_cast<uint32_t>(stages) ? issued : stages;
    for (uint32_t i = issued - n; i < issued; ++i)
        if (!bwait_drain(&full[i % stages], (i / stages) & 1u, abort_flag, p)) break;
}

// Vocab mode from 32 rows of H up: one ring of joint stages, each holding one K block of W
// (128 vocabulary rows, operand A, 16 KB) and of H (all M rows, operand B); one thread loads
// both, so the MMA warp waits once and commits once per K block.  The first `pre` stages' W copies (and their
// expect) went out before the wait on the previous kernel; their H copies go out here.
__device__ __forceinline__ void produce_vocab(const GemmParams &p, const CUtensorMap *tmA,
                                              const CUtensorMap *tmB, uint8_t *sA, uint8_t *sB,
                                              uint32_t b_bytes, uint64_t *full, uint64_t *empty,
                                              int unit0, int unit_stride,
                                              volatile int *abort_flag, uint32_t pre) {
    const int stages = p.stages_a;
    const uint64_t pol_w = policy_evict_first(), pol_h = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < p.num_tiles; tile += unit_stride) {
        const TileCoord c = tile_coord<true>(p, tile, 0);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (issued >= pre) {
                if (!bwait(&empty[stage], phase ^ 1u, abort_flag, p)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], kStageBytesA + b_bytes);
                load_w_block(sA + stage * kStageBytesA, tmA, &full[stage], p, c, kb * kBlockK,
                             c.a_row, pol_w);
            }
            tma_load_2d(sB + stage * b_bytes, tmB, &full[stage], kb * kBlockK, c.b_row, pol_h);
            ++issued;
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // Drain: the last `stages` issues may still be landing (only possible after an abort;
    // on the normal path the MMA warp consumed every one of them).
    const uint32_t n = issued < static_cast<uint32_t>(stages) ? issued : stages;
    for (uint32_t i = issued - n; i < issued; ++i)
        if (!bwait_drain(&full[i % stages], (i / stages) & 1u, abort_flag, p)) break;
}

// Rows mode: the L2 policy of the W copies (kWEvictFirstGroups).
__device__ __forceinline__ uint64_t rows_w_policy(const GemmParams &p) {
    return p.m_groups <= kWEvictFirstGroups ? policy_evict_first() : policy_evict_last();
}

// Rows mode (CTA pairs): one ring of joint stages, each holding this CTA's 128 H rows (A)
// and its half of the W tile (B) for one K block of ATOMS 64-wide atoms (16 KB per atom and
// operand); one thread per CTA loads both.  The leader's full barrier counts every
// copy of the pair; the peer's copies complete on it (at the same offset), and the leader's
// single MMA commit per stage frees the stage in both CTAs (the peer waits on its own empty
// barrier with cluster-scope acquire).  The first `pre` stages' W copies (and the leader's
// expect) went out before the wait on the previous kernel; their H copies go out here.
template <int ATOMS>
__device__ __forceinline__ void produce_pair(const GemmParams &p, const CUtensorMap *tmA,
                                             const CUtensorMap *tmB, uint8_t *sA, uint8_t *sB,
                                             uint32_t b_atom, uint64_t *full, uint64_t *empty,
                                             int rank, int unit0, int unit_stride,
                                             volatile int *abort_flag, uint32_t pre) {
    const bool peer = rank == 1;
    const int stages = p.stages_a;
    const uint32_t a_stage = kStageBytesA * ATOMS, b_stage = b_atom * ATOMS;
    const uint64_t pol_a = policy_evict_last(), pol_b = rows_w_policy(p);
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < p.num_tiles; tile += unit_stride) {
        const TileCoord c = tile_coord<false>(p, tile, rank);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            const bool w_done = issued < pre;
            if (!w_done) {
                if (!bwait_cl(&empty[stage], phase ^ 1u, abort_flag, p)) {
                    ok = false;
                    break;
                }
                if (!peer) mbar_arrive_expect_tx(&full[stage], 2 * (a_stage + b_stage));
            }
            uint8_t *da = sA + stage * a_stage;
            uint8_t *db = sB + stage * b_stage;
            const uint32_t fb = peer ? mapa_rank(&full[stage], 0) : 0u;
#pragma unroll
            for (int at = 0; at < ATOMS; ++at) {
                const int k0 = (kb * ATOMS + at) * kBlockK;  // past d: read as zeros
                if (peer) {
                    tma_load_2d_pair(da + at * kStageBytesA, tmA, fb, k0, c.a_row, pol_a);
                    if (!w_done)
                        load_w_block_pair(db + at * b_atom, tmB, fb, p, c, k0, c.b_row, pol_b);
                } else {
                    tma_load_2d(da + at * kStageBytesA, tmA, &full[stage], k0, c.a_row, pol_a);
                    if (!w_done)
                        load_w_block(db + at * b_atom, tmB, &full[stage], p, c, k0, c.b_row,
                                     pol_b);
                }
            }
            ++issued;
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (peer) {
        // the peer cannot observe its copies (they complete on the leader's barrier); after
        // an abort it gives the last ones a bounded time to land (they were issued at least
        // one wait limit before an abort can happen, so this is normally already the case)
        if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 50000u) {
            }
        }
        return;
    }
    // The leader's barrier also waits for the peer's bytes, which never come for a stage the
    // peer did not issue: the drain stops at the first wait that runs out.
    const uint32_t n = issued < static_cast<uint32_t>(stages) ? issued : stages;
    for (uint32_t i = issued - n; i < issued; ++i)
        if (!bwait_drain(&full[i % stages], (i / stages) & 1u, abort_flag, p)) break;
}

// ATOMS: rows mode, 64-wide K slices per joint stage.  JOINT: vocab mode, one joint ring
// (otherwise one ring per operand).
template <bool VOCAB, int EPI, int ATOMS, bool JOINT>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const GemmParams p, const uint32_t tmem_cols) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const SmemLayout L = make_layout(p.nb, p.stages_a, p.stages_b, VOCAB, p.flags, p.topk,
                                     ATOMS);
    uint8_t *sA = smem + L.a_off;
    uint8_t *sB = smem + L.b_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *fullA = bars;
    uint64_t *emptyA = bars + kMaxStages;
    uint64_t *fullB = bars + 2 * kMaxStages;
    uint64_t *emptyB = bars + 3 * kMaxStages;
    uint64_t *tfull = bars + 4 * kMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *stall = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);
    int32_t *tgt_s = reinterpret_cast<int32_t *>(smem + L.tgt_off);
    float *scratch = reinterpret_cast<float *>(smem + L.scratch_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Rows mode runs on CTA pairs (2-CTA clusters): one cta_group::2 MMA (M = 256) per K
    // step, issued by rank 0, with each CTA staging only its half of the W tile (UMMA B split
    // along N) and its own H tile (A split along M); each CTA's TMEM holds its 128 rows.  The
    // peer's copies complete on the leader's stage barriers, which count both CTAs' bytes.
    constexpr int CS = VOCAB ? 1 : kRowsCluster;
    constexpr bool PAIR = !VOCAB;
    // B bytes per 64-wide K atom (vocab mode: one atom per stage; rows mode: ATOMS)
    const uint32_t b_stage_bytes = static_cast<uint32_t>(PAIR ? p.nb / 2 : p.nb) * 128u;
    // CTAs of a cluster walk the same work units in lockstep (same ring positions).
    const int rank = CS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit0 = blockIdx.x / CS;
    const int unit_stride = gridDim.x / CS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages_a; ++i) {
            mbar_init(&fullA[i], 1);
            mbar_init(&emptyA[i], 1);
        }
        for (int i = 0; i < p.stages_b; ++i) {
            mbar_init(&fullB[i], 1);
            mbar_init(&emptyB[i], 1);  // one MMA commit (in a pair: the leader's)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            // pair: the leader's accumulator is free once both CTAs' epilogues are done
            mbar_init(&tempty[i], PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(stall, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if (PAIR) {  // both CTAs' warps allocate together
            tmem_alloc2(tmem_slot, tmem_cols);
            tmem_relinquish2();
        } else {
            tmem_alloc(tmem_slot, tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (CS > 1) cluster_sync();  // the peer's barriers are initialised before any copy lands
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The setup above touches no global memory, so it overlaps the previous kernel in the
    // stream (this kernel is a programmatic dependent launch).  In vocab mode W (operand A)
    // is the output-head weight, which that kernel does not write, so ring A's first stages
    // are filled before the wait (the W stream starts under the previous kernel's tail); H,
    // the targets and the workspace may belong to that kernel, so everything else waits.
    uint32_t a_pre = 0;
    if (VOCAB && warp == 0 && lane == 0 && unit0 < p.num_tiles) {
        a_pre = static_cast<uint32_t>(p.stages_a < p.kblocks ? p.stages_a : p.kblocks);
        const TileCoord c = tile_coord<VOCAB>(p, unit0, rank);
        const uint64_t pol = policy_evict_first();
        for (uint32_t kb = 0; kb < a_pre; ++kb) {
            mbar_arrive_expect_tx(&fullA[kb], kStageBytesA + (JOINT ? b_stage_bytes : 0u));
            load_w_block(sA + kb * kStageBytesA, &tmA, &fullA[kb], p, c,
                         static_cast<int>(kb) * kBlockK, c.a_row, pol);
        }
    }
    // Rows mode with CTA pairs: the same for W, operand B, in both CTAs of the pair, into the
    // joint stages (the leader expects the whole stage, H included, which its producer loads
    // after the wait; the peer's copies complete on the leader's barriers).
    uint32_t b_pre = 0;
    if (PAIR && warp == 0 && lane == 0 && unit0 < p.num_tiles) {
        b_pre = static_cast<uint32_t>(p.stages_a < p.kblocks ? p.stages_a : p.kblocks);
        const TileCoord c = tile_coord<VOCAB>(p, unit0, rank);
        const uint64_t pol = rows_w_policy(p);
        for (uint32_t kb = 0; kb < b_pre; ++kb) {
            uint8_t *dst = sB + kb * b_stage_bytes * ATOMS;
            if (rank == 0)
                mbar_arrive_expect_tx(&fullA[kb], 2 * ATOMS * (kStageBytesA + b_stage_bytes));
#pragma unroll
            for (int at = 0; at < ATOMS; ++at) {
                const int k0 = (static_cast<int>(kb) * ATOMS + at) * kBlockK;
                if (rank == 0)
                    load_w_block(dst + at * b_stage_bytes, &tmB, &fullA[kb], p, c, k0, c.b_row,
                                 pol);
                else
                    load_w_block_pair(dst + at * b_stage_bytes, &tmB, mapa_rank(&fullA[kb], 0),
                                      p, c, k0, c.b_row, pol);
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.ws.epoch = p.epoch;
    if (VOCAB && (p.flags & kFlagTargets))
        for (int i = threadIdx.x; i < p.M; i += blockDim.x) tgt_s[i] = p.targets[i];
    // Scoring targets outside [0, V) would leave their log-prob undefined: CTA 0 checks them
    // and reports SB_ERR_INVALID_ARG through the status word (the outputs stay undefined).
    if (blockIdx.x == 0 && (p.flags & kFlagTargets)) {
        bool bad = false;
        for (int i = threadIdx.x; i < p.M; i += blockDim.x) {
            const int t = p.targets[i];
            bad |= (t < 0 || t >= p.V);
        }
        if (bad) record_status(p.ws.status, p.epoch, 1u);  // SB_ERR_INVALID_ARG
    }
    if (VOCAB && (p.flags & kFlagTargets)) __syncthreads();  // tgt_s is complete
    // Let the record combine (a programmatic dependent launch) get scheduled early; it
    // waits for this whole grid to finish before it reads any record.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------ TMA producers (one lane each):
        // warp 0 fills the joint stages (warp 2 then has no work), or, in vocab mode with
        // separate rings, warp 0 ring A (W) and warp 2 ring B (H).
        if (lane == 0) {
            if (!VOCAB) {
                if (warp == 0)
                    produce_pair<ATOMS>(p, &tmA, &tmB, sA, sB, b_stage_bytes, fullA, emptyA, rank,
                                 unit0, unit_stride, abort_flag, b_pre);
            } else if (JOINT) {
                if (warp == 0)
                    produce_vocab(p, &tmA, &tmB, sA, sB, b_stage_bytes, fullA, emptyA, unit0,
                                  unit_stride, abort_flag, a_pre);
            } else if (warp == 0) {
                produce_ring(p, &tmA, sA, kStageBytesA, p.stages_a, fullA, emptyA, true,
                             policy_evict_first(), unit0, unit_stride, abort_flag, a_pre);
            } else {
                produce_ring(p, &tmB, sB, b_stage_bytes, p.stages_b, fullB, emptyB, false,
                             policy_evict_last(), unit0, unit_stride, abort_flag, 0);
            }
        }
    } else if (warp == 1) {
        if (PAIR && rank == 1) {
            // pair peer: its copies complete on the leader's barriers; no MMA to issue
        } else if (PAIR) {
            // ------------------------------------------------ pair leader: one M = 256 MMA
            // over both CTAs' stages per K step
            if (lane == 0) {
                const uint32_t idesc = idesc_bf16_f32(2 * kTileA, p.nb);
                constexpr uint16_t kBoth = 3;
                // descriptors of stage 0; a stage / atom / 16-column step adds its byte offset
                // >> 4 to the start-address field (shared memory stays below 256 KB, so the
                // 14-bit field never carries)
                const uint64_t adesc0 = sw128_kmajor_desc(smem_u32(sA));
                const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(sB));
                const uint32_t a_step = (kStageBytesA * ATOMS) >> 4;
                const uint32_t b_step = (b_stage_bytes * ATOMS) >> 4;
                int st = 0;
                uint32_t ph = 0, a_off = 0, b_off = 0;
                bool ok = true, any = false;
                int it = 0;
                for (int tile = unit0; ok && tile < p.num_tiles; tile += unit_stride, ++it) {
                    const int b = it & 1;
                    const uint32_t tph = (it >> 1) & 1;
                    if (!bwait_cl(&tempty[b], tph ^ 1u, abort_flag, p)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.nb);
                    for (int kb = 0; kb < p.kblocks; ++kb) {
                        // the leader's barrier counts the whole joint stage of both CTAs
                        if (!bwait(&fullA[st], ph, abort_flag, p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int at = 0; at < ATOMS; ++at) {
                            const uint64_t adesc = adesc0 + a_off + at * (kStageBytesA >> 4);
                            const uint64_t bdesc = bdesc0 + b_off + at * (b_stage_bytes >> 4);
#pragma unroll
                            for (int ks = 0; ks < kBlockK / 16; ++ks)
                                umma_bf16_pair(d_tmem, adesc + 2u * ks, bdesc + 2u * ks, idesc,
                                               (kb | at | ks) != 0 ? 1u : 0u);
                        }
                        // one commit per stage (each commit costs the tensor pipe time):
                        // frees the joint stage in both CTAs
                        umma_commit_pair(&emptyA[st], kBoth);
                        any = true;
                        a_off += a_step;
                        b_off += b_step;
                        if (++st == p.stages_a) {
                            st = 0;
                            ph ^= 1u;
                            a_off = 0;
                            b_off = 0;
                        }
                    }
                    if (ok) umma_commit_pair(&tfull[b], kBoth);
                }
                if (any) {  // wait until every MMA this thread issued has completed
                    umma_commit_pair(drain, 1);
                    bwait_drain(drain, 0, abort_flag, p);
                }
            }
        } else if (lane == 0) {
            // ------------------------------------------------ MMA issuer (one lane, vocab mode)
            const uint32_t idesc = idesc_bf16_f32(kTileA, p.nb);
            int st = 0, sb = 0;
            uint32_t ph = 0, pb = 0;
            bool ok = true, any = false;
            int it = 0;
            for (int tile = unit0; ok && tile < p.num_tiles; tile += unit_stride, ++it) {
                const int b = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (!bwait(&tempty[b], tph ^ 1u, abort_flag, p)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.nb);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!bwait(&fullA[st], ph, abort_flag, p) ||
                        (!JOINT && !bwait(&fullB[sb], pb, abort_flag, p))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + st * kStageBytesA));
                    const uint64_t bdesc =
                        sw128_kmajor_desc(smem_u32(sB + (JOINT ? st : sb) * b_stage_bytes));
#pragma unroll
                    for (int ks = 0; ks < kBlockK / 16; ++ks)
                        umma_bf16(d_tmem, adesc + 2u * ks, bdesc + 2u * ks, idesc,
                                  (kb | ks) != 0 ? 1u : 0u);
                    umma_commit(&emptyA[st]);  // joint ring: frees the whole stage
                    if (!JOINT) umma_commit(&emptyB[sb]);
                    any = true;
                    if (++st == p.stages_a) {
                        st = 0;
                        ph ^= 1u;
                    }
                    if (!JOINT && ++sb == p.stages_b) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
                if (ok) umma_commit(&tfull[b]);
            }
            if (any) {  // wait until every MMA this thread issued has completed
                umma_commit(drain);
                bwait_drain(drain, 0, abort_flag, p);
            }
        }
    } else {
        // ------------------------------------------------ epilogue warps 3..10
        const int q = warp & 3;              // TMEM lane quadrant this warp may read
        const int h = (warp - 3) >> 2;       // which of the quadrant's two warps
        int it = 0;
        for (int tile = unit0; tile < p.num_tiles; tile += unit_stride, ++it) {
            const int b = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            bool ok;
            if (p.debug_stall)
                ok = bwait(stall, 0, abort_flag, p);  // nothing ever arrives here
            else if (PAIR)
                ok = bwait_cl(&tfull[b], tph, abort_flag, p);  // the leader's commit
            else
                ok = bwait(&tfull[b], tph, abort_flag, p);
            if (epi_vote_any(!ok)) break;
            tc_fence_after();
            const TileCoord c = tile_coord<VOCAB>(p, tile, rank);
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * p.nb);
            if (VOCAB)
                epilogue_vocab<EPI>(p, c, taddr, &tempty[b], q, h, lane, tgt_s, scratch);
            else
                epilogue_rows<EPI>(p, c, taddr, &tempty[b], q, h, lane,
                                   PAIR && rank == 1 ? mapa_rank(&tempty[b], 0) : 0u);
        }
    }

    tc_fence_before();
    __syncthreads();
    // Every role has drained what it issued (its TMA copies, its MMAs and their commits to
    // the peers); wait until the peers have too, so nothing lands here after exit.
    if (CS > 1) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc2(tmem_base, tmem_cols);
        else
            tmem_dealloc(tmem_base, tmem_cols);
    }
}

template <bool VOCAB, int EPI, int ATOMS, bool JOINT>
cudaError_t launch_t1(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p,
                     size_t smem, int num_sms, cudaStream_t stream) {
    constexpr int CS = VOCAB ? 1 : kRowsCluster;
    auto kern = lmhead_kernel<VOCAB, EPI, ATOMS, JOINT>;
    // The shared-memory opt-in is per device; every launch asks for at most kSmemLimit.
    static std::atomic<uint64_t> opted_in{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(opted_in.load() & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
        if (e != cudaSuccess) return e;
        opted_in.fetch_or(bit);
    }
    uint32_t cols = 512;
    if (VOCAB) {
        cols = 32;
        while (cols < static_cast<uint32_t>(2 * p.nb)) cols <<= 1;
    }
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // a programmatic dependent of the previous kernel in the stream: its CTAs may start
    // their setup early and wait (griddepcontrol.wait) before touching global memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // persistent grid: as many clusters as can be resident at once (one CTA per SM)
    int clusters = num_sms / CS;
    if (CS > 1) {
        // co-resident clusters (GPCs may not pair every SM), queried for this launch's
        // shared-memory footprint and cached per device for the last footprint asked
        static std::atomic<unsigned long long> cache_by_dev[64];  // (smem << 32) | active
        const unsigned long long c = dev < 64 ? cache_by_dev[dev].load() : 0;
        int active = (c >> 32) == smem ? static_cast<int>(c & 0xFFFFFFFFu) : 0;
        if (active <= 0) {
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3(CS * clusters);
            if (cudaOccupancyMaxActiveClusters(&active, kern, &q) != cudaSuccess) active = 0;
            if (active > 0 && dev < 64)
                cache_by_dev[dev].store((static_cast<unsigned long long>(smem) << 32) |
                                        static_cast<unsigned>(active));
        }
        if (active > 0) clusters = active < clusters ? active : clusters;
    }
    if (clusters > p.num_tiles) clusters = p.num_tiles;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(CS * clusters);
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p, cols);
}

// The kernel specialised for the call's pipeline: rows mode, atoms per joint stage (1 or 2);
// vocab mode, joint ring or one ring per operand.
template <bool VOCAB, int EPI>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p,
                     size_t smem, int num_sms, cudaStream_t stream) {
    if constexpr (!VOCAB) {
        if (p.atoms == kMaxPairAtoms)
            return launch_t1<false, EPI, kMaxPairAtoms, true>(tmA, tmB, p, smem, num_sms,
                                                              stream);
        return launch_t1<false, EPI, 1, true>(tmA, tmB, p, smem, num_sms, stream);
    } else {
        if (p.joint)
            return launch_t1<true, EPI, 1, true>(tmA, tmB, p, smem, num_sms, stream);
        return launch_t1<true, EPI, 1, false>(tmA, tmB, p, smem, num_sms, stream);
    }
}

// The packed copy of W (layout in sb.h at sb_pack_weights): one thread per 16 bytes of the
// packed buffer, zeros for the rows past a shard's end in its last tile and for the
// columns past d in the last K block.
__global__ void pack_weights_kernel(const uint4 *__restrict__ W, uint4 *__restrict__ P,
                                    long long V, long long d, int k) {
    const long long S = V / k, t128 = (S + kTileA - 1) / kTileA;
    const long long kbs = (d + kBlockK - 1) / kBlockK, d8 = d / 8;
    const long long n = static_cast<long long>(k) * t128 * kbs * kTileA * (kBlockK / 8);
    for (long long o = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; o < n;
         o += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long j8 = o % (kBlockK / 8);
        const long long i = (o / (kBlockK / 8)) % kTileA;
        const long long kb = (o / (kBlockK / 8 * kTileA)) % kbs;
        const long long tile = o / (kBlockK / 8 * kTileA * kbs);
        const long long s = tile / t128, t = tile % t128;
        const long long r = t * kTileA + i;  // row within the shard
        const long long c8 = kb * (kBlockK / 8) + j8;
        P[o] = (r < S && c8 < d8) ? W[(s * S + r) * d8 + c8] : make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace

cudaError_t launch_pack_weights(const void *W, void *P, long long V, long long d, int k,
                                int num_sms, cudaStream_t stream) {
    pack_weights_kernel<<<num_sms * 8, 256, 0, stream>>>(static_cast<const uint4 *>(W),
                                                         static_cast<uint4 *>(P), V, d, k);
    return cudaGetLastError();
}

size_t lmhead_smem_bytes(int nb, int stages_a, int stages_b, bool vocab_mode, int flags,
                         int topk, int atoms) {
    return make_layout(nb, stages_a, stages_b, vocab_mode, flags, topk, atoms).total;
}

cudaError_t launch_lmhead(bool vocab_mode, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const GemmParams &p, size_t smem, int num_sms, cudaStream_t stream) {
    const int epi = (p.flags & kFlagGumbel) ? kEpiGumbel
                    : (p.flags & kFlagFull) ? kEpiFull
                    : (p.flags & kFlagTopk) ? kEpiTopk
                                            : kEpiPlain;
    switch (epi) {
    case kEpiGumbel:
        return vocab_mode ? launch_t<true, kEpiGumbel>(tmA, tmB, p, smem, num_sms, stream)
                          : launch_t<false, kEpiGumbel>(tmA, tmB, p, smem, num_sms, stream);
    case kEpiFull:
        return vocab_mode ? launch_t<true, kEpiFull>(tmA, tmB, p, smem, num_sms, stream)
                          : launch_t<false, kEpiFull>(tmA, tmB, p, smem, num_sms, stream);
    case kEpiTopk:
        if (vocab_mode) return launch_t<true, kEpiTopk>(tmA, tmB, p, smem, num_sms, stream);
        if (p.topk <= 4) return launch_t<false, kEpiTopk4>(tmA, tmB, p, smem, num_sms, stream);
        if (p.topk <= 8) return launch_t<false, kEpiTopk8>(tmA, tmB, p, smem, num_sms, stream);
        return launch_t<false, kEpiTopk>(tmA, tmB, p, smem, num_sms, stream);
    default:
        return vocab_mode ? launch_t<true, kEpiPlain>(tmA, tmB, p, smem, num_sms, stream)
                          : launch_t<false, kEpiPlain>(tmA, tmB, p, smem, num_sms, stream);
    }
}

}  // namespace sb
