// sb_api.cu -- host side of the libsb C ABI: argument validation, workspace layout,
// TMA tensor-map encoding, variant choice and kernel launches on the caller's stream.
// The library allocates no device memory and never synchronises.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sb.h"
#include "sb_internal.h"

namespace {
using namespace sb;

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

std::atomic<uint32_t> g_epoch{0x5B000000u};
std::atomic<int> g_debug_stall{0};
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct WsLayout {
    size_t m, idx, s, gk, gi, gz, tkv, tki, tz, total;
};

WsLayout ws_layout(int64_t M, int32_t k, int32_t T, bool gumbel, int topk = 0) {
    const size_t n = static_cast<size_t>(M) * k * T;
    WsLayout L{};
    size_t off = 256;
    L.m = off;
    off += al256(4 * n);
    L.idx = off;
    off += al256(4 * n);
    L.s = off;
    off += al256(4 * n);
    if (gumbel) {
        L.gk = off;
        off += al256(4 * n);
        L.gi = off;
        off += al256(4 * n);
        L.gz = off;
        off += al256(4 * n);
    }
    if (topk > 0) {
        L.tkv = off;
        off += al256(4 * n * topk);
        L.tki = off;
        off += al256(4 * n * topk);
    }
    L.tz = off;
    off += al256(4 * static_cast<size_t>(M));
    L.total = off;
    return L;
}

Workspace ws_views(void *base, const WsLayout &L, bool gumbel, int topk = 0) {
    uint8_t *b = static_cast<uint8_t *>(base);
    Workspace w{};
    w.epoch = reinterpret_cast<uint32_t *>(b);
    w.status = reinterpret_cast<unsigned long long *>(b + 8);
    w.m = reinterpret_cast<float *>(b + L.m);
    w.idx = reinterpret_cast<int32_t *>(b + L.idx);
    w.s = reinterpret_cast<float *>(b + L.s);
    if (gumbel) {
        w.gk = reinterpret_cast<float *>(b + L.gk);
        w.gi = reinterpret_cast<int32_t *>(b + L.gi);
        w.gz = reinterpret_cast<float *>(b + L.gz);
    }
    if (topk > 0) {
        w.tkv = reinterpret_cast<float *>(b + L.tkv);
        w.tki = reinterpret_cast<int32_t *>(b + L.tki);
    }
    w.tz = reinterpret_cast<float *>(b + L.tz);
    return w;
}

bool shape_ok(int64_t M, int64_t V, int32_t k) {
    return M >= 1 && M <= (int64_t(1) << 30) && V >= 1 && V < (int64_t(1) << 31) && k >= 1 &&
           k <= kMaxShards && V % k == 0;
}

bool vocab_mode(int64_t M) { return M <= kMaxVocabModeRows; }

// Records per (row, shard): one per 128 vocabulary columns, whatever the tiling.
int32_t tiles_per_shard(int64_t /*M*/, int64_t V, int32_t k) {
    const int64_t S = V / k;
    return static_cast<int32_t>((S + kRecordCols - 1) / kRecordCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A few recently encoded maps, keyed by everything the encoding depends on (a map holds no
// device state, so reusing one for the same pointer and shape is exact).
struct MapCacheEntry {
    const void *base;
    int64_t rows, d;
    int box_rows;
    int packed_k;  // 0: a 2-D map over a row-major matrix; k: the 4-D map of a packed W
    CUtensorMap map;
    bool used;
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapCacheEntry g_map_cache[kMapCache];
int g_map_next = 0;

// 2-D map over a row-major bf16 matrix [rows, d]: boxes of 64 x box_rows, 128-byte swizzle,
// out-of-range elements read as zero.
bool make_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t d, int box_rows) {
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (const auto &e : g_map_cache)
            if (e.used && e.base == base && e.rows == rows && e.d == d &&
                e.box_rows == box_rows && e.packed_k == 0) {
                *tm = e.map;
                return true;
            }
    }
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_map_cache[g_map_next] = MapCacheEntry{base, rows, d, box_rows, 0, *tm, true};
    g_map_next = (g_map_next + 1) % kMapCache;
    return true;
}

// The packed W layout of sb_pack_weights for V rows, d columns and k lane shards: tiles of
// 128 rows (ceil(S / 128) per shard) x K blocks of 64 columns, each block 16 KB contiguous.
int64_t packed_t128(int64_t V, int32_t k) { return (V / k + kTileA - 1) / kTileA; }
int64_t packed_kblocks(int64_t d) { return (d + kBlockK - 1) / kBlockK; }
size_t packed_bytes(int64_t V, int64_t d, int32_t k) {
    return static_cast<size_t>(k) * packed_t128(V, k) * packed_kblocks(d) * kTileA * kBlockK * 2;
}

// 4-D map over a packed W: (element, row in the tile, K block, tile), boxes of one 16 KB
// block, 128-byte swizzle (the same shared-memory image as a 64 x 128 box of the 2-D map).
bool make_packed_map(CUtensorMap *tm, const void *base, int64_t V, int64_t d, int32_t k) {
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (const auto &e : g_map_cache)
            if (e.used && e.base == base && e.rows == V && e.d == d && e.packed_k == k) {
                *tm = e.map;
                return true;
            }
    }
    auto enc = encoder();
    if (!enc) return false;
    const int64_t kbs = packed_kblocks(d);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(kBlockK), static_cast<cuuint64_t>(kTileA),
                          static_cast<cuuint64_t>(kbs),
                          static_cast<cuuint64_t>(k * packed_t128(V, k))};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(kBlockK) * 2,
                             static_cast<cuuint64_t>(kBlockK) * 2 * kTileA,
                             static_cast<cuuint64_t>(kBlockK) * 2 * kTileA * kbs};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(kTileA), 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    g_map_cache[g_map_next] = MapCacheEntry{base, V, d, kTileA, k, *tm, true};
    g_map_next = (g_map_next + 1) % kMapCache;
    return true;
}

struct DevInfo {
    int sms = 0, cc = 0;
};

int32_t current_device(DevInfo *out) {
    static DevInfo cache[64];
    static std::atomic<uint64_t> known{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SB_ERR_CUDA;
    if (dev < 64 && (known.load() >> dev) & 1) {
        *out = cache[dev];
    } else {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SB_ERR_CUDA;
        out->sms = sms;
        out->cc = major * 10 + minor;
        if (dev < 64) {
            cache[dev] = *out;
            known.fetch_or(uint64_t(1) << dev);
        }
    }
    return out->cc == 103 ? SB_OK : SB_ERR_UNSUPPORTED;
}

int32_t check_outputs(const sb_outputs *out, int32_t surface, bool need_ws) {
    if (!out || !out->token) return SB_ERR_INVALID_ARG;
    if (surface == SB_TOPK_LOGPROB &&
        (!out->topk_ids || !out->topk_logprob || out->topk < 1 || out->topk > kMaxTopK))
        return SB_ERR_INVALID_ARG;
    if ((surface == SB_TOKEN_LOGPROB || surface == SB_GUMBEL_TOKEN) && !out->token_logprob)
        return SB_ERR_INVALID_ARG;
    if (surface == SB_FULL_LOGITS && !out->logits_bf16) return SB_ERR_INVALID_ARG;
    if ((out->target_ids == nullptr) != (out->target_logprob == nullptr)) return SB_ERR_INVALID_ARG;
    if (need_ws && !out->workspace) return SB_ERR_INVALID_ARG;
    if (!aligned(out->token, 4) || !aligned(out->token_logprob, 4) || !aligned(out->lse, 4) ||
        !aligned(out->target_ids, 4) || !aligned(out->target_logprob, 4) ||
        !aligned(out->logits_bf16, 16) || !aligned(out->workspace, 256) ||
        (surface == SB_TOPK_LOGPROB &&
         (!aligned(out->topk_ids, 4) || !aligned(out->topk_logprob, 4))))
        return SB_ERR_ALIGNMENT;
    return SB_OK;
}

// Ring depths.  Joint ring (rows mode; vocab mode from 32 rows of H): one K block of both
// operands per stage (vocab mode: 128 W rows and all M rows of H; rows mode: this CTA's H
// rows and its half of the W tile for `atoms` 64-wide slices), as many as fit.  Vocab mode at
// 16 rows: one ring per operand, H a fixed depth and W every remaining stage (decode at
// 16 rows is bound by the W bytes in flight, and H costs only 2 KB per stage).
constexpr int kVocabStagesH = 4;
bool pick_stages(int nb, bool vm, bool joint, int atoms, int flags, int topk, int *sa,
                 int *sb) {
    const int at = vm ? 1 : atoms;
    for (*sa = kMaxStages; *sa > 1; --*sa) {
        *sb = joint ? *sa : kVocabStagesH;
        if (lmhead_smem_bytes(nb, *sa, *sb, vm, flags, topk, at) <= kSmemLimit) break;
    }
    *sb = joint ? *sa : kVocabStagesH;
    return lmhead_smem_bytes(nb, *sa, *sb, vm, flags, topk, at) <= kSmemLimit && *sa >= 2;
}

CombineParams combine_params(const sb_outputs *out, const Workspace &w, int64_t M, int32_t k,
                             int32_t T, int flags, float inv_t) {
    CombineParams c{};
    c.M = static_cast<int>(M);
    c.k = k;
    c.T = T;
    c.flags = flags;
    c.inv_t = inv_t;
    c.ws = w;
    c.token = out->token;
    c.token_logprob = out->token_logprob;
    c.lse = out->lse;
    c.target_logprob = out->target_ids ? out->target_logprob : nullptr;
    if (flags & kFlagTopk) {
        c.topk = out->topk;
        c.topk_ids = out->topk_ids;
        c.topk_logprob = out->topk_logprob;
    }
    return c;
}

}  // namespace

namespace sb {
bool encode_bf16_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols,
                     int box_rows) {
    return make_map(tm, base, rows, cols, box_rows);
}
int32_t device_sms_cc(int *sms, int *cc) {
    DevInfo dev;
    const int32_t e = current_device(&dev);
    if (sms) *sms = dev.sms;
    if (cc) *cc = dev.cc;
    return e;
}
uint32_t next_epoch() { return g_epoch.fetch_add(1) + 1; }
unsigned long long wait_limit_ns() { return g_timeout_ns.load(); }
}  // namespace sb

extern "C" {

size_t sb_workspace_bytes(int64_t M, int64_t V, int32_t k, int32_t surface) {
    surface &= ~SB_W_PACKED;  // the records do not depend on the layout of W
    if (!shape_ok(M, V, k) || surface < SB_TOKEN || surface > SB_TOPK_LOGPROB) return 0;
    return ws_layout(M, k, tiles_per_shard(M, V, k), surface == SB_GUMBEL_TOKEN,
                     surface == SB_TOPK_LOGPROB ? kMaxTopK : 0)
        .total;
}

int32_t sb_tiles_per_shard(int64_t M, int64_t V, int32_t k) {
    if (!shape_ok(M, V, k)) return -1;
    return tiles_per_shard(M, V, k);
}

size_t sb_packed_weight_bytes(int64_t V, int64_t d, int32_t k) {
    if (!shape_ok(1, V, k) || d < 8 || d > (int64_t(1) << 24) || d % 8 != 0) return 0;
    return packed_bytes(V, d, k);
}

int32_t sb_pack_weights(const void *W, int64_t V, int64_t d, int32_t k, void *W_packed,
                        size_t bytes, void *stream) {
    if (!W || !W_packed || !shape_ok(1, V, k) || d < 8 || d > (int64_t(1) << 24))
        return SB_ERR_INVALID_ARG;
    if (d % 8 != 0 || !aligned(W, 16) || !aligned(W_packed, 16)) return SB_ERR_ALIGNMENT;
    if (bytes < packed_bytes(V, d, k)) return SB_ERR_WORKSPACE_TOO_SMALL;
    DevInfo dev;
    if (int32_t e = current_device(&dev)) return e;
    if (launch_pack_weights(W, W_packed, V, d, k, dev.sms, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SB_ERR_CUDA;
    return SB_OK;
}

}  // extern "C"

namespace {

// The device address of host memory the device can read and write directly (pinned and
// mapped, as cudaHostAlloc / cudaHostRegister memory is under unified addressing); null
// for any other memory (pageable host memory, device memory, unknown pointers).
void *device_view(const void *host) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer leaves an error behind: clear it
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

// A validated call: kernel parameters and tensor maps, ready to enqueue.
struct Prepared {
    GemmParams p;
    CUtensorMap tmA, tmB;
    size_t smem;
    int sms;
    bool vm;
    CombineParams c;
};

// Validates a call and builds its launch state; enqueues nothing.
int32_t prepare(const void *H, const void *W, int64_t M, int64_t d, int64_t V, int32_t k,
                int32_t surface, float temperature, uint64_t seed, const sb_outputs *out,
                Prepared *pr) {
    const bool packed = (surface & SB_W_PACKED) != 0;
    surface &= ~SB_W_PACKED;
    if (!H || !W || !shape_ok(M, V, k) || d < 8 || d > (int64_t(1) << 24) ||
        surface < SB_TOKEN || surface > SB_TOPK_LOGPROB)
        return SB_ERR_INVALID_ARG;
    const bool gumbel = surface == SB_GUMBEL_TOKEN;
    const bool topk = surface == SB_TOPK_LOGPROB;
    if (gumbel && !(std::isfinite(temperature) && temperature > 0.f)) return SB_ERR_INVALID_ARG;
    if (int32_t e = check_outputs(out, surface, true)) return e;
    if (topk && (out->topk > V || k > kMaxTopKShards)) return SB_ERR_INVALID_ARG;
    if (d % 8 != 0 || !aligned(H, 16) || !aligned(W, 16)) return SB_ERR_ALIGNMENT;
    const int32_t T = tiles_per_shard(M, V, k);
    const int K = topk ? out->topk : 0;
    const WsLayout L = ws_layout(M, k, T, gumbel, K);
    if (out->workspace_bytes < L.total) return SB_ERR_WORKSPACE_TOO_SMALL;
    DevInfo dev;
    if (int32_t e = current_device(&dev)) return e;

    const bool vm = vocab_mode(M);
    const int flags = (gumbel ? kFlagGumbel : 0) | (surface == SB_FULL_LOGITS ? kFlagFull : 0) |
                      (out->target_ids ? kFlagTargets : 0) | (topk ? kFlagTopk : 0);
    const float inv_t = gumbel ? 1.0f / temperature : 1.0f;
    GemmParams &p = pr->p;
    p = GemmParams{};
    p.M = static_cast<int>(M);
    p.d = static_cast<int>(d);
    p.V = static_cast<int>(V);
    p.k = k;
    p.S = static_cast<int>(V / k);
    p.T = T;
    p.tv = vm ? kVocabTileV : kRowsTileN;
    p.Tt = static_cast<int>((V / k + p.tv - 1) / p.tv);
    p.nb = vm ? static_cast<int>((M + 15) / 16 * 16) : kRowsTileN;
    p.m_tiles = vm ? 1 : static_cast<int>((M + kTileA - 1) / kTileA);
    p.cluster = vm ? 1 : kRowsCluster;
    p.m_groups = (p.m_tiles + p.cluster - 1) / p.cluster;
    const int64_t tiles = static_cast<int64_t>(k) * p.Tt * p.m_groups;
    if (tiles >= (int64_t(1) << 31)) return SB_ERR_INVALID_ARG;
    p.num_tiles = static_cast<int>(tiles);
    // K blocks: 64 columns in vocab mode.  Rows mode: K blocks of two 64-wide atoms (half the
    // barrier waits and MMA commits per flop, 3 joint stages) when the rows span several CTA
    // pairs, so that each W tile is shared by several pairs and the tensor pipe sets the pace;
    // one atom (7 joint stages, deeper buffering of the W stream) for a single pair of M tiles.
    p.atoms = (vm || p.m_groups < 2) ? 1 : kMaxPairAtoms;
    p.joint = (!vm || p.nb >= 32) ? 1 : 0;
    const int64_t kb_cols = static_cast<int64_t>(p.atoms) * kBlockK;
    p.kblocks = static_cast<int>((d + kb_cols - 1) / kb_cols);
    if (!pick_stages(p.nb, vm, p.joint != 0, p.atoms, flags, K, &p.stages_a, &p.stages_b))
        return SB_ERR_UNSUPPORTED;
    p.flags = flags;
    p.topk = K;
    p.inv_t = inv_t;
    p.seed = seed;
    p.targets = out->target_ids;
    p.logits = out->logits_bf16;
    p.ws = ws_views(out->workspace, L, gumbel, K);
    p.timeout_ns = g_timeout_ns.load();
    p.debug_stall = g_debug_stall.load();

    // rows mode: each CTA of a cluster loads 256 / cluster rows of the shared W tile; with a
    // packed W every W box (128 rows, 64 columns) is one 16 KB block of the packed layout
    p.packed = packed ? 1 : 0;
    p.t128 = static_cast<int>(packed_t128(V, k));
    CUtensorMap *wmap = vm ? &pr->tmA : &pr->tmB;
    const bool ok =
        (vm ? make_map(&pr->tmB, H, M, d, p.nb) : make_map(&pr->tmA, H, M, d, kTileA)) &&
        (packed ? make_packed_map(wmap, W, V, d, k)
                : make_map(wmap, W, V, d, vm ? kTileA : kRowsTileN / p.cluster));
    if (!ok) return SB_ERR_CUDA;
    pr->smem = lmhead_smem_bytes(p.nb, p.stages_a, p.stages_b, vm, flags, K, p.atoms);
    pr->sms = dev.sms;
    pr->vm = vm;
    pr->c = combine_params(out, p.ws, M, k, T, flags, inv_t);
    return SB_OK;
}

// Enqueues a prepared call: the fused GEMM + record epilogue and, when `with_combine`, the
// record combine.  Each launch gets a new epoch.
int32_t launch(Prepared &pr, void *stream, bool with_combine) {
    pr.p.epoch = g_epoch.fetch_add(1) + 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (launch_lmhead(pr.vm, pr.tmA, pr.tmB, pr.p, pr.smem, pr.sms, st) != cudaSuccess)
        return SB_ERR_CUDA;
    if (!with_combine) return SB_OK;
    if (launch_combine(pr.c, st) != cudaSuccess) return SB_ERR_CUDA;
    return SB_OK;
}

int32_t enqueue(const void *H, const void *W, int64_t M, int64_t d, int64_t V, int32_t k,
                int32_t surface, float temperature, uint64_t seed, const sb_outputs *out,
                void *stream, bool with_combine) {
    Prepared pr;
    if (int32_t e = prepare(H, W, M, d, V, k, surface, temperature, seed, out, &pr)) return e;
    return launch(pr, stream, with_combine);
}

}  // namespace

extern "C" {

int32_t sb_lmhead_project(const void *H, const void *W, int64_t M, int64_t d, int64_t V,
                          int32_t k, int32_t surface, float temperature, uint64_t seed,
                          const sb_outputs *out, void *stream) {
    return enqueue(H, W, M, d, V, k, surface, temperature, seed, out, stream, true);
}

int32_t sb_lmhead_records(const void *H, const void *W, int64_t M, int64_t d, int64_t V,
                          int32_t k, int32_t surface, float temperature, uint64_t seed,
                          const sb_outputs *out, void *stream) {
    return enqueue(H, W, M, d, V, k, surface, temperature, seed, out, stream, false);
}

int32_t sb_lmhead_project_from_host(const void *H_host, void *H_dev, const void *W, int64_t M,
                                    int64_t d, int64_t V, int32_t k, int32_t surface,
                                    float temperature, uint64_t seed, const sb_outputs *out,
                                    int32_t *token_host, float *token_logprob_host,
                                    void *stream) {
    if (!H_host || !token_host) return SB_ERR_INVALID_ARG;
    Prepared pr;
    if (int32_t e = prepare(H_dev, W, M, d, V, k, surface, temperature, seed, out, &pr)) return e;
    if (token_logprob_host && !out->token_logprob) return SB_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t h_bytes = static_cast<size_t>(M) * d * 2;  // a multiple of 16 (d % 8 == 0)
    // Host buffers the device can address (pinned and mapped) are read and written by the
    // kernels themselves: no copy-engine operations, whose fixed cost is several
    // microseconds each.  Other host memory goes through cudaMemcpyAsync.
    const void *h_view = device_view(H_host);
    int32_t *tok_view = static_cast<int32_t *>(device_view(token_host));
    float *lp_view = token_logprob_host ? static_cast<float *>(device_view(token_logprob_host))
                                        : nullptr;
    const bool results_direct = tok_view && aligned(tok_view, 4) &&
                                (!token_logprob_host || (lp_view && aligned(lp_view, 4)));
    if (h_view && aligned(h_view, 16)) {
        if (launch_copy16(H_dev, h_view, h_bytes / 16, pr.sms, st) != cudaSuccess)
            return SB_ERR_CUDA;
    } else if (cudaMemcpyAsync(H_dev, H_host, h_bytes, cudaMemcpyHostToDevice, st) !=
               cudaSuccess) {
        return SB_ERR_CUDA;
    }
    if (results_direct) {
        pr.c.token_host = tok_view;
        pr.c.token_logprob_host = lp_view;
    }
    if (int32_t e = launch(pr, stream, true)) return e;
    if (results_direct) return SB_OK;
    // token and log-prob stored back to back on both sides: one copy
    const size_t n = static_cast<size_t>(M) * 4;
    const bool joined =
        token_logprob_host &&
        reinterpret_cast<const char *>(out->token_logprob) ==
            reinterpret_cast<const char *>(out->token) + n &&
        reinterpret_cast<const char *>(token_logprob_host) ==
            reinterpret_cast<const char *>(token_host) + n;
    if (cudaMemcpyAsync(token_host, out->token, joined ? 2 * n : n, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess)
        return SB_ERR_CUDA;
    if (token_logprob_host && !joined &&
        cudaMemcpyAsync(token_logprob_host, out->token_logprob, n, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess)
        return SB_ERR_CUDA;
    return SB_OK;
}

// A host-buffer decode step captured once into a CUDA graph: the copy kernel, the GEMM and
// the combine with the host stores, replayed by one graph launch per step.
struct sb_host_step {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

int32_t sb_host_step_create(const void *H_host, void *H_dev, const void *W, int64_t M,
                            int64_t d, int64_t V, int32_t k, int32_t surface,
                            float temperature, uint64_t seed, const sb_outputs *out,
                            int32_t *token_host, float *token_logprob_host,
                            sb_host_step **step) {
    if (!step) return SB_ERR_INVALID_ARG;
    *step = nullptr;
    if (!H_host || !token_host) return SB_ERR_INVALID_ARG;
    Prepared pr;
    if (int32_t e = prepare(H_dev, W, M, d, V, k, surface, temperature, seed, out, &pr)) return e;
    if (token_logprob_host && !out->token_logprob) return SB_ERR_INVALID_ARG;
    const void *h_view = device_view(H_host);
    int32_t *tok_view = static_cast<int32_t *>(device_view(token_host));
    float *lp_view = token_logprob_host ? static_cast<float *>(device_view(token_logprob_host))
                                        : nullptr;
    // only device-addressable host buffers: a graph replays kernels, not pageable copies
    if (!h_view || !aligned(h_view, 16) || !tok_view || !aligned(tok_view, 4) ||
        (token_logprob_host && (!lp_view || !aligned(lp_view, 4))))
        return SB_ERR_UNSUPPORTED;
    pr.c.token_host = tok_view;
    pr.c.token_logprob_host = lp_view;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return SB_ERR_CUDA;
    cudaGraph_t graph = nullptr;
    bool ok = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (ok) {
        const size_t h_bytes = static_cast<size_t>(M) * d * 2;
        const bool enq = launch_copy16(H_dev, h_view, h_bytes / 16, pr.sms, cs) == cudaSuccess &&
                         launch(pr, cs, true) == SB_OK;
        ok = cudaStreamEndCapture(cs, &graph) == cudaSuccess && enq && graph;
    }
    cudaStreamDestroy(cs);
    cudaGraphExec_t exec = nullptr;
    if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
    if (!ok) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return SB_ERR_CUDA;
    }
    *step = new sb_host_step{graph, exec};
    return SB_OK;
}

int32_t sb_host_step_launch(sb_host_step *step, void *stream) {
    if (!step) return SB_ERR_INVALID_ARG;
    return cudaGraphLaunch(step->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SB_OK
               : SB_ERR_CUDA;
}

void sb_host_step_destroy(sb_host_step *step) {
    if (!step) return;
    cudaGraphExecDestroy(step->exec);
    cudaGraphDestroy(step->graph);
    delete step;
}

int32_t sb_combine_shard_records(const void *workspace, int64_t M, int32_t k,
                                 int32_t tiles_per_shard_, int32_t surface, float temperature,
                                 const sb_outputs *out, void *stream) {
    if (!workspace || M < 1 || M > (int64_t(1) << 30) || k < 1 || k > kMaxShards ||
        tiles_per_shard_ < 1 ||
        surface < SB_TOKEN || surface > SB_TOPK_LOGPROB)
        return SB_ERR_INVALID_ARG;
    const bool gumbel = surface == SB_GUMBEL_TOKEN;
    const bool topk = surface == SB_TOPK_LOGPROB;
    if (topk && k > kMaxTopKShards) return SB_ERR_INVALID_ARG;
    if (gumbel && !(std::isfinite(temperature) && temperature > 0.f)) return SB_ERR_INVALID_ARG;
    if (int32_t e = check_outputs(out, surface == SB_FULL_LOGITS ? SB_TOKEN : surface, true))
        return e;
    if (out->workspace != workspace) return SB_ERR_INVALID_ARG;
    const int K = topk ? out->topk : 0;
    const WsLayout L = ws_layout(M, k, tiles_per_shard_, gumbel, K);
    if (out->workspace_bytes < L.total) return SB_ERR_WORKSPACE_TOO_SMALL;
    DevInfo dev;
    if (int32_t e = current_device(&dev)) return e;
    const int flags = (gumbel ? kFlagGumbel : 0) | (out->target_ids ? kFlagTargets : 0) |
                      (topk ? kFlagTopk : 0);
    const Workspace w = ws_views(const_cast<void *>(workspace), L, gumbel, K);
    const CombineParams c = combine_params(out, w, M, k, tiles_per_shard_, flags,
                                           gumbel ? 1.0f / temperature : 1.0f);
    if (launch_combine(c, static_cast<cudaStream_t>(stream)) != cudaSuccess) return SB_ERR_CUDA;
    return SB_OK;
}

size_t sb_payload_bytes(int64_t M, int32_t k, int32_t surface) {
    if (M < 1 || M > (int64_t(1) << 30) || k < 1 || k > kMaxShards) return 0;
    if (surface != SB_TOKEN && surface != SB_TOKEN_LOGPROB && surface != SB_FULL_LOGITS &&
        surface != SB_GUMBEL_TOKEN)
        return 0;
    return static_cast<size_t>(M) * k * (surface == SB_GUMBEL_TOKEN ? 24 : 12);
}

int32_t sb_pack_shard_records(const void *workspace, int64_t M, int32_t k,
                              int32_t tiles_per_shard_, int32_t surface, int64_t col_offset,
                              void *payload, void *stream) {
    const size_t pb = sb_payload_bytes(M, k, surface);
    if (!workspace || !payload || pb == 0 || tiles_per_shard_ < 1 || col_offset < 0 ||
        col_offset >= (int64_t(1) << 31))
        return SB_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(payload, 4)) return SB_ERR_ALIGNMENT;
    DevInfo dev;
    if (int32_t e = current_device(&dev)) return e;
    const bool gumbel = surface == SB_GUMBEL_TOKEN;
    const WsLayout L = ws_layout(M, k, tiles_per_shard_, gumbel);
    const Workspace w = ws_views(const_cast<void *>(workspace), L, gumbel);
    if (launch_pack(w, static_cast<int>(M), k, tiles_per_shard_, gumbel, col_offset, payload,
                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SB_ERR_CUDA;
    return SB_OK;
}

int32_t sb_merge_shard_payload(const void *payload, int64_t M, int32_t k, int32_t surface,
                               float temperature, const sb_outputs *out, void *stream) {
    if (!payload || sb_payload_bytes(M, k, surface) == 0 || !out || !out->token)
        return SB_ERR_INVALID_ARG;
    const bool gumbel = surface == SB_GUMBEL_TOKEN;
    if (gumbel && !(std::isfinite(temperature) && temperature > 0.f)) return SB_ERR_INVALID_ARG;
    if ((surface == SB_TOKEN_LOGPROB || gumbel) && !out->token_logprob) return SB_ERR_INVALID_ARG;
    if (!aligned(payload, 4) || !aligned(out->token, 4) || !aligned(out->token_logprob, 4) ||
        !aligned(out->lse, 4))
        return SB_ERR_ALIGNMENT;
    DevInfo dev;
    if (int32_t e = current_device(&dev)) return e;
    CombineParams c{};
    c.M = static_cast<int>(M);
    c.k = k;
    c.flags = gumbel ? kFlagGumbel : 0;
    c.inv_t = gumbel ? 1.0f / temperature : 1.0f;
    c.token = out->token;
    c.token_logprob = out->token_logprob;
    c.lse = out->lse;
    if (launch_merge_payload(c, payload, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SB_ERR_CUDA;
    return SB_OK;
}

int32_t sb_select_source_projection(double bytes_ref, double bytes_proj, double frames_ref,
                                    double frames_proj, double link_bytes_per_s,
                                    double frame_startup_s, double local_proj_s,
                                    double local_ref_s, double *margin_s) {
    const double in[] = {bytes_ref, bytes_proj, frames_ref, frames_proj, frame_startup_s};
    for (double v : in)
        if (!(v >= 0.0) || !std::isfinite(v)) return -1;
    if (!(link_bytes_per_s > 0.0) || !std::isfinite(link_bytes_per_s) ||
        !std::isfinite(local_proj_s) || !std::isfinite(local_ref_s))
        return -1;
    const double saved = (bytes_ref - bytes_proj) / link_bytes_per_s +
                         frame_startup_s * (frames_ref - frames_proj);
    const double added = local_proj_s - local_ref_s;
    if (margin_s) *margin_s = saved - added;
    return saved > added ? 1 : 0;
}

int32_t sb_last_device_status(const sb_outputs *out) {
    if (!out || !out->workspace || out->workspace_bytes < 16) return SB_ERR_INVALID_ARG;
    uint64_t hdr[2] = {0, 0};
    if (cudaMemcpy(hdr, out->workspace, sizeof hdr, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SB_ERR_CUDA;
    const uint32_t epoch = static_cast<uint32_t>(hdr[0] & 0xFFFFFFFFu);
    const uint64_t st = hdr[1];
    const uint32_t code = static_cast<uint32_t>(st);
    if (static_cast<uint32_t>(st >> 32) == epoch &&
        (code == SB_ERR_DEVICE_TIMEOUT || code == SB_ERR_INVALID_ARG))
        return static_cast<int32_t>(code);
    return SB_OK;
}

const char *sb_status_string(int32_t status) {
    switch (status) {
    case SB_OK: return "ok";
    case SB_ERR_INVALID_ARG: return "invalid argument";
    case SB_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case SB_ERR_ALIGNMENT: return "misaligned pointer or d not a multiple of 8";
    case SB_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SB_ERR_CUDA: return "CUDA runtime or driver error";
    case SB_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int32_t sb_device_info(int32_t *num_sms, int32_t *cc) {
    DevInfo dev;
    const int32_t e = current_device(&dev);
    if (e == SB_ERR_CUDA) return -1;
    if (num_sms) *num_sms = dev.sms;
    if (cc) *cc = dev.cc;
    return 0;
}

int32_t sb_debug_configure(int32_t stall_epilogue, uint64_t wait_limit_ns) {
    if (wait_limit_ns == 0) return SB_ERR_INVALID_ARG;
    g_debug_stall.store(stall_epilogue ? 1 : 0);
    g_timeout_ns.store(wait_limit_ns);
    return SB_OK;
}

}  // extern "C"
