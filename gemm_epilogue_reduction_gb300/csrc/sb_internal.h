// sb_internal.h -- types shared by the libsb host code and its kernels (not part of the ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sb {

constexpr int kBlockK = 64;          // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kTileA = 128;          // rows of the MMA A operand (the UMMA M)
constexpr int kRowsTileN = 256;      // vocabulary columns per tile when H rows are the A operand
constexpr int kVocabTileV = 128;     // vocabulary columns per tile when W rows are the A operand
constexpr int kRecordCols = 128;     // vocabulary columns covered by one projection record
#ifndef SB_MAX_VOCAB_MODE_ROWS
#define SB_MAX_VOCAB_MODE_ROWS 128
#endif
constexpr int kMaxVocabModeRows = SB_MAX_VOCAB_MODE_ROWS;  // largest M with W as the A operand
constexpr int kMaxStages = 16;
constexpr int kMaxShards = 1024;  // largest k (the combine keeps k shard records in smem)
// rows mode: a cluster of two CTAs (consecutive M tiles) shares each W tile; one
// cta_group::2 MMA per pair, each CTA staging its own half of the W tile
constexpr int kRowsCluster = 2;
// rows mode: each joint pipeline stage holds 1 or kMaxPairAtoms 64-wide K slices ("atoms")
// of both operands; with 2 (K block 128) the MMA warp waits once and commits once per
// 8 MMAs, with 1 more stages fit in shared memory
constexpr int kMaxPairAtoms = 2;
// rows mode: the L2 policy of W.  A W tile is read by the m_groups CTA pairs of its column
// range at about the same time.  Up to this many pairs W is loaded evict-first (no pair reads
// it again, and the space keeps H, loaded evict-last); beyond it W is loaded evict-last like
// H, as the tile must stay in L2 until every pair has read it (measured: 1 to 4 pairs 1-6 %
// faster evict-first than evict-normal, 8 and 16 pairs 2-5 % slower; at 8 and 16 pairs
// evict-last 1-3 % faster than evict-normal)
constexpr int kWEvictFirstGroups = 4;

constexpr int kEpiWarps = 8;         // two epilogue warps per TMEM lane quadrant
constexpr int kFirstEpiWarp = 3;     // warps 0 and 2 load, warp 1 issues MMAs + owns TMEM
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr size_t kSmemLimit = 232448;  // 227 KB dynamic shared memory per CTA

constexpr int kMaxTopK = 16;         // largest K of the top-K log-prob surface
constexpr int kMaxTopKShards = 128;  // largest k with the top-K surface (combine smem)

// Surface flags the kernels specialise on.
enum : int { kFlagGumbel = 1, kFlagFull = 2, kFlagTargets = 4, kFlagTopk = 8 };
// Epilogue variants (one per surface family).
// The top-K family has one variant per list length (rows mode keeps a sorted list of the
// smallest of 4, 8, 16 entries that holds K per thread; vocab mode uses kEpiTopk for any K).
enum : int { kEpiPlain = 0, kEpiFull = 1, kEpiGumbel = 2, kEpiTopk = 3, kEpiTopk8 = 4,
             kEpiTopk4 = 5 };

struct Workspace {       // device views into the caller's workspace
    uint32_t *epoch;     // header word 0
    unsigned long long *status;  // header word 1: (epoch << 32) | code
    float *m;
    int32_t *idx;
    float *s;
    float *gk;
    int32_t *gi;
    float *gz;
    float *tkv;          // [n][topk] top-K values per record (top-K surface)
    int32_t *tki;        // [n][topk] their columns
    float *tz;
};

struct GemmParams {
    int M, d, V, k, S, T;  // T = records per shard (128-column record tiles)
    int Tt;                // GEMM tiles per shard
    int tv;                // vocabulary columns per GEMM tile
    int nb;                // rows of the B operand per tile (UMMA N)
    int m_tiles;           // tiles along M (1 when W rows are the A operand)
    int m_groups;          // groups of `cluster` consecutive M tiles (rows mode)
    int cluster;           // CTAs per cluster sharing each W tile (1 or 2)
    int num_tiles;
    int kblocks;
    int stages_a;          // ring depth of the UMMA A operand (16 KB stages)
    int stages_b;          // ring depth of the UMMA B operand (nb * 128 B stages)
    int atoms;             // rows mode: 64-wide K atoms per joint stage (1 or 2)
    int joint;             // vocab mode: one joint ring (1) or one ring per operand (0)
    int packed;            // W in the packed layout (tile-contiguous 16 KB boxes, 4-D map)
    int t128;              // packed layout: 128-row tiles per shard
    int flags;
    int topk;              // K of the top-K surface (0 otherwise)
    float inv_t;
    unsigned long long seed;
    const int32_t *targets;
    uint16_t *logits;
    Workspace ws;
    uint32_t epoch;
    unsigned long long timeout_ns;
    int debug_stall;
};

struct CombineParams {
    int M, k, T;
    int flags;
    int topk;
    int32_t *topk_ids;
    float *topk_logprob;
    float inv_t;
    Workspace ws;
    int32_t *token;
    float *token_logprob;
    float *lse;
    float *target_logprob;
    // optional second copies of token / token_logprob in host memory the device can address
    // (pinned, mapped): the host-buffer entry point's results, written without a copy
    int32_t *token_host;
    float *token_logprob_host;
};

// Launchers (lmhead.cu, combine.cu).  Return cudaSuccess or the launch error.
cudaError_t launch_lmhead(bool vocab_mode, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const GemmParams &p, size_t smem, int num_sms, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
// The packed copy of W [V, d] for k lane shards (layout in sb.h, sb_pack_weights).
cudaError_t launch_pack_weights(const void *W, void *P, long long V, long long d, int k,
                                int num_sms, cudaStream_t stream);
cudaError_t launch_pack(const Workspace &ws, int M, int k, int T, bool gumbel,
                        long long col_offset, void *payload, cudaStream_t stream);
cudaError_t launch_merge_payload(const CombineParams &c, const void *payload,
                                 cudaStream_t stream);
// Copies n16 16-byte words from src (host memory the device can address) to dst (device),
// as a programmatic dependent launch that writes dst only after the previous kernel ends.
cudaError_t launch_copy16(void *dst, const void *src, size_t n16, int num_sms,
                          cudaStream_t stream);

size_t lmhead_smem_bytes(int nb, int stages_a, int stages_b, bool vocab_mode, int flags,
                         int topk, int atoms);

// Host helpers shared by the entry points (sb_api.cu).
bool encode_bf16_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols,
                     int box_rows);
int32_t device_sms_cc(int *sms, int *cc);  // SB_OK, SB_ERR_CUDA or SB_ERR_UNSUPPORTED
uint32_t next_epoch();
unsigned long long wait_limit_ns();

}  // namespace sb
