/*
 * sb.h -- C ABI of libsb: the LM-head contraction logits = H·Wᵀ over a vocabulary split
 * into k contiguous lane shards, fused on one GPU (sm_103a) with the consumer-surface
 * projection, so that only the surface the consumer asked for leaves the kernel.
 *
 * Source of the operation -- "SemBridge: Compiling Consumer Observations into
 * Cross-Stack Communication Plans" (Chen, Zhu, Lin):
 *   - Section 5.2 (Data, Result, and Control Paths): the tail output head materialises
 *     full logits; a complete-logits or log-probability request slices them by TP lane
 *     and rebuilds the full value; a token-only request applies the deterministic
 *     sampler to the same tensor and sends int32 IDs.
 *   - Section 2.2 (Consumer Surfaces and Delivery Obligations): the consumer surfaces are
 *     complete logits, log-probabilities, token IDs or another registered projection.
 *   - Section 3.1 (Boundary Contract): the registered projection operator names its
 *     input/output types and deterministic tie-breaking (here: the lowest global
 *     vocabulary index wins a tie).
 *   - Figure 1: full-logit transfer and source projection expose the same token; they
 *     differ only in where argmax runs.  Here argmax runs inside the GEMM epilogue.
 *   - Section 5.2 also notes the transport reserves no persistent device-buffer pool;
 *     likewise this library allocates no device memory: the caller owns every buffer.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must point to device memory of the current CUDA device
 *     and be 16-byte aligned; sizes are element counts unless named *_bytes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     All device work is enqueued asynchronously on it; nothing synchronises.
 *   - The return value is an sb_status.  It covers argument validation and launch
 *     errors only; when it is not SB_OK nothing was enqueued.  Errors found on the
 *     device (a bounded wait that ran out) are recorded in the workspace status word
 *     and read with sb_last_device_status() after the caller synchronises.
 *   - There is no CPU fallback: a device that is not sm_103 returns SB_ERR_UNSUPPORTED.
 *   - Calls that share a workspace must not overlap on the GPU (they would race on it).
 *   - The calls enqueue kernels only (no host synchronisation), so they can be captured in
 *     a CUDA graph; arguments are checked and tensor maps encoded at capture time.  Every
 *     replay then carries the captured call's launch epoch, so after replays
 *     sb_last_device_status reports the worst device status since the capture.
 */
#ifndef SB_H
#define SB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Consumer surface (Section 2.2).  Every surface produces the token; the surface
 * decides which other outputs are mandatory and whether logits are written. */
typedef enum sb_surface {
    SB_TOKEN = 0,        /* deterministic argmax token (int32, lowest index on ties)      */
    SB_TOKEN_LOGPROB = 1,/* token + its natural-log log-probability over the full vocab   */
    SB_FULL_LOGITS = 2,  /* token + bf16 logits [M, V] in shard-to-full (global) layout    */
    SB_GUMBEL_TOKEN = 3, /* counter-based Gumbel-max sample from softmax(z / T) + log-prob */
    SB_TOPK_LOGPROB = 4  /* token + the K most likely tokens and their log-probabilities   */
} sb_surface;

/* Largest K of the SB_TOPK_LOGPROB surface. */
#define SB_MAX_TOPK 16

/* Layout flag OR'ed into the `surface` argument of the calls that read W (sb_lmhead_project,
 * sb_lmhead_records, sb_lmhead_project_from_host, sb_host_step_create,
 * sb_lmhead_project_static_scratch): W points to the packed copy written by
 * sb_pack_weights for the same V, d and k instead of the row-major [V, d] matrix.  The
 * results are bit for bit those of the row-major call (the same operands reach the same
 * MMAs); only the memory layout of W, and so how fast it streams, differs.
 * sb_workspace_bytes ignores the flag; the other calls reject it. */
#define SB_W_PACKED 0x100

typedef enum sb_status {
    SB_OK = 0,
    SB_ERR_INVALID_ARG = 1,          /* a size, enum, pointer or temperature is out of range */
    SB_ERR_UNSUPPORTED = 2,          /* the current device is not an sm_103 GPU               */
    SB_ERR_ALIGNMENT = 3,            /* a pointer is not 16-byte aligned, or d % 8 != 0       */
    SB_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace_bytes < sb_workspace_bytes(...)             */
    SB_ERR_CUDA = 5,                 /* a CUDA runtime or driver call failed                  */
    SB_ERR_DEVICE_TIMEOUT = 6        /* device side: a bounded wait gave up (after sync)      */
} sb_status;

/*
 * Output buffers of one projection call.  All pointers are device pointers owned by the
 * caller; NULL means "not requested".  Every surface fills every non-NULL output.
 *   token           int32 [M]      required for every surface.
 *   token_logprob   float [M]      log p(token); required for SB_TOKEN_LOGPROB and
 *                                  SB_GUMBEL_TOKEN.  For SB_GUMBEL_TOKEN the distribution
 *                                  is softmax(z / T), the one sampled from.
 *   lse             float [M]      natural-log logsumexp of z (of z / T for SB_GUMBEL_TOKEN).
 *   logits_bf16     uint16 [M*V]   bf16 bit patterns of z, row-major [M][V], column = the
 *                                  global vocabulary index (lane shard s holds columns
 *                                  [s*V/k, (s+1)*V/k)); required iff SB_FULL_LOGITS and
 *                                  written only then.
 *   target_ids      int32 [M]      optional scoring targets, each in [0, V).  Values out of
 *                                  range are found on the device: sb_last_device_status
 *                                  then reports SB_ERR_INVALID_ARG and the outputs are
 *                                  undefined.
 *   target_logprob  float [M]      log p(target_ids[r]); required iff target_ids != NULL.
 *   workspace       bytes          scratch of at least sb_workspace_bytes(M, V, k, surface)
 *                                  bytes, 256-byte aligned; holds the per-tile records, the
 *                                  target logits and the device status word.  Its contents
 *                                  need no initialisation.
 *   topk_ids        int32 [M*K]    SB_TOPK_LOGPROB: per row the K columns with the largest
 *                                  logits, largest first, equal logits by ascending column.
 *   topk_logprob    float [M*K]    SB_TOPK_LOGPROB: their log-probabilities z_j - lse.
 *   topk            K              SB_TOPK_LOGPROB: 1 <= K <= min(SB_MAX_TOPK, V); ignored by
 *                                  the other surfaces (as are the two arrays above).
 */
typedef struct sb_outputs {
    int32_t *token;
    float *token_logprob;
    float *lse;
    uint16_t *logits_bf16;
    const int32_t *target_ids;
    float *target_logprob;
    void *workspace;
    size_t workspace_bytes;
    int32_t *topk_ids;
    float *topk_logprob;
    int32_t topk;
} sb_outputs;

/*
 * Workspace layout (byte offsets from `workspace`; n = M * k * T with T =
 * sb_tiles_per_shard(M, V, k); each array starts on a 256-byte boundary, in this order):
 *   [0, 256)      header: uint32 epoch of the last launch, uint32 reserved,
 *                 uint64 status word = (epoch << 32) | sb_status of that launch
 *   float   m[n]     per-tile record: max of y over the tile's columns
 *   int32   idx[n]   lowest global column attaining m
 *   float   s[n]     sum over the tile of exp(y - m)
 *   float   gkey[n]  SB_GUMBEL_TOKEN only: max of y + g over the tile
 *   int32   gidx[n]  SB_GUMBEL_TOKEN only: lowest column attaining gkey
 *   float   gz[n]    SB_GUMBEL_TOKEN only: z at gidx
 *   float   tkv[n][K] SB_TOPK_LOGPROB only: the tile's K largest logits, largest first
 *   int32   tki[n][K] SB_TOPK_LOGPROB only: their columns (INT32_MAX marks an empty slot)
 *   float   tz[M]    z at target_ids[r] (written only when targets are given)
 * Record (r, s, t) sits at index (r * k + s) * T + t and covers the global columns
 * [s*S + 128t, min(s*S + 128(t+1), (s+1)*S)) with S = V/k and T = ceil(S / 128).  y is z,
 * or z * (1/T) for SB_GUMBEL_TOKEN with 1/T rounded to fp32 on the host; g is the Gumbel
 * noise of sb_lmhead_project.
 */

/* Bytes of workspace one call needs (for SB_TOPK_LOGPROB: with K = SB_MAX_TOPK, enough for
 * every K); 0 if the arguments are invalid. */
size_t sb_workspace_bytes(int64_t M, int64_t V, int32_t k, int32_t surface);

/*
 * The packed layout of W for the calls with SB_W_PACKED: every (128-row tile, 64-column K
 * block) box the kernels read is one contiguous 16 KB block, so each box is one linear
 * stream of HBM reads instead of 128 rows of 128 bytes, 2d bytes apart.  With S = V/k,
 * T128 = ceil(S / 128) tiles per shard and KB = ceil(d / 64) K blocks, element (r, c) of W
 * (row r of shard s = r / S, i = (r - s*S) mod 128 in tile t = (r - s*S) / 128; column c in
 * K block kb = c / 64 at j = c mod 64) is bf16 number
 *     (((s * T128 + t) * KB + kb) * 128 + i) * 64 + j
 * of the packed buffer; the rows past a shard's end in its last tile and the columns past d
 * in the last K block are zero.  A weight is packed once (it is a model parameter) and then
 * read by every call.
 */
/* Bytes of the packed copy of a [V, d] W for k lane shards: k * T128 * KB * 16384; 0 if the
 * arguments are invalid (the same shape rules as sb_lmhead_project, d % 8 == 0). */
size_t sb_packed_weight_bytes(int64_t V, int64_t d, int32_t k);
/* Writes the packed copy of the row-major W [V, d] (device, bf16, 16-byte aligned) into
 * W_packed (device, 16-byte aligned, `bytes` >= sb_packed_weight_bytes), enqueued on
 * `stream`.  SB_ERR_WORKSPACE_TOO_SMALL if `bytes` is short, SB_ERR_ALIGNMENT for a
 * misaligned pointer or d % 8 != 0. */
int32_t sb_pack_weights(const void *W, int64_t V, int64_t d, int32_t k, void *W_packed,
                        size_t bytes, void *stream);

/* Records per (row, lane shard): T = ceil((V / k) / 128), one per 128 vocabulary columns;
 * -1 if the arguments are invalid.  (M is accepted for symmetry and does not change T.) */
int32_t sb_tiles_per_shard(int64_t M, int64_t V, int32_t k);

/*
 * One projection call: logits z = H·Wᵀ (fp32 accumulation on the tensor cores, no bias,
 * scale or soft-cap), projected per Section 5.2 onto `surface`, in two kernels enqueued on
 * `stream` -- the fused GEMM + record epilogue, then the record combine
 * (sb_combine_shard_records) -- with no host synchronisation.
 *   H          device bf16 [M, d] row-major (K-major), 16-byte aligned.
 *   W          device bf16 [V, d] row-major (the output-head weight), 16-byte aligned; or,
 *              with SB_W_PACKED in `surface`, its packed copy (sb_pack_weights, same k).
 *   M, d, V    M >= 1, d >= 8 with d % 8 == 0, V >= 1.
 *   k          number of contiguous lane shards, 1 <= k <= 1024 and V % k == 0.
 *   surface    an sb_surface, optionally OR'ed with SB_W_PACKED.
 *   temperature  SB_GUMBEL_TOKEN: finite and > 0 (the key is z * (1/T) + g); ignored
 *              otherwise.
 *   seed       SB_GUMBEL_TOKEN: the SplitMix64 stream seed.  Column j of row r draws the
 *              output at stream index n = r*V + j, i.e. the SplitMix64 finaliser of
 *              seed + (n + 1) * 0x9E3779B97F4A7C15; u = (x >> 40) * 2^-24 and
 *              g = -log(-log u) in fp32 to within 2e-6 absolute (u = 0 gives g = -inf).
 *              Ignored otherwise.
 *   out        outputs and workspace (see sb_outputs); read on the host during the call.
 * The GEMM is a programmatic dependent launch that starts loading W before the preceding
 * kernel in the stream has finished, so W must not be written by a kernel that can still be
 * running then (one that signals its dependents early); H, the targets and the workspace are
 * read only after that kernel has finished.
 * Returns SB_OK, or an error with nothing enqueued.
 */
int32_t sb_lmhead_project(const void *H, const void *W, int64_t M, int64_t d, int64_t V,
                          int32_t k, int32_t surface, float temperature, uint64_t seed,
                          const sb_outputs *out, void *stream);

/*
 * The first kernel of sb_lmhead_project alone: the fused GEMM + record epilogue, which
 * writes the per-tile records (and the target logits) into out->workspace and, for
 * SB_FULL_LOGITS, the bf16 logits; token, log-prob and lse outputs are left unwritten.
 * Same arguments, validation and return values as sb_lmhead_project.  It is the step a
 * vocabulary-sharded caller runs before exchanging records (Section 5.2: each TP lane
 * projects its own shard) and then finishing with sb_combine_shard_records.
 */
int32_t sb_lmhead_records(const void *H, const void *W, int64_t M, int64_t d, int64_t V,
                          int32_t k, int32_t surface, float temperature, uint64_t seed,
                          const sb_outputs *out, void *stream);

/*
 * sb_lmhead_project for a caller whose hidden states are in host memory and who wants the
 * token surface back in host memory ("SemBridge", Section 5.2: the consumer observes the
 * projected surface, never the logits).  Enqueues on stream, in order: H_host into H_dev,
 * the projection of sb_lmhead_project on H_dev, and the token (and, when
 * token_logprob_host is not NULL, the chosen log-probability) into the host buffers; the
 * device outputs in out are written as well.
 * Host buffers the device can address (pinned memory from cudaHostAlloc or
 * cudaHostRegister, mapped under unified addressing) are moved by the kernels themselves:
 * a copy kernel reads H_host and the combine writes the host results directly, with no
 * copy-engine operations.  Other host memory (pageable) is moved with cudaMemcpyAsync
 * (synchronous with respect to the host for pageable memory).
 *   H_host              host bf16 [M, d].
 *   H_dev               device staging buffer of M * d bf16, 16-byte aligned; overwritten
 *                       once the previous kernel in the stream has finished.
 *   out                 device outputs and workspace as for sb_lmhead_project.
 *   token_host          host int32 [M] (required); token_logprob_host host float [M] or NULL
 *                       (then out->token_logprob may be NULL).
 * On the copy path, when out->token_logprob directly follows out->token (M int32) and
 * token_logprob_host directly follows token_host, both come back in one copy.  The caller
 * synchronises stream before reading the host outputs.  Every argument is checked before
 * anything is enqueued; returns an sb_status.
 */
int32_t sb_lmhead_project_from_host(const void *H_host, void *H_dev, const void *W, int64_t M,
                                    int64_t d, int64_t V, int32_t k, int32_t surface,
                                    float temperature, uint64_t seed, const sb_outputs *out,
                                    int32_t *token_host, float *token_logprob_host,
                                    void *stream);

/*
 * The host-buffer call of a serving loop, captured once: sb_host_step_create checks the
 * arguments as sb_lmhead_project_from_host does and records that call (the copy kernel
 * reading H_host, the projection, the combine storing into the host buffers) into a CUDA
 * graph; sb_host_step_launch enqueues one replay on `stream` (one graph launch, about a
 * quarter of the host-side time of the plain call); sb_host_step_destroy releases it.
 * Every buffer is bound at creation: each replay reads the current contents of H_host and
 * overwrites token_host / token_logprob_host and the device outputs of `out`.
 *   H_host, token_host, token_logprob_host  host memory the device can address (pinned:
 *              cudaHostAlloc / cudaHostRegister under unified addressing); other host memory
 *              gives SB_ERR_UNSUPPORTED (use sb_lmhead_project_from_host).
 *   step       receives the handle (NULL on any error).
 * Replays reuse the launch epoch of the creation, so sb_last_device_status reports the worst
 * device status since then.  Returns an sb_status; creation enqueues nothing on any stream.
 */
typedef struct sb_host_step sb_host_step;
int32_t sb_host_step_create(const void *H_host, void *H_dev, const void *W, int64_t M,
                            int64_t d, int64_t V, int32_t k, int32_t surface,
                            float temperature, uint64_t seed, const sb_outputs *out,
                            int32_t *token_host, float *token_logprob_host,
                            sb_host_step **step);
int32_t sb_host_step_launch(sb_host_step *step, void *stream);
void sb_host_step_destroy(sb_host_step *step);

/*
 * The record combine alone (the second kernel of sb_lmhead_project): reads the per-tile
 * records of `workspace` (layout above; tiles_per_shard = T) and writes token,
 * token_logprob, lse and target_logprob of `out` (those that are non-NULL).  Per row it
 * merges the T records of each shard in a fixed tree (shard-local completion), then the k
 * shard results in ascending shard order (the cross-shard merge that replaces "AllGather
 * the logits, then argmax" of Section 5.2).  The merge of two records keeps the larger
 * max, the lower index on an equal max, and rescales the exp-sums to the new max; the
 * fixed order makes the output bits a function of the record bits alone.
 *   temperature  as for sb_lmhead_project (used by SB_GUMBEL_TOKEN and the target
 *              log-prob only).
 *   out->logits_bf16 is ignored; out->workspace must equal `workspace`.
 */
int32_t sb_combine_shard_records(const void *workspace, int64_t M, int32_t k,
                                 int32_t tiles_per_shard, int32_t surface, float temperature,
                                 const sb_outputs *out, void *stream);

/*
 * sb_lmhead_project without a caller-supplied workspace (the SemBridge paper has no
 * counterpart; this entry point exists for callers that cannot allocate device memory).
 * Some callers cannot call cudaMalloc: a plug-in inside a host engine that owns the whole
 * device-memory pool, code on a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not allowed, or a foreign-function caller that links only this
 * library.  This call takes its scratch from an 8 MiB array compiled into the library
 * (every GPU that loads libsb holds it until the process exits) and allocates nothing.
 *   Arguments, outputs and return values are those of sb_lmhead_project, except that
 *   out->workspace and out->workspace_bytes are ignored.  A problem whose
 *   sb_workspace_bytes(M, V, k, surface) exceeds 8 MiB (8388608 bytes) is rejected with
 *   SB_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   The first call on each device looks up the array's device address (with that device
 *   current); make that first call before any stream capture.
 *   Every call on a device shares the one array and leaves its records there; nothing in
 *   it needs clearing between calls, but calls that overlap on the GPU (different streams,
 *   or host threads without ordering) race on it and give undefined results.
 *   The device status word also lives in the array, out of the caller's reach: read it with
 *   sb_static_scratch_last_status() (not sb_last_device_status) after synchronising.  Both
 *   errors found on the device land there: a bounded wait that ran out
 *   (SB_ERR_DEVICE_TIMEOUT) and a scoring target outside [0, V) (SB_ERR_INVALID_ARG).
 */
int32_t sb_lmhead_project_static_scratch(const void *H, const void *W, int64_t M, int64_t d,
                                         int64_t V, int32_t k, int32_t surface,
                                         float temperature, uint64_t seed,
                                         const sb_outputs *out, void *stream);

/*
 * The device status of the last sb_lmhead_project_static_scratch call on the current device
 * (no paper counterpart): SB_OK, SB_ERR_DEVICE_TIMEOUT or SB_ERR_INVALID_ARG, as
 * sb_last_device_status reports for a caller's workspace; SB_ERR_CUDA if the array cannot be
 * read.  Synchronises with the device (a blocking device-to-host copy of 16 bytes into host
 * stack memory; allocates nothing).  Call it after the static-scratch call has completed and
 * before the next one is enqueued.
 */
int32_t sb_static_scratch_last_status(void);

/* Test hook: the two functions of the record merge, as the combine kernels evaluate them,
 * on count entries of device arrays (enqueued on stream): op 0 gives y[i] = e^x[i] for
 * x <= 0 (the hardware base-2 exponential of x * log2(e), the product rounded to fp32);
 * op 1 gives y[i] = ln x[i].  With these two, a host restatement of the merge order in
 * fp32 reproduces sb_combine_shard_records bit for bit. */
int32_t sb_debug_combine_math(int32_t op, const float *x, float *y, int64_t count,
                              void *stream);

/* Test hook: g[i] = the Gumbel noise the projection kernels derive from the 24-bit
 * uniform bits[i] & 0xFFFFFF (u = bits * 2^-24), for count entries of device arrays,
 * enqueued on stream. */
int32_t sb_debug_gumbel_from_bits(const uint32_t *bits, float *g, int64_t count, void *stream);

/*
 * Shard payloads: what each vocabulary lane would send to the others instead of its logit
 * slice (Figure 1 and Section 5.2: full-logit transfer ships V logit elements in k frames,
 * source projection ships the per-lane projection).  A lane's payload is its shard-local
 * completion: per row one record (m, idx, s) = (max logit, lowest global column attaining
 * it, sum of exp(z - m)) -- 12 bytes; the Gumbel surface adds (gkey, gidx, gz) -- 24 bytes.
 * The top-K surface has no payload form.
 * Layout: lane-major, record (lane s, row r) at byte (s * M + r) * record_bytes; fields are
 * float32 / int32 in that order.  Merging the k payloads in ascending lane order gives the
 * same bits as sb_combine_shard_records on the same records.
 */

/* k * M * record_bytes for the surfaces above; 0 for invalid arguments or SB_TOPK_LOGPROB. */
size_t sb_payload_bytes(int64_t M, int32_t k, int32_t surface);

/*
 * Shard-local completion of the k lanes' records in `workspace` (as left by
 * sb_lmhead_records for M, k and T = tiles_per_shard) into `payload` (device, 4-byte
 * aligned, sb_payload_bytes(M, k, surface) bytes), adding col_offset (>= 0) to every column
 * so that a caller holding only a slice of W (for example one device of a
 * vocabulary-sharded head) produces global columns.  Enqueued on stream.
 */
int32_t sb_pack_shard_records(const void *workspace, int64_t M, int32_t k,
                              int32_t tiles_per_shard, int32_t surface, int64_t col_offset,
                              void *payload, void *stream);

/*
 * Cross-lane merge of k lane payloads (device, lane-major as above): writes out->token and,
 * where non-NULL, out->token_logprob and out->lse (target log-probs are not carried by the
 * payload; out->workspace is not used).  temperature as for sb_lmhead_project.
 */
int32_t sb_merge_shard_payload(const void *payload, int64_t M, int32_t k, int32_t surface,
                               float temperature, const sb_outputs *out, void *stream);

/*
 * Row-parallel partial completion ("SemBridge", Section 6.4 and Table 3: in a row-parallel
 * MLP down projection each tensor-parallel lane owns a slice of the reduction dimension and
 * produces an incomplete full-width partial; the partials must be summed -- the completion
 * obligation of Section 3.5 -- before a consumer observes the value).
 *   Y[m][n] = sum over lanes l (ascending) of P_l[m][n],
 *   P_l[m][n] = sum over lane l's reduction columns of X[m][i] * W[n][i].
 *   X          device bf16 [M, K] row-major (activations), 16-byte aligned; 1 <= M <= 256.
 *   W          device bf16 [N, K] row-major (weights), 16-byte aligned; N >= 1.
 *   K          a multiple of 64 * lanes (each lane's slice is whole 64-column blocks).
 *   lanes      >= 1.
 *   Y          device [M, N] row-major: fp32 when y_bf16 == 0, else bf16 (round to nearest).
 *   workspace  device, 256-byte aligned, >= sb_partial_workspace_bytes(M, N, K, lanes):
 *              header (read by sb_last_device_status) and fp32 partials; no
 *              initialisation.  One call at a time per workspace.
 * The (128-feature tile, 64-column K block) work is split evenly over the SMs; each SM cuts
 * its share at lane boundaries and accumulates every piece in fp32 on the tensor cores.  A
 * second kernel (a programmatic dependent of the first) sums each tile's pieces in
 * ascending K order (lane 0's first), so the result bits do not depend on scheduling.  Two
 * kernels are enqueued on stream; returns SB_OK or an error with nothing enqueued.
 * The first kernel is a programmatic dependent launch: it starts loading W before the
 * preceding kernel in the stream has finished, so W must not be written by a kernel that
 * can still be running then (one that signals its dependents early); X and the workspace
 * are read only after that kernel has finished.
 * sb_partial_workspace_bytes depends on the shape and on the SM count of the current
 * device; it returns 0 for an invalid shape or when no CUDA device is usable.
 */
size_t sb_partial_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t lanes);
int32_t sb_partial_completion(const void *X, const void *W, int64_t M, int64_t N, int64_t K,
                              int32_t lanes, void *Y, int32_t y_bf16, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * The decision before the path ("SemBridge", Section 8.2, Equation (7)): between the
 * checker-accepted plans, project at the source (plan s) rather than transfer the complete
 * logits (plan r) when the transfer saved exceeds the local cost added:
 *   (bytes_ref - bytes_proj) / link_bytes_per_s + frame_startup_s * (frames_ref - frames_proj)
 *       > local_proj_s - local_ref_s.
 * Bytes and frames are those crossing the link per step; the local costs are the two plans'
 * on-device times (for example this library's sb_lmhead_project time for the projected
 * surface and for SB_FULL_LOGITS).  *margin_s (may be NULL) receives left minus right side.
 * Returns 1 (project), 0 (transfer complete logits), or -1 for a non-positive or non-finite
 * bandwidth or a negative or non-finite byte, frame or startup argument.  Host only.
 */
int32_t sb_select_source_projection(double bytes_ref, double bytes_proj, double frames_ref,
                                    double frames_proj, double link_bytes_per_s,
                                    double frame_startup_s, double local_proj_s,
                                    double local_ref_s, double *margin_s);

/* Device status of the last call that used out->workspace: SB_OK, SB_ERR_DEVICE_TIMEOUT
 * (a bounded wait gave up) or SB_ERR_INVALID_ARG (a scoring target outside [0, V); when
 * both happen the timeout is reported).  Synchronous: copies the header to the host (call
 * it after synchronising the stream).  Returns SB_ERR_CUDA if the copy fails. */
int32_t sb_last_device_status(const sb_outputs *out);

/* Static description of a status code; never NULL. */
const char *sb_status_string(int32_t status);

/* Number of SMs and compute capability (major * 10 + minor) of the current device, as the
 * library sees them; -1 without a usable device. */
int32_t sb_device_info(int32_t *num_sms, int32_t *cc);

/* Test hook for the device watchdog.  stall_epilogue != 0 makes the epilogue warps of
 * later sb_lmhead_project calls wait on a barrier that nothing ever arrives at, so their
 * bounded wait runs out and the call reports SB_ERR_DEVICE_TIMEOUT through
 * sb_last_device_status (the outputs are then undefined).  wait_limit_ns (> 0) is the
 * time limit of every device-side wait (default 2 s).  Process-wide; not for production.
 * Returns SB_ERR_INVALID_ARG for wait_limit_ns == 0. */
int32_t sb_debug_configure(int32_t stall_epilogue, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SB_H */
