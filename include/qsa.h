/*
 * qsa.h -- C ABI of the GB300 (sm_103a) query-sparse-attention block selection
 * library, libqsa.so.
 *
 * The path selects, for every query, the KV blocks (64 tokens each) that a
 * sparse attention step will read:
 *
 *   1. block scorer:  score[q][b] = sum_h w[q][h] * relu(dot(q[q][h][:], kblk[b][:]))
 *      over the indexer heads h, head dim 128, one key row per block (the last,
 *      partial block of a context has a key like any other);
 *   2. block top-k:   the k blocks of highest score, ties to the lower block id,
 *      emitted as ids in ascending block order, -1 padded when n < k.
 *
 * Sources: the scorer is the "qsa_block_scores" step of "#1091 qsa_select:
 * FP32 tiled block scores below sm_80" (section "What": rows = query x indexer
 * head, K = 128, ReLU per head summed per block; the tail block).  The top-k
 * rule is the threshold / "above" / tie-budget rule of "#2093 sm_75: the
 * prompt path's top-k with one full read of the scores" (description, steps
 * 1-4), and the decode split is the two-stage split of Strata PR #3987
 * (section "Approach").
 *
 * Conventions for every entry point:
 *  - Every pointer argument except the ones marked "host" is DEVICE memory owned
 *    by the caller.  The library never allocates or frees memory on a call and
 *    never synchronises the device.  Scratch lives in the caller's workspace, with
 *    one exception: qsa_block_topk_static uses a fixed scratch array compiled into
 *    the library (see there); no other entry point keeps device state between calls.
 *  - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default stream)
 *    and runs asynchronously; the return value reports host-side validation and
 *    launch errors only.  Device-side contract violations are recorded as bits in
 *    the workspace flags word (QSA_FLAG_*), readable with qsa_read_flags().
 *  - On any error status nothing is enqueued; qsa_last_error() (thread-local)
 *    returns a one-line reason.
 *  - One workspace must not be used by two calls that can run concurrently
 *    (e.g. on two streams); give each stream its own workspace.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_VERSION 1

/* Head dimension of q and kblk rows; the only value supported. */
#define QSA_HEAD_DIM 128
/* Largest k (blocks selected per query). */
#define QSA_MAX_K 1024
/* Largest max_blocks (KV capacity in blocks). */
#define QSA_MAX_BLOCKS (1 << 24)

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or enum value */
    QSA_ERR_UNSUPPORTED = 2, /* a forced path that cannot run this shape */
    QSA_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than qsa_workspace_bytes() */
    QSA_ERR_CUDA = 4         /* a CUDA runtime/driver call or a launch failed */
} qsa_status;

typedef enum {
    QSA_F32 = 0,  /* IEEE binary32 */
    QSA_BF16 = 1, /* bfloat16 (upper half of a binary32) */
    QSA_E4M3 = 2, /* 8-bit floating point E4M3 of the OCP FP8 specification (sign, 4 exponent bits
                     with bias 7, 3 mantissa bits; no infinities, S.1111.111 = NaN) */
    QSA_F16 = 3   /* IEEE binary16 (qsa_select_attention only) */
} qsa_dtype;

/* Top-k path.  AUTO picks from host-visible sizes only; the others force a path
 * (tests).  Every path returns the same ids. */
typedef enum {
    QSA_PATH_AUTO = 0,
    QSA_PATH_SPLIT = 1,    /* multi-CTA chunk split + last-CTA merge (decode windows) */
    QSA_PATH_SAMPLE = 2,   /* one read against a sampled lower bound (+ radix fallback) */
    QSA_PATH_REGISTER = 3, /* whole row in registers, one CTA per query */
    QSA_PATH_RADIX = 4,    /* multi-pass radix select over global memory, any size */
    QSA_PATH_WARP = 5      /* k <= 32, rows of up to 8,192 blocks held in registers (one warp per
                              1,024): a bound from the row's lane maxima keeps a few more than k
                              scores, which are ranked exactly; heavy ties take a per-chunk select
                              and merge */
} qsa_path;

typedef void *qsa_stream; /* a cudaStream_t */

/* Bits of the workspace flags word (sticky until cleared by qsa_read_flags). */
#define QSA_FLAG_NBLOCKS_CLAMPED 0x1u /* some n_blocks[q] was < 0 or > its bound; clamped */
#define QSA_FLAG_WAIT_TIMEOUT 0x2u    /* a kernel gave up a bounded wait; its outputs are invalid */
#define QSA_FLAG_INTERNAL 0x4u        /* an internal consistency check failed */
#define QSA_FLAG_SAMPLE_FALLBACK 0x8u /* not an error: some query of the sampled filter had too few
                                         or too many candidates and was selected from its whole row */
#define QSA_FLAG_BAD_ID 0x10u         /* qsa_select_attention skipped an id outside its query's
                                         context (an id other than -1) */

/* Query heads per KV head (GQA group) of qsa_select_attention. */
#define QSA_ATTN_GROUP 16
/* Largest k of qsa_select_attention. */
#define QSA_ATTN_MAX_K 64

/*
 * Workspace size in bytes for calls with these sizes: fused != 0 for the fused
 * form of qsa_select (its per-CTA candidate lists take up to 4,096 entries per
 * query), else any other call.  A workspace sized for (nq, max_blocks, k, fused)
 * serves every call with sizes at or below these.  The workspace must be zero-filled before its first use (e.g. by
 * qsa_workspace_init); every call leaves it in a reusable state.  Returns 0 for
 * invalid sizes.
 */
size_t qsa_workspace_bytes(int nq, int max_blocks, int k, int fused);

/* Zero-fill `ws_bytes` bytes of workspace `ws` on `stream` (cudaMemsetAsync). */
qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, qsa_stream stream);

/*
 * Block scores: scores[q * scores_stride + b] for 0 <= b < n_blocks[q].
 *
 *   q        [nq][n_heads][128]  dtype `dt` (fp32, bf16 or fp8 e4m3), row-major, 16-byte aligned
 *   w        [nq][n_heads]       fp32
 *   kblk     [max_blocks][128]   dtype `dt`, row-major, 16-byte aligned
 *   n_blocks [nq]                int32 on the DEVICE: blocks in each query's context,
 *                                clamped on the device to [0, bound] where bound =
 *                                active_blocks if active_blocks >= 0, else max_blocks
 *                                (a clamp sets QSA_FLAG_NBLOCKS_CLAMPED)
 *   active_blocks                host int: -1 (unknown) or an upper bound on every
 *                                n_blocks[q] (values above max_blocks act as max_blocks);
 *                                it sizes the grid and never changes a result
 *   scores   [nq][scores_stride] fp32, scores_stride >= max_blocks; entries at
 *                                b >= n_blocks[q] are not written
 *   ws, ws_bytes                 workspace (may be NULL/0: then device flags are not
 *                                recorded)
 *
 * Arithmetic: products on the tensor cores (bf16 x bf16 -> fp32, e4m3 x e4m3 ->
 * fp32, or fp32 split in three tf32 products), accumulated in fp32; ReLU and the
 * head-weighted sum in fp32.  n_heads must be 1, 2, 4, 8 or 16.  e4m3 stores the
 * indexer keys (and queries) in 8 bits, as the pages' engine stores its KV cache
 * in 8 bits ("--kv int8"); the tensor-core 8-bit format of this GPU is e4m3.
 * Launch: the kernel is launched as a programmatic dependent of the work before it
 * on `stream`: its CTAs may be scheduled while that work drains, and wait at entry,
 * before they take tensor memory or touch any buffer, until it has completed.
 * Errors: QSA_ERR_INVALID_ARG for NULL q/w/kblk/n_blocks/scores, nq < 1,
 * head_dim != 128, unsupported n_heads, max_blocks outside [1, QSA_MAX_BLOCKS],
 * scores_stride < max_blocks, misaligned q/kblk, a dtype other than QSA_F32,
 * QSA_BF16 or QSA_E4M3.
 */
qsa_status qsa_block_scores(const void *q, const float *w, const void *kblk, qsa_dtype dt,
                            const int32_t *n_blocks, int nq, int n_heads, int head_dim,
                            int max_blocks, int active_blocks, float *scores,
                            int64_t scores_stride, void *ws, size_t ws_bytes, qsa_stream stream);

/*
 * Block top-k over given fp32 scores.
 *
 *   scores   [nq][scores_stride] fp32 (NaN is outside the contract; -0 == +0); every
 *            entry below the bound (active_blocks, else max_blocks) must be readable
 *            memory: entries at or past n_blocks[q] may be read but never affect ids
 *   n_blocks [nq] int32 on the DEVICE, clamped as for qsa_block_scores
 *   k        1 <= k <= QSA_MAX_K
 *   ids      [nq][k] int32 out: the selected block ids in ascending order; when
 *            n_blocks[q] < k the first n_blocks[q] slots hold 0..n-1 and the rest -1
 *   ws       workspace of at least qsa_workspace_bytes(nq, max_blocks, k, 0) bytes
 *   path     QSA_PATH_AUTO, or a forced path (QSA_ERR_UNSUPPORTED if it cannot run
 *            this shape)
 *
 * Selection: keep the blocks that come first in the order (score descending,
 * block id ascending).  Every path gives the same ids.
 */
qsa_status qsa_block_topk(const float *scores, int64_t scores_stride, const int32_t *n_blocks,
                          int nq, int max_blocks, int active_blocks, int k, int32_t *ids,
                          void *ws, size_t ws_bytes, qsa_path path, qsa_stream stream);

/*
 * Block top-k for callers that cannot allocate device memory.  No passage of the
 * source pages has a counterpart to this call; it exists for callers that may
 * not call cudaMalloc where they select blocks (a fixed memory arena that must
 * not grow, a plug-in given only its input and output buffers, a serving path
 * where device allocation is forbidden).
 *
 * Same arguments, results and errors as qsa_block_topk, without ws / ws_bytes:
 * the scratch is an 8 MiB array compiled into the library, held on every GPU
 * that loads it until the process exits.  Sizes whose workspace
 * (qsa_workspace_bytes(nq, max_blocks, k, 0)) exceeds 8 MiB are rejected with
 * QSA_ERR_WORKSPACE and nothing is launched.  The call never allocates.
 *
 * The first call on each device looks up the scratch's device address (a CUDA
 * runtime query, with that device current) and caches it, and looks it up again
 * when the device's context has been replaced (after cudaDeviceReset); make that
 * first call before any stream capture.  A call rejected by its argument checks
 * enqueues nothing, not even the clear below.  All calls share the one scratch array: the parts
 * that must start at zero are cleared on `stream` at the start of every call,
 * and calls that can overlap on the GPU (different streams or host threads)
 * race with each other.  The device flags of these calls are not readable.
 */
qsa_status qsa_block_topk_static(const float *scores, int64_t scores_stride, const int32_t *n_blocks, int nq,
                                 int max_blocks, int active_blocks, int k, int32_t *ids, qsa_path path,
                                 qsa_stream stream);

/*
 * KV-sharded selection, stage A: the candidates of one shard of the KV blocks.
 * A query's selection restricted to a subset of its blocks is a prefix of that
 * subset's selection order (score descending, block id ascending), so the k best
 * blocks of every shard, merged by qsa_merge_candidates, select exactly the blocks
 * one call over all of them selects (Strata PR #3987, section "Approach": each
 * chunk keeps its top k, one CTA per query selects over the union).  The shards
 * may live on different GPUs: each computes its candidates, an all-gather collects
 * nq x k of them per shard, and every GPU merges.
 *
 *   scores, scores_stride, n_blocks, nq, max_blocks, active_blocks, k, ws, ws_bytes,
 *   path           as for qsa_block_topk, over this shard's blocks (local ids 0 ..
 *                  n_blocks[q] - 1)
 *   block_offset   host int: the global id of the shard's first block; ids
 *                  block_offset + max_blocks - 1 must stay below 2^31 - 1
 *   cand_ids       [nq][k] int32 out: the shard's selection as global ids
 *                  (block_offset + local id), ascending, -1 padded when n_blocks[q] < k
 *   cand_scores    [nq][k] fp32 out: each candidate's score (-inf where the id is -1)
 *
 * Two launches on `stream`: the top-k (any path) into cand_ids, then a kernel that
 * reads the candidates' scores and offsets their ids.
 * Errors: as qsa_block_topk, plus QSA_ERR_INVALID_ARG for NULL cand_scores /
 * cand_ids or a block_offset outside the range above.
 */
qsa_status qsa_block_candidates(const float *scores, int64_t scores_stride, const int32_t *n_blocks, int nq,
                                int max_blocks, int active_blocks, int k, int32_t block_offset, float *cand_scores,
                                int32_t *cand_ids, void *ws, size_t ws_bytes, qsa_path path, qsa_stream stream);

/*
 * KV-sharded selection, stage B: the k blocks of highest score over every shard's
 * candidates, ties to the lower global id, emitted as ids in ascending order (-1
 * padded when all shards together hold fewer than k candidates).
 *
 *   cand_scores  [n_shards][nq][k] fp32: the shards' qsa_block_candidates outputs,
 *                shard-major (the layout an all-gather of the [nq][k] arrays leaves)
 *   cand_ids     [n_shards][nq][k] int32: their global ids; entries < 0 are empty;
 *                the shards' ids must be distinct (disjoint block ranges)
 *   ids          [nq][k] int32 out
 *
 * One launch (one CTA per query), no workspace.
 * Errors: QSA_ERR_INVALID_ARG for NULL pointers, nq < 1, k outside [1, QSA_MAX_K],
 * n_shards < 1, n_shards x nq x k >= 2^31; QSA_ERR_UNSUPPORTED when n_shards x k
 * exceeds 4,096 candidates per query.
 */
qsa_status qsa_merge_candidates(const float *cand_scores, const int32_t *cand_ids, int n_shards, int nq, int k,
                                int32_t *ids, qsa_stream stream);

/*
 * Score then select, in one call.
 *
 * fused == 0 (chained): the scorer writes `scores` (required), then the top-k
 *   reads them; both are the calls above.
 * fused != 0: the scores never go to HBM.  The scorer keeps each CTA's block
 *   range of scores on chip and, per query, one warp lists every block of that
 *   range that can be in the selection (the scores at or above the k-th largest
 *   lane maximum for k <= 32, else the range's exact top k) in the workspace with
 *   the list's length; a merge kernel, launched as its programmatic dependent
 *   with one CTA per query, selects over the lists (a query's selection
 *   restricted to a range is a prefix of that range's order: Strata PR #3987,
 *   section "Approach").  No CTA waits for another.  `scores` may be NULL; when
 *   given, it also receives the scores (the same values the chained scorer
 *   writes).  `path` must be QSA_PATH_AUTO.  Shapes whose per-CTA scores do not
 *   fit on chip, or whose lists exceed the merge's 4,096 candidates per query
 *   (large k with very long contexts), return QSA_ERR_UNSUPPORTED; use the
 *   chained form for those.
 * Arguments as in qsa_block_scores / qsa_block_topk; ws must hold
 * qsa_workspace_bytes(nq, max_blocks, k, fused) bytes.
 */
qsa_status qsa_select(const void *q, const float *w, const void *kblk, qsa_dtype dt,
                      const int32_t *n_blocks, int nq, int n_heads, int head_dim, int max_blocks,
                      int active_blocks, int k, int32_t *ids, float *scores,
                      int64_t scores_stride, int fused, void *ws, size_t ws_bytes,
                      qsa_path path, qsa_stream stream);

/*
 * Selection attention, forward, over the blocks each query selected: the step
 * that reads the ids, as described in "[wave] NSA: LDS optimization for
 * block-gather in selection attention" (section "Problem": a query reads the
 * tokens of its selected blocks; "LDS staging strategies" 1: the heads of a GQA
 * group read one on-chip copy of each block's K and V).  For query q and
 * attention head h, with KV head g = h / QSA_ATTN_GROUP:
 *
 *   s_t       = dot(qa[q][h][:], K[g][t][:])
 *   o[q][h]   = sum_t exp(scale (s_t - m)) V[g][t][:] / sum_t exp(scale (s_t - m)),  m = max_t s_t
 *   lse[q][h] = scale m + log(sum_t exp(scale (s_t - m)))
 *
 * over the tokens t = 64 b + r (0 <= r < 64) of the distinct ids b >= 0 of
 * ids[q][0..k) with t < n_tokens[q].  A query with no such token gets o = 0 and
 * lse = -inf.
 *
 *   dt        QSA_BF16 or QSA_F16: the format of qa, kcache and vcache_t
 *   qa        [nq][n_heads][128] dtype `dt`, row-major, 16-byte aligned
 *   kcache    [n_kv_heads][capacity][128] dtype `dt` (K[g][t] = token rows), 16-byte aligned
 *   vcache_t  [n_kv_heads][capacity / 64][128][64] dtype `dt`: each 64-token block of V
 *             stored dimension-major, element [g][b][d][r] = V[g][64 b + r][d];
 *             16-byte aligned
 *   ids       [nq][k] int32: block ids (e.g. the ids of qsa_select), -1 = none, in
 *             any order; an id outside [0, ceil(n_tokens[q] / 64)) is skipped and sets
 *             QSA_FLAG_BAD_ID; a repeated id counts once
 *   n_tokens  [nq] int32 on the DEVICE: context length of each query, clamped to
 *             [0, capacity] (a clamp sets QSA_FLAG_NBLOCKS_CLAMPED)
 *   out       [nq][n_heads][128] fp32 out
 *   lse       [nq][n_heads] fp32 out, or NULL
 *   scale     softmax scale (host float), finite and > 0 (usually 1 / sqrt(128))
 *   ws        a workspace of at least 256 bytes (its flags word is used), or NULL
 *             (then device flags are not recorded)
 *
 * Arithmetic: the q.k products on the tensor cores (16-bit x 16-bit -> fp32); the
 * weights exp2((s - m) scale log2 e) in fp32, rounded to `dt` for the P.V product
 * on the tensor cores (-> fp32), and divided by the sum of the rounded weights.
 * Tokens at or past n_tokens take no part, whatever their K and V rows hold.
 * Launch: the kernel is launched as a programmatic dependent of the work before it
 * on `stream`; it reads nothing the caller wrote until that work has completed, so
 * behind a top-k of this library it starts while the top-k finishes.
 * Errors: QSA_ERR_INVALID_ARG for NULL qa/kcache/vcache_t/ids/n_tokens/out,
 * nq < 1, head_dim != 128, n_kv_heads < 1, n_heads != QSA_ATTN_GROUP *
 * n_kv_heads, k outside [1, QSA_ATTN_MAX_K], capacity < 64 or not a multiple of
 * 64, n_kv_heads * capacity >= 2^30, nq * n_heads >= 2^30, misaligned
 * qa/kcache/vcache_t, scale not finite or <= 0, ws smaller than 256 bytes or
 * not 256-byte aligned; QSA_ERR_UNSUPPORTED for a dtype other than QSA_BF16 or
 * QSA_F16.
 */
qsa_status qsa_select_attention(const void *qa, const void *kcache, const void *vcache_t, qsa_dtype dt,
                                const int32_t *ids, int k, const int32_t *n_tokens, int nq, int n_heads,
                                int n_kv_heads, int head_dim, int capacity, float scale, float *out,
                                float *lse, void *ws, size_t ws_bytes, qsa_stream stream);

/*
 * The V cache layout qsa_select_attention reads, from the token-row layout: for
 * every KV head g and every block b in [first_block, first_block + n_blocks),
 * vcache_t[g][b][d][r] = v[g][64 b + r][d] (d < 128, r < 64), copied bit for bit.
 * A cache writer converts the blocks an append touched (the last, partial block
 * again as it fills).  No passage of the source pages defines this call: it
 * serves the layout reading of the attention (each block of V dimension-major, so
 * the P.V product's operand is K-major).
 *
 *   v           [n_kv_heads][capacity][128] 16-bit values (bf16 or fp16), 16-byte aligned
 *   vcache_t    [n_kv_heads][capacity / 64][128][64], same element size, 16-byte aligned;
 *               must not overlap v
 *   capacity    tokens per KV head, a positive multiple of 64
 * Errors: QSA_ERR_INVALID_ARG for NULL or misaligned pointers, n_kv_heads outside
 * [1, 65535], capacity not a positive multiple of 64, n_kv_heads * capacity >= 2^30, a block
 * range outside [0, capacity / 64), n_blocks < 0.
 */
qsa_status qsa_vcache_transpose(const void *v, void *vcache_t, int n_kv_heads, int capacity, int first_block,
                                int n_blocks, qsa_stream stream);

/*
 * Copy the workspace flags word (QSA_FLAG_* bits) to host `*flags`, waiting for
 * `stream` to finish; clear it on the device when `clear` is nonzero.
 */
qsa_status qsa_read_flags(void *ws, uint32_t *flags /* host */, int clear, qsa_stream stream);

/* The path QSA_PATH_AUTO takes for these host-visible sizes (no launch). */
qsa_path qsa_auto_path(int nq, int max_blocks, int active_blocks, int k);

/* One-line reason for the last error status returned on this thread. */
const char *qsa_last_error(void);

/* QSA_VERSION of the loaded library. */
int qsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
