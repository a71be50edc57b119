// qsa_internal.h -- host-side declarations shared by the translation units of
// libqsa.so (launchers, workspace layout, error reporting).  Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qsa.h"

namespace qsa {

// Record a one-line reason for the status about to be returned (thread-local).
qsa_status fail(qsa_status st, const char *fmt, ...);
// Map a CUDA error to QSA_ERR_CUDA with a reason; QSA_OK when err == cudaSuccess.
qsa_status check_cuda(cudaError_t err, const char *what);

int num_sms();  // SM count of the current device (cached per device)

// A 2-D TMA tensor map over a row-major [rows][inner] array of esize-byte elements
// (4: fp32, 2: bf16 or fp16, 1: 8-bit; the bytes are copied as they are), box of
// 128 bytes x box_rows, 128-byte swizzle;
// encoded once per (pointer, shape, device).
qsa_status get_map(CUtensorMap *out, const void *ptr, int esize, uint32_t inner, uint64_t rows, uint32_t box_rows);

// Candidate slots per (query, chunk) are sized for chunks of at least this many blocks.
constexpr int kMinChunk = 128;
// Shared-memory candidate capacity of the sampled-bound filter.
constexpr int kSampleCap = 4096;
// Largest row the register and sample paths hold on chip (1024 threads x 8 keys).
constexpr int kRegisterCap = 8192;
// Stage-B capacity of the split (slots of nchunks x k held by 256 threads x 16).
constexpr int kSplitSlots = 4096;
// Largest chunk of the split's stage A (256 threads x 4 keys).
constexpr int kSplitMaxChunk = 1024;
// Candidates per query the merge of sharded selections holds on chip (shards x k).
constexpr int kMergeCap = 4096;

// Workspace layout; every region starts on a 256-byte boundary.
struct WsLayout {
    size_t flags;     // uint32 flags word (QSA_FLAG_*)
    size_t tickets;   // uint32 [nq]       last-CTA tickets (zero between calls)
    size_t qflags;    // uint32 [nq]       per-query fallback flags of the sampled filter
    size_t counts;    // int32  [nq][maxch] candidates per chunk
    size_t ckeys;     // uint32 [nq][maxch][k]
    size_t cids;      // int32  [nq][maxch][k]
    size_t total;
    int maxch;
};
// fused: the candidate arrays hold at least kMergeCap entries per query (the fused
// select's per-CTA candidate lists)
WsLayout ws_layout(int nq, int max_blocks, int k, bool fused = false);

struct TopkArgs {
    const float *scores;
    int64_t stride;
    const int32_t *n_blocks;
    int nq;
    int bound;   // clamp bound of n_blocks (active blocks or capacity)
    int k;
    int32_t *ids;
    uint32_t *flags;
    uint32_t *tickets;
    uint32_t *qflags;
    int32_t *counts;
    uint32_t *ckeys;
    int32_t *cids;
    int maxch;
};

// Split geometry for a bound; chunk_len == 0 when the split cannot take it.
struct SplitGeom {
    int chunk_len;
    int nchunks;
};
SplitGeom split_geometry(int bound, int nq, int k, int maxch);

qsa_status launch_topk_radix(const TopkArgs &a, bool flagged_only, cudaStream_t s);
qsa_status launch_topk_register(const TopkArgs &a, cudaStream_t s);
qsa_status launch_topk_sample(const TopkArgs &a, cudaStream_t s);
// behind_scorer: the top-k follows the scorer of a chained select on the stream (its
// CTAs are launched early and wait on the SMs the scorer leaves free)
qsa_status launch_topk_warp(const TopkArgs &a, bool behind_scorer, cudaStream_t s);
qsa_status launch_topk_split(const TopkArgs &a, const SplitGeom &g, cudaStream_t s);

// Sharded selection: the candidates' scores and global ids after a shard's top-k
// (ids [nq][k] in place), and the merge of [n_shards][nq][k] candidates into ids.
qsa_status launch_candidates(const float *scores, int64_t stride, int32_t *ids, float *cand_scores, int nq, int k,
                             int32_t offset, cudaStream_t s);
// counts == nullptr: every slot with id >= 0; else the first counts[q * counts_stride + g]
// slots of shard g.  Shard g's candidates of query q start at
// ((g nq) + q) kslot; n_shards * kslot <= kMergeCap.
qsa_status launch_merge(const float *cand_scores, const int32_t *cand_ids, const int32_t *counts, int counts_stride,
                        int n_shards, int nq, int kslot, int k, int32_t *ids, cudaStream_t s);

struct ScorerArgs {
    const void *q;
    const float *w;
    const void *kblk;
    qsa_dtype dt;
    const int32_t *n_blocks;
    int nq;
    int n_heads;
    int max_blocks;
    int bound;
    float *scores;
    int64_t stride;
    uint32_t *flags;
    // fused score-then-select (fused != 0): scores may be null; the CTAs' candidate
    // lists go to cand_scores / cand_ids (the workspace's ckeys / cids regions) with
    // their lengths in counts, and a merge kernel writes ids
    bool fused;
    int32_t *ids;
    int k;
    float *cand_scores;
    int32_t *cand_ids;
    int32_t *counts;
    int maxch;
};
qsa_status launch_scorer(const ScorerArgs &a, cudaStream_t s);

struct AttnArgs {
    qsa_dtype dt;   // QSA_BF16 or QSA_F16
    const void *qa;
    const void *kcache;
    const void *vcache_t;
    const int32_t *ids;
    int k;
    const int32_t *n_tokens;
    int nq;
    int n_heads;
    int n_kv_heads;
    int capacity;
    float scale;
    float *out;
    float *lse;
    uint32_t *flags;
};
qsa_status launch_select_attention(const AttnArgs &a, cudaStream_t s);
qsa_status launch_vcache_transpose(const void *v, void *vcache_t, int n_kv_heads, int capacity, int first_block,
                                   int n_blocks, cudaStream_t s);

}  // namespace qsa
