// qsa_api.cu -- the C ABI of libqsa.so: argument checks, workspace layout,
// top-k path dispatch, and the chained select.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "qsa_internal.h"

namespace qsa {

static thread_local char g_err[512] = "";

qsa_status fail(qsa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

qsa_status check_cuda(cudaError_t err, const char *what) {
    if (err == cudaSuccess) return QSA_OK;
    return fail(QSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

int num_sms() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(int nq, int max_blocks, int k, bool fused) {
    WsLayout L{};
    L.maxch = (max_blocks + kMinChunk - 1) / kMinChunk;
    const size_t per_query = std::max<size_t>((size_t)L.maxch * k, fused ? (size_t)kMergeCap : 0);
    size_t off = 0;
    L.flags = off;
    off += 256;
    L.tickets = off;
    off += align256(sizeof(uint32_t) * (size_t)nq);
    L.qflags = off;
    off += align256(sizeof(uint32_t) * (size_t)nq);
    L.counts = off;
    off += align256(sizeof(int32_t) * (size_t)nq * L.maxch);
    L.ckeys = off;
    off += align256(sizeof(uint32_t) * (size_t)nq * per_query);
    L.cids = off;
    off += align256(sizeof(int32_t) * (size_t)nq * per_query);
    L.total = off;
    return L;
}

static int effective_bound(int max_blocks, int active_blocks) {
    return active_blocks >= 0 ? (active_blocks < max_blocks ? active_blocks : max_blocks) : max_blocks;
}

// Prompt calls above this many active blocks take the sampled filter; below it the
// register path reads the row once too and has no sampling step.
static constexpr int kSampleMinBlocks = 2048;

// Rows of up to 8,192 blocks at k <= 32 (every workload of the pages) take the warp
// path: one HBM read per row and no block-wide barrier in the selection; on GB300 it
// beats the split (decode), sampled (prompt) and register paths at every such size.
static constexpr int kWarpPathMaxK = 32;
static constexpr int kWarpPathMaxBlocks = 8192;

static qsa_path auto_path(int nq, int max_blocks, int active_blocks, int k) {
    const int bound = effective_bound(max_blocks, active_blocks);
    if (k <= kWarpPathMaxK && bound <= kWarpPathMaxBlocks) return QSA_PATH_WARP;
    const WsLayout L = ws_layout(nq, max_blocks, k);
    if (active_blocks < 0 && nq <= 16 && bound > k && split_geometry(bound, nq, k, L.maxch).chunk_len > 0)
        return QSA_PATH_SPLIT;
    if (bound <= kRegisterCap) {
        if (active_blocks >= 0 && bound >= kSampleMinBlocks) return QSA_PATH_SAMPLE;
        return QSA_PATH_REGISTER;
    }
    return QSA_PATH_RADIX;
}

static qsa_status check_common(int nq, int max_blocks, int active_blocks) {
    if (nq < 1) return fail(QSA_ERR_INVALID_ARG, "nq must be >= 1 (got %d)", nq);
    if (max_blocks < 1 || max_blocks > QSA_MAX_BLOCKS)
        return fail(QSA_ERR_INVALID_ARG, "max_blocks must be in [1, %d] (got %d)", QSA_MAX_BLOCKS,
                    max_blocks);
    if (active_blocks < -1)
        return fail(QSA_ERR_INVALID_ARG, "active_blocks must be -1 or >= 0 (got %d)", active_blocks);
    return QSA_OK;
}

static qsa_status check_ws(void *ws, size_t ws_bytes, int nq, int max_blocks, int k, bool fused = false) {
    if (!ws) return fail(QSA_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(QSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const size_t need = ws_layout(nq, max_blocks, k, fused).total;
    if (ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace too small: %zu bytes, need %zu", ws_bytes, need);
    return QSA_OK;
}

static qsa_status check_scorer_args(const void *q, const float *w, const void *kblk, int dt,
                                    const int32_t *n_blocks, int nq, int n_heads, int head_dim,
                                    int max_blocks, int active_blocks, const float *scores,
                                    int64_t stride, bool scores_required) {
    qsa_status st = check_common(nq, max_blocks, active_blocks);
    if (st != QSA_OK) return st;
    if (!q || !w || !kblk || !n_blocks) return fail(QSA_ERR_INVALID_ARG, "NULL q, w, kblk or n_blocks");
    if (scores_required && !scores) return fail(QSA_ERR_INVALID_ARG, "scores is NULL");
    if (dt != QSA_F32 && dt != QSA_BF16 && dt != QSA_E4M3) return fail(QSA_ERR_INVALID_ARG, "bad dtype %d", dt);
    if (head_dim != QSA_HEAD_DIM)
        return fail(QSA_ERR_INVALID_ARG, "head_dim must be %d (got %d)", QSA_HEAD_DIM, head_dim);
    if (n_heads != 1 && n_heads != 2 && n_heads != 4 && n_heads != 8 && n_heads != 16)
        return fail(QSA_ERR_INVALID_ARG, "n_heads must be 1, 2, 4, 8 or 16 (got %d)", n_heads);
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kblk)) & 15u)
        return fail(QSA_ERR_INVALID_ARG, "q and kblk must be 16-byte aligned");
    if (scores && stride < max_blocks)
        return fail(QSA_ERR_INVALID_ARG, "scores_stride %lld < max_blocks %d", (long long)stride,
                    max_blocks);
    if ((long long)nq * n_heads > (1ll << 30)) return fail(QSA_ERR_INVALID_ARG, "nq * n_heads too large");
    return QSA_OK;
}

static TopkArgs make_topk_args(const float *scores, int64_t stride, const int32_t *n_blocks, int nq,
                               int bound, int k, int32_t *ids, void *ws, const WsLayout &L) {
    char *base = static_cast<char *>(ws);
    TopkArgs a{};
    a.scores = scores;
    a.stride = stride;
    a.n_blocks = n_blocks;
    a.nq = nq;
    a.bound = bound;
    a.k = k;
    a.ids = ids;
    a.flags = reinterpret_cast<uint32_t *>(base + L.flags);
    a.tickets = reinterpret_cast<uint32_t *>(base + L.tickets);
    a.qflags = reinterpret_cast<uint32_t *>(base + L.qflags);
    a.counts = reinterpret_cast<int32_t *>(base + L.counts);
    a.ckeys = reinterpret_cast<uint32_t *>(base + L.ckeys);
    a.cids = reinterpret_cast<int32_t *>(base + L.cids);
    a.maxch = L.maxch;
    return a;
}

static qsa_status run_topk(const float *scores, int64_t stride, const int32_t *n_blocks, int nq,
                           int max_blocks, int active_blocks, int k, int32_t *ids, void *ws,
                           qsa_path path, cudaStream_t s, bool behind_scorer = false) {
    const int bound = effective_bound(max_blocks, active_blocks);
    const WsLayout L = ws_layout(nq, max_blocks, k);
    const TopkArgs a = make_topk_args(scores, stride, n_blocks, nq, bound, k, ids, ws, L);
    if (path == QSA_PATH_AUTO) path = auto_path(nq, max_blocks, active_blocks, k);
    switch (path) {
    case QSA_PATH_SPLIT: {
        const SplitGeom g = split_geometry(bound, nq, k, L.maxch);
        return launch_topk_split(a, g, s);
    }
    case QSA_PATH_SAMPLE:
        if (bound > kRegisterCap)
            return fail(QSA_ERR_UNSUPPORTED, "sample path holds at most %d blocks per row (bound %d)",
                        kRegisterCap, bound);
        return launch_topk_sample(a, s);
    case QSA_PATH_REGISTER:
        return launch_topk_register(a, s);
    case QSA_PATH_RADIX:
        return launch_topk_radix(a, false, s);
    case QSA_PATH_WARP:
        return launch_topk_warp(a, behind_scorer, s);
    default:
        return fail(QSA_ERR_INVALID_ARG, "bad path %d", (int)path);
    }
}

}  // namespace qsa

using namespace qsa;

extern "C" {

size_t qsa_workspace_bytes(int nq, int max_blocks, int k, int fused) {
    if (nq < 1 || max_blocks < 1 || max_blocks > QSA_MAX_BLOCKS || k < 1 || k > QSA_MAX_K) return 0;
    return ws_layout(nq, max_blocks, k, fused != 0).total;
}

qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, qsa_stream stream) {
    if (!ws) return fail(QSA_ERR_WORKSPACE, "workspace is NULL");
    return check_cuda(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)),
                      "cudaMemsetAsync(workspace)");
}

qsa_status qsa_block_scores(const void *q, const float *w, const void *kblk, qsa_dtype dt,
                            const int32_t *n_blocks, int nq, int n_heads, int head_dim,
                            int max_blocks, int active_blocks, float *scores,
                            int64_t scores_stride, void *ws, size_t ws_bytes, qsa_stream stream) {
    qsa_status st = check_scorer_args(q, w, kblk, (int)dt, n_blocks, nq, n_heads, head_dim,
                                      max_blocks, active_blocks, scores, scores_stride, true);
    if (st != QSA_OK) return st;
    if (ws && ws_bytes < 256) return fail(QSA_ERR_WORKSPACE, "workspace smaller than its 256-byte header");
    ScorerArgs a{};
    a.q = q;
    a.w = w;
    a.kblk = kblk;
    a.dt = dt;
    a.n_blocks = n_blocks;
    a.nq = nq;
    a.n_heads = n_heads;
    a.max_blocks = max_blocks;
    a.bound = effective_bound(max_blocks, active_blocks);
    a.scores = scores;
    a.stride = scores_stride;
    a.flags = ws ? reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + ws_layout(nq, max_blocks, 1).flags)
                 : nullptr;
    return launch_scorer(a, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_block_topk(const float *scores, int64_t scores_stride, const int32_t *n_blocks,
                          int nq, int max_blocks, int active_blocks, int k, int32_t *ids,
                          void *ws, size_t ws_bytes, qsa_path path, qsa_stream stream) {
    qsa_status st = check_common(nq, max_blocks, active_blocks);
    if (st != QSA_OK) return st;
    if (!scores || !n_blocks || !ids) return fail(QSA_ERR_INVALID_ARG, "NULL scores, n_blocks or ids");
    if (k < 1 || k > QSA_MAX_K) return fail(QSA_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", QSA_MAX_K, k);
    if (scores_stride < max_blocks)
        return fail(QSA_ERR_INVALID_ARG, "scores_stride %lld < max_blocks %d", (long long)scores_stride,
                    max_blocks);
    st = check_ws(ws, ws_bytes, nq, max_blocks, k);
    if (st != QSA_OK) return st;
    return run_topk(scores, scores_stride, n_blocks, nq, max_blocks, active_blocks, k, ids, ws, path,
                    static_cast<cudaStream_t>(stream));
}

qsa_status qsa_block_candidates(const float *scores, int64_t scores_stride, const int32_t *n_blocks, int nq,
                                int max_blocks, int active_blocks, int k, int32_t block_offset, float *cand_scores,
                                int32_t *cand_ids, void *ws, size_t ws_bytes, qsa_path path, qsa_stream stream) {
    qsa_status st = check_common(nq, max_blocks, active_blocks);
    if (st != QSA_OK) return st;
    if (!scores || !n_blocks || !cand_scores || !cand_ids)
        return fail(QSA_ERR_INVALID_ARG, "NULL scores, n_blocks, cand_scores or cand_ids");
    if (k < 1 || k > QSA_MAX_K) return fail(QSA_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", QSA_MAX_K, k);
    if (scores_stride < max_blocks)
        return fail(QSA_ERR_INVALID_ARG, "scores_stride %lld < max_blocks %d", (long long)scores_stride,
                    max_blocks);
    if (block_offset < 0 || (long long)block_offset + max_blocks > 0x7fffffffll)
        return fail(QSA_ERR_INVALID_ARG, "block_offset %d: global ids must lie in [0, 2^31 - 1)", block_offset);
    st = check_ws(ws, ws_bytes, nq, max_blocks, k);
    if (st != QSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = run_topk(scores, scores_stride, n_blocks, nq, max_blocks, active_blocks, k, cand_ids, ws, path, s);
    if (st != QSA_OK) return st;
    return launch_candidates(scores, scores_stride, cand_ids, cand_scores, nq, k, block_offset, s);
}

qsa_status qsa_merge_candidates(const float *cand_scores, const int32_t *cand_ids, int n_shards, int nq, int k,
                                int32_t *ids, qsa_stream stream) {
    if (!cand_scores || !cand_ids || !ids) return fail(QSA_ERR_INVALID_ARG, "NULL cand_scores, cand_ids or ids");
    if (nq < 1) return fail(QSA_ERR_INVALID_ARG, "nq must be >= 1 (got %d)", nq);
    if (k < 1 || k > QSA_MAX_K) return fail(QSA_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", QSA_MAX_K, k);
    if (n_shards < 1) return fail(QSA_ERR_INVALID_ARG, "n_shards must be >= 1 (got %d)", n_shards);
    if ((long long)n_shards * k > kMergeCap)
        return fail(QSA_ERR_UNSUPPORTED, "n_shards x k = %lld candidates per query; the merge holds at most %d",
                    (long long)n_shards * k, kMergeCap);
    if ((long long)n_shards * nq * k >= (1ll << 31))
        return fail(QSA_ERR_INVALID_ARG, "n_shards x nq x k too large");
    return launch_merge(cand_scores, cand_ids, nullptr, 0, n_shards, nq, k, k, ids, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_select(const void *q, const float *w, const void *kblk, qsa_dtype dt,
                      const int32_t *n_blocks, int nq, int n_heads, int head_dim, int max_blocks,
                      int active_blocks, int k, int32_t *ids, float *scores,
                      int64_t scores_stride, int fused, void *ws, size_t ws_bytes,
                      qsa_path path, qsa_stream stream) {
    qsa_status st = check_scorer_args(q, w, kblk, (int)dt, n_blocks, nq, n_heads, head_dim,
                                      max_blocks, active_blocks, scores, scores_stride, !fused);
    if (st != QSA_OK) return st;
    if (!ids) return fail(QSA_ERR_INVALID_ARG, "ids is NULL");
    if (k < 1 || k > QSA_MAX_K) return fail(QSA_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", QSA_MAX_K, k);
    st = check_ws(ws, ws_bytes, nq, max_blocks, k, fused != 0);
    if (st != QSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fused) {
        if (path != QSA_PATH_AUTO)
            return fail(QSA_ERR_UNSUPPORTED, "fused score-then-select has no top-k path to force (got %d)", (int)path);
        const WsLayout L = ws_layout(nq, max_blocks, k, true);
        char *base = static_cast<char *>(ws);
        ScorerArgs a{};
        a.q = q;
        a.w = w;
        a.kblk = kblk;
        a.dt = dt;
        a.n_blocks = n_blocks;
        a.nq = nq;
        a.n_heads = n_heads;
        a.max_blocks = max_blocks;
        a.bound = effective_bound(max_blocks, active_blocks);
        a.scores = scores;   // may be null
        a.stride = scores_stride;
        a.flags = reinterpret_cast<uint32_t *>(base + L.flags);
        a.fused = true;
        a.ids = ids;
        a.k = k;
        a.cand_scores = reinterpret_cast<float *>(base + L.ckeys);
        a.cand_ids = reinterpret_cast<int32_t *>(base + L.cids);
        a.counts = reinterpret_cast<int32_t *>(base + L.counts);
        a.maxch = L.maxch;
        return launch_scorer(a, s);
    }
    st = qsa_block_scores(q, w, kblk, dt, n_blocks, nq, n_heads, head_dim, max_blocks, active_blocks,
                          scores, scores_stride, ws, ws_bytes, stream);
    if (st != QSA_OK) return st;
    return run_topk(scores, scores_stride, n_blocks, nq, max_blocks, active_blocks, k, ids, ws, path, s, true);
}

qsa_status qsa_select_attention(const void *qa, const void *kcache, const void *vcache_t, qsa_dtype dt,
                                const int32_t *ids, int k, const int32_t *n_tokens, int nq, int n_heads,
                                int n_kv_heads, int head_dim, int capacity, float scale, float *out,
                                float *lse, void *ws, size_t ws_bytes, qsa_stream stream) {
    if (!qa || !kcache || !vcache_t || !ids || !n_tokens || !out)
        return fail(QSA_ERR_INVALID_ARG, "NULL qa, kcache, vcache_t, ids, n_tokens or out");
    if (nq < 1) return fail(QSA_ERR_INVALID_ARG, "nq must be >= 1 (got %d)", nq);
    if (head_dim != QSA_HEAD_DIM)
        return fail(QSA_ERR_INVALID_ARG, "head_dim must be %d (got %d)", QSA_HEAD_DIM, head_dim);
    if (n_kv_heads < 1 || (long long)n_heads != (long long)QSA_ATTN_GROUP * n_kv_heads)
        return fail(QSA_ERR_INVALID_ARG, "n_heads must be %d x n_kv_heads (got %d heads, %d KV heads)",
                    QSA_ATTN_GROUP, n_heads, n_kv_heads);
    if (k < 1 || k > QSA_ATTN_MAX_K)
        return fail(QSA_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", QSA_ATTN_MAX_K, k);
    if (capacity < 64 || capacity % 64)
        return fail(QSA_ERR_INVALID_ARG, "capacity must be a positive multiple of 64 (got %d)", capacity);
    if ((long long)n_kv_heads * capacity >= (1ll << 30))
        return fail(QSA_ERR_INVALID_ARG, "n_kv_heads * capacity too large");
    if ((long long)nq * n_heads >= (1ll << 30)) return fail(QSA_ERR_INVALID_ARG, "nq * n_heads too large");
    if ((reinterpret_cast<uintptr_t>(qa) | reinterpret_cast<uintptr_t>(kcache) |
         reinterpret_cast<uintptr_t>(vcache_t)) & 15u)
        return fail(QSA_ERR_INVALID_ARG, "qa, kcache and vcache_t must be 16-byte aligned");
    if (!(scale > 0.0f) || !(scale <= 3.4e38f)) return fail(QSA_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (ws && (ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return fail(QSA_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold at least 256 bytes");
    if (dt != QSA_BF16 && dt != QSA_F16)
        return fail(QSA_ERR_UNSUPPORTED, "selection attention takes bf16 or fp16 inputs (dtype %d)", dt);
    AttnArgs a{};
    a.dt = dt;
    a.qa = qa;
    a.kcache = kcache;
    a.vcache_t = vcache_t;
    a.ids = ids;
    a.k = k;
    a.n_tokens = n_tokens;
    a.nq = nq;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.capacity = capacity;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.flags = ws ? static_cast<uint32_t *>(ws) : nullptr;
    return launch_select_attention(a, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_vcache_transpose(const void *v, void *vcache_t, int n_kv_heads, int capacity, int first_block,
                                int n_blocks, qsa_stream stream) {
    if (!v || !vcache_t) return fail(QSA_ERR_INVALID_ARG, "NULL v or vcache_t");
    if ((reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(vcache_t)) & 15u)
        return fail(QSA_ERR_INVALID_ARG, "v and vcache_t must be 16-byte aligned");
    if (n_kv_heads < 1 || n_kv_heads > 65535)   // one grid row per KV head
        return fail(QSA_ERR_INVALID_ARG, "n_kv_heads must be in [1, 65535] (got %d)", n_kv_heads);
    if (capacity < 64 || capacity % 64)
        return fail(QSA_ERR_INVALID_ARG, "capacity must be a positive multiple of 64 (got %d)", capacity);
    if ((long long)n_kv_heads * capacity >= (1ll << 30))
        return fail(QSA_ERR_INVALID_ARG, "n_kv_heads * capacity too large");
    if (n_blocks < 0 || first_block < 0 || (long long)first_block + n_blocks > capacity / 64)
        return fail(QSA_ERR_INVALID_ARG, "blocks [%d, %d + %d) outside [0, %d)", first_block, first_block, n_blocks,
                    capacity / 64);
    const size_t bytes = (size_t)n_kv_heads * capacity * QSA_HEAD_DIM * 2;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(v), b0 = reinterpret_cast<uintptr_t>(vcache_t);
    if (a0 < b0 + bytes && b0 < a0 + bytes) return fail(QSA_ERR_INVALID_ARG, "v and vcache_t overlap");
    return launch_vcache_transpose(v, vcache_t, n_kv_heads, capacity, first_block, n_blocks,
                                   static_cast<cudaStream_t>(stream));
}

qsa_status qsa_read_flags(void *ws, uint32_t *flags, int clear, qsa_stream stream) {
    if (!ws || !flags) return fail(QSA_ERR_INVALID_ARG, "NULL workspace or flags");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    qsa_status st = check_cuda(cudaMemcpyAsync(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s),
                               "cudaMemcpyAsync(flags)");
    if (st != QSA_OK) return st;
    st = check_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (st != QSA_OK) return st;
    if (clear) return check_cuda(cudaMemsetAsync(ws, 0, sizeof(uint32_t), s), "cudaMemsetAsync(flags)");
    return QSA_OK;
}

qsa_path qsa_auto_path(int nq, int max_blocks, int active_blocks, int k) {
    if (nq < 1 || max_blocks < 1 || k < 1) return QSA_PATH_AUTO;
    return auto_path(nq, max_blocks, active_blocks, k);
}

const char *qsa_last_error(void) { return g_err; }

int qsa_version(void) { return QSA_VERSION; }

}  // extern "C"
