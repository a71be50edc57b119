// warp_topk.cuh -- one warp's exact top-k (k <= 32) of a chunk of a query's scores,
// and the merge of chunks' top-k lists: the selection steps of the warp top-k path
// (rows read from HBM) and of the fused score-then-select kernel (rows in shared
// memory).
//
// The selection is the one of "#2093 sm_75: the prompt path's top-k with one
// full read of the scores" (description, step 3): the k largest keys, ties
// to the lower block id.  Candidates travel packed as (key << 32) | ~id, so a
// larger packed value is exactly "taken first".  Each step bounds the k-th
// largest key from below with a few keys that are provably distinct entries,
// keeps only the entries at or above the bound (a few more than k on continuous
// scores) and ranks those exactly; heavy ties (more than 64 survivors) report
// failure and the caller falls back to the radix warp select.
#pragma once

#include "qsa_device.cuh"

namespace qsa {

// The exact top-k (k <= 32) of a chunk of n > k scores (block ids lo + i), written
// to dst[0..k) as packed candidates in descending order, the chunk held in registers
// (n <= 128 * NV, one read).  Each lane keeps the two largest keys of its share; the
// k-th largest of those 64 bounds the answer from below; the keys at or above it
// (about k + 4 on continuous scores) are gathered into buf (64 entries) at offsets
// from one warp scan of the lanes' counts, and their exact ranks pick the top k.
// Returns false, having written nothing, when more than 64 keys reach the bound
// (heavy ties) or fewer than k of the 64 keys are nonzero.  load4(v) returns entries
// 4v .. 4v + 3 (called for 4v < n; entries at or past n may hold anything); load1(i)
// returns entry i again for the few that reach the bound.  FULL: the caller
// guarantees n == 128 * NV, and no entry is tested against n.
template <int NV, bool FULL = false, typename Load4, typename Load1>
__device__ __forceinline__ bool warp_top_regs(Load4 &&load4, Load1 &&load1, int n, int k, int lo, uint64_t *buf,
                                              uint64_t *dst) {
    static_assert(NV * 4 <= 32, "one survivor bit per entry of a lane");
    const int lane = threadIdx.x & 31;
    // every load in flight before the first use
    float4 f[NV];
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int v = lane + 32 * t;
        f[t] = FULL || 4 * v < n ? load4(v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t key[NV][4];
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int v = lane + 32 * t;
        const float e[4] = {f[t].x, f[t].y, f[t].z, f[t].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) key[t][c] = FULL || 4 * v + c < n ? score_key(e[c]) : 0u;
    }
    uint32_t a1[4] = {0u, 0u, 0u, 0u}, a2[4] = {0u, 0u, 0u, 0u};   // one top-2 per component
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            a2[c] = max(a2[c], min(a1[c], key[t][c]));
            a1[c] = max(a1[c], key[t][c]);
        }
    uint32_t m1 = a1[0], m2 = a2[0];
#pragma unroll
    for (int c = 1; c < 4; ++c) {   // top-2 of two top-2 pairs
        m2 = max(min(m1, a1[c]), max(m2, a2[c]));
        m1 = max(m1, a1[c]);
    }
    // absent entries have key 0, below any nonzero bound; a zero bound (fewer than k
    // nonzero keys among the 64) gives no filter
    const uint32_t lb = warp_bound_from_top2(m1, m2, k);
    if (lb == 0u) return false;
    uint32_t surv = 0u;   // bit 4t + c: entry (t, c) of this lane reaches the bound
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (key[t][c] >= lb) surv |= 1u << (4 * t + c);
    const int nk = __popc(surv);
    const int incl = warp_incl_scan(nk);
    const int m = __shfl_sync(kFull, incl, 31);
    if (m > 64) return false;
    int pos = incl - nk;
    while (surv) {   // about one survivor per lane: read it again rather than test every entry
        const int bit = __ffs(surv) - 1;
        surv &= surv - 1u;
        const int i = 4 * (lane + 32 * (bit >> 2)) + (bit & 3);
        buf[pos++] = pack_cand(score_key(load1(i)), lo + i);
    }
    __syncwarp();
    warp_rank_top(buf, m, k, [&](int r, uint64_t c) { dst[r] = c; });
    return true;
}

// The register form on a shared-memory row whose storage extends to a multiple of
// four entries past n (the fused kernel's rows start on 512-byte boundaries).
template <int NV>
__device__ __forceinline__ bool stage_a_regs(const float *row, int n, int k, int lo, uint64_t *buf, uint64_t *dst) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    auto load4 = [&](int v) { return r4[v]; };
    auto load1 = [&](int i) { return row[i]; };
    return n == 128 * NV ? warp_top_regs<NV, true>(load4, load1, n, k, lo, buf, dst)
                         : warp_top_regs<NV>(load4, load1, n, k, lo, buf, dst);
}

// The same selection for shared-memory rows too long for registers: the row is read
// three times (top-2, count, gather) instead of once.
__device__ __forceinline__ bool stage_a_smem(const float *row, int n, int k, int lo, uint64_t *buf, uint64_t *dst) {
    const int lane = threadIdx.x & 31;
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int n4 = (n + 3) >> 2;
    uint32_t a1[4] = {0u, 0u, 0u, 0u}, a2[4] = {0u, 0u, 0u, 0u};
#pragma unroll 2
    for (int v = lane; v < n4; v += 32) {
        const float4 f = r4[v];
        const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t key = 4 * v + c < n ? score_key(e[c]) : 0u;
            a2[c] = max(a2[c], min(a1[c], key));
            a1[c] = max(a1[c], key);
        }
    }
    uint32_t m1 = a1[0], m2 = a2[0];
#pragma unroll
    for (int c = 1; c < 4; ++c) {
        m2 = max(min(m1, a1[c]), max(m2, a2[c]));
        m1 = max(m1, a1[c]);
    }
    const uint32_t lb = warp_bound_from_top2(m1, m2, k);
    int nk = 0;
#pragma unroll 2
    for (int v = lane; v < n4; v += 32) {
        const float4 f = r4[v];
        const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) nk += 4 * v + c < n && score_key(e[c]) >= lb;
    }
    const int incl = warp_incl_scan(nk);
    const int m = __shfl_sync(kFull, incl, 31);
    if (m > 64) return false;
    int pos = incl - nk;
    for (int v = lane; v < n4; v += 32) {
        const float4 f = r4[v];
        const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t key = score_key(e[c]);
            if (4 * v + c < n && key >= lb) buf[pos++] = pack_cand(key, lo + 4 * v + c);
        }
    }
    __syncwarp();
    warp_rank_top(buf, m, k, [&](int r, uint64_t c) { dst[r] = c; });
    return true;
}

// Stage B of one query, fast form (k <= 32).  list holds the query's chunks, chunk
// c at list[c * kc], its cnt_c = min(kc, max(0, n - c * S)) candidates in
// descending order.  The keys of 64 sampled heads (rank e / nch of chunk e % nch,
// e < 64) bound the k-th largest key from below; the candidates at or above it
// are a prefix of each chunk, gathered into buf and ranked exactly.  The
// selected ids go to out[0..k) ascending.  Every step counts against values
// broadcast from shared memory rather than running a sorting network, which
// keeps the dependent chain short: stage B runs on one CTA while the rest of
// the GPU is idle.  Returns false, having written nothing, when more than 64
// candidates reach the bound.
__device__ __forceinline__ bool stage_b_fast(const uint64_t *list, int nch, int kc, int S, int n, int k,
                                             uint64_t *buf, int32_t *sid, int32_t *out) {
    const int lane = threadIdx.x & 31;
    uint32_t *bk = reinterpret_cast<uint32_t *>(buf);   // the 64 sampled keys, then the gathered candidates
    uint32_t x[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int e = 2 * lane + s, c = e % nch, rr = e / nch;
        x[s] = rr < min(kc, n - c * S) ? cand_key(list[c * kc + rr]) : 0u;
        bk[e] = x[s];
    }
    __syncwarp();
    // the k-th largest sample: the largest x with at least k samples >= x
    int ge0 = 0, ge1 = 0;
    const uint4 *bk4 = reinterpret_cast<const uint4 *>(bk);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint4 q = bk4[j];
        ge0 += (q.x >= x[0]) + (q.y >= x[0]) + (q.z >= x[0]) + (q.w >= x[0]);
        ge1 += (q.x >= x[1]) + (q.y >= x[1]) + (q.z >= x[1]) + (q.w >= x[1]);
    }
    const uint32_t lb = warp_max(max(ge0 >= k ? x[0] : 0u, ge1 >= k ? x[1] : 0u));
    __syncwarp();
    if (lb == 0u) return false;   // fewer than k nonzero heads: no bound
    int m = 0;
    for (int c0 = 0; c0 < nch; c0 += 32) {
        const int c = c0 + lane;
        int p = 0;
        if (c < nch) {
            const int cc = min(kc, n - c * S);
            while (p < cc && cand_key(list[c * kc + p]) >= lb) ++p;
        }
        const int incl = warp_incl_scan(p);
        const int off = m + incl - p;
        for (int i = 0; i < p && off + i < 64; ++i) buf[off + i] = list[c * kc + i];
        m += __shfl_sync(kFull, incl, 31);
    }
    __syncwarp();
    if (m > 64) return false;
    warp_rank_top(buf, m, k, [&](int r, uint64_t c) { sid[r] = cand_id(c); });
    // ascending ids: each selected id's slot is the number of selected ids below it
    if (lane < k) {
        const int32_t id = sid[lane];
        int below = 0;
        for (int t = 0; t < k; ++t) below += sid[t] < id;
        out[below] = id;
    }
    __syncwarp();
    return true;
}

}  // namespace qsa
