// topk.cu -- block top-k kernels over fp32 score rows.
//
// Four paths, all giving the ids of the rule in qsa_device.cuh:
//  * register: one CTA per query holds its whole row in registers (<= 8,192
//    blocks) and selects with no re-read -- the "register kernel" the pages name
//    for contexts within its reach (Strata PR #3987, "Problem and result").
//  * sample:   one CTA per query reads its row once; a lower bound LB taken as the
//    KS-th largest key among every 32nd block (KS = 2k/32 + 16) keeps the keys
//    >= LB as candidates on chip; with at least k and at most 4,096 candidates
//    the threshold, "above" and the tie budget over the candidates equal the
//    row's, else the query is flagged for the radix kernel ("#2093 sm_75: the
//    prompt path's top-k with one full read of the scores", steps 1-4).
//  * radix:    one CTA per query, multi-pass radix select straight from global
//    memory (four digit passes and the emit); any row length.  It is the
//    fallback of the sampled filter (run for flagged queries only).
//  * split:    stage A, one CTA per (query, chunk), keeps the chunk's top-k
//    candidates in the workspace; the last CTA of a query to finish (atomic
//    ticket, nothing waits) runs stage B over the candidates.  A query's
//    selection restricted to a chunk is a prefix of that chunk's order, so every
//    selected block is among its chunk's candidates (Strata PR #3987,
//    "Approach").
#include <algorithm>
#include <cstdio>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

__device__ __forceinline__ int clamp_blocks(const int32_t *n_blocks, int q, int bound,
                                            uint32_t *flags) {
    int n = n_blocks[q];
    if (n < 0 || n > bound) {
        if (flags && threadIdx.x == 0) atomicOr(flags, QSA_FLAG_NBLOCKS_CLAMPED);
        n = n < 0 ? 0 : bound;
    }
    return n;
}

// n <= k: every block is selected, in order, then -1.
__device__ __forceinline__ void emit_all(int n, int k, int32_t *out) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
}

// Load keys of row[0, n) in the register layout: round r, thread t, component e
// holds position r*NT*4 + t*4 + e.  float4 loads when the row is 16-byte aligned.
template <int NT, int R>
__device__ __forceinline__ uint32_t load_row_keys(const float *row, int n, uint32_t (&keys)[R * 4]) {
    uint32_t valid = 0;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int p = r * NT * 4 + (int)threadIdx.x * 4;
        if (vec && p + 3 < n) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(row + p));
            keys[r * 4 + 0] = score_key(v.x);
            keys[r * 4 + 1] = score_key(v.y);
            keys[r * 4 + 2] = score_key(v.z);
            keys[r * 4 + 3] = score_key(v.w);
            valid |= 0xfu << (r * 4);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (p + e < n) {
                    keys[r * 4 + e] = score_key(__ldcs(row + p + e));
                    valid |= 1u << (r * 4 + e);
                } else {
                    keys[r * 4 + e] = 0u;
                }
            }
        }
    }
    return valid;
}

template <int NT, int R>
__device__ __forceinline__ void row_ids(int base, int32_t (&ids)[R * 4]) {
#pragma unroll
    for (int i = 0; i < R * 4; ++i) ids[i] = base + (i / 4) * NT * 4 + (int)threadIdx.x * 4 + (i % 4);
}

// ---------------------------------------------------------------------------- register

template <int NT, int R>
__global__ void __launch_bounds__(NT) topk_register_kernel(TopkArgs a) {
    __shared__ BlockScratch sm;
    const int q = blockIdx.x;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, a.flags);
    int32_t *out = a.ids + (size_t)q * a.k;
    if (n <= a.k) {
        emit_all(n, a.k, out);
        return;
    }
    if (n > NT * 4 * R) {   // cannot happen: the host sizes R from the bound
        if (threadIdx.x == 0) atomicOr(a.flags, QSA_FLAG_INTERNAL);
        emit_all(0, a.k, out);
        return;
    }
    uint32_t keys[R * 4];
    int32_t ids[R * 4];
    const uint32_t valid = load_row_keys<NT, R>(a.scores + (size_t)q * a.stride, n, keys);
    row_ids<NT, R>(0, ids);
    const Threshold th = radix_threshold<NT, R * 4>(keys, valid, a.k, sm);
    int gb = 0, eb = 0;
    ordered_emit<NT, R, 4>(keys, ids, valid, th,
                           [&](int slot, uint32_t, int32_t id) { if (slot < k) out[slot] = id; }, sm, gb, eb);
}

// ---------------------------------------------------------------------------- sample

template <int NT, int R>
__global__ void __launch_bounds__(NT) topk_sample_kernel(TopkArgs a) {
    constexpr int RC = kSampleCap / NT;          // candidate rounds per thread
    constexpr int kMaxSamples = NT * 4 * R / 32;
    __shared__ BlockScratch sm;
    __shared__ uint32_t cand_key[kSampleCap];
    __shared__ int32_t cand_id[kSampleCap];
    __shared__ uint32_t samples[kMaxSamples];
    const int q = blockIdx.x;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, a.flags);
    int32_t *out = a.ids + (size_t)q * k;
    if (n <= k) {
        emit_all(n, k, out);
        if (threadIdx.x == 0) a.qflags[q] = 0u;
        return;
    }
    if (n > NT * 4 * R) {
        if (threadIdx.x == 0) a.qflags[q] = 1u;
        return;
    }
    uint32_t keys[R * 4];
    int32_t ids[R * 4];
    const uint32_t valid = load_row_keys<NT, R>(a.scores + (size_t)q * a.stride, n, keys);
    row_ids<NT, R>(0, ids);

    // 1. the bound: KS-th largest key among blocks 0, 32, 64, ...
    const int ns = (n + 31) / 32;
    const int KS = 2 * k / 32 + 16;
    if ((threadIdx.x & 7) == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (valid >> (r * 4) & 1u) samples[(r * NT * 4 + (int)threadIdx.x * 4) / 32] = keys[r * 4];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t lb = 0u;   // fewer samples than KS: every key is a candidate
        if (ns >= KS) {
            constexpr int SPL = (kMaxSamples + 31) / 32;
            uint32_t s[SPL];
#pragma unroll
            for (int j = 0; j < SPL; ++j) {
                const int idx = j * 32 + (int)threadIdx.x;
                s[j] = idx < ns ? samples[idx] : 0u;   // key 0 is below every finite score
            }
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t c = lb | (1u << bit);
                int cnt = 0;
#pragma unroll
                for (int j = 0; j < SPL; ++j) cnt += s[j] >= c;
                cnt = (int)__reduce_add_sync(kFull, (unsigned)cnt);
                if (cnt >= KS) lb = c;
            }
        }
        if (threadIdx.x == 0) sm.misc[4] = (int)lb;
    }
    __syncthreads();
    const uint32_t lb = (uint32_t)sm.misc[4];

    // 2. one pass over the row: keys >= LB go to shared memory, in block order
    int m = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        int c = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) c += (valid >> (r * 4 + e) & 1u) && keys[r * 4 + e] >= lb;
        int total;
        int pos = m + block_excl_scan<NT>(c, sm, total);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = r * 4 + e;
            if ((valid >> i & 1u) && keys[i] >= lb) {
                if (pos < kSampleCap) {
                    cand_key[pos] = keys[i];
                    cand_id[pos] = ids[i];
                }
                ++pos;
            }
        }
        m += total;
    }
    // 3./4. enough candidates and not too many: select among them; else flag
    if (m < k || m > kSampleCap) {
        if (threadIdx.x == 0) a.qflags[q] = 1u;
        return;
    }
    __syncthreads();
    uint32_t ck[RC];
    int32_t ci[RC];
    uint32_t cvalid = 0;
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        const int idx = r * NT + (int)threadIdx.x;
        if (idx < m) {
            ck[r] = cand_key[idx];
            ci[r] = cand_id[idx];
            cvalid |= 1u << r;
        } else {
            ck[r] = 0u;
            ci[r] = -1;
        }
    }
    const Threshold th = radix_threshold<NT, RC>(ck, cvalid, k, sm);
    int gb = 0, eb = 0;
    ordered_emit<NT, RC, 1>(ck, ci, cvalid, th,
                            [&](int slot, uint32_t, int32_t id) { if (slot < k) out[slot] = id; }, sm, gb, eb);
    if (threadIdx.x == 0) a.qflags[q] = 0u;
}

// ---------------------------------------------------------------------------- radix

template <int NT>
__global__ void __launch_bounds__(NT) topk_radix_kernel(TopkArgs a, int flagged_only) {
    __shared__ BlockScratch sm;
    const int q = blockIdx.x;
    if (flagged_only && a.qflags[q] == 0u) return;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, flagged_only ? nullptr : a.flags);
    int32_t *out = a.ids + (size_t)q * k;
    if (n <= k) {
        emit_all(n, k, out);
        return;
    }
    const float *row = a.scores + (size_t)q * a.stride;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int TILE = NT * 4;
    uint32_t prefix = 0u;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += NT) sm.hist[i] = 0u;
        __syncthreads();
        for (int base = 0; base < n; base += TILE) {
            uint32_t keys[4];
            const uint32_t valid = load_row_keys<NT, 1>(row + base, n - base, keys);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool match = (valid >> e & 1u) &&
                                   (shift == 24 || (keys[e] >> (shift + 8)) == (prefix >> (shift + 8)));
                const uint32_t d = match ? (keys[e] >> shift) & 0xffu : 0xffffffffu;
                const unsigned peers = __match_any_sync(kFull, d);
                if (match && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[d], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        if (wid == 0) {
            uint32_t c[8];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = sm.hist[255 - 8 * lane - j];
                sum += (int)c[j];
            }
            const int incl = warp_incl_scan(sum);
            int run = incl - sum;
            if (run < remaining && remaining <= incl) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + (int)c[j] >= remaining) {
                        sm.misc[0] = 255 - 8 * lane - j;
                        sm.misc[1] = run;
                        break;
                    }
                    run += (int)c[j];
                }
            }
        }
        __syncthreads();
        remaining -= sm.misc[1];
        prefix |= (uint32_t)sm.misc[0] << shift;
        __syncthreads();
    }
    Threshold th;
    th.T = prefix;
    th.above = k - remaining;
    th.budget = remaining;
    int gb = 0, eb = 0;
    for (int base = 0; base < n; base += TILE) {
        uint32_t keys[4];
        int32_t ids[4];
        const uint32_t valid = load_row_keys<NT, 1>(row + base, n - base, keys);
        row_ids<NT, 1>(base, ids);
        ordered_emit<NT, 1, 4>(keys, ids, valid, th,
                               [&](int slot, uint32_t, int32_t id) { if (slot < k) out[slot] = id; }, sm, gb, eb);
    }
}

// ---------------------------------------------------------------------------- split

template <int NT, int RB>
__global__ void __launch_bounds__(NT) topk_split_kernel(TopkArgs a, int chunk_len) {
    __shared__ BlockScratch sm;
    __shared__ int s_last;
    const int q = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, c == 0 ? a.flags : nullptr);
    const size_t slot0 = ((size_t)q * a.maxch + c) * k;
    uint32_t *ck = a.ckeys + slot0;
    int32_t *ci = a.cids + slot0;

    // stage A: this chunk's candidates, in block order
    if (n > k) {
        const int lo = c * chunk_len;
        const int len = max(0, min(chunk_len, n - lo));
        const float *row = a.scores + (size_t)q * a.stride + lo;
        if (len <= k) {
            for (int i = threadIdx.x; i < len; i += NT) {
                ck[i] = score_key(__ldcs(row + i));
                ci[i] = lo + i;
            }
        } else {
            uint32_t keys[4];
            int32_t ids[4];
            const uint32_t valid = load_row_keys<NT, 1>(row, len, keys);
            row_ids<NT, 1>(lo, ids);
            const Threshold th = radix_threshold<NT, 4>(keys, valid, k, sm);
            int gb = 0, eb = 0;
            ordered_emit<NT, 1, 4>(keys, ids, valid, th,
                                   [&](int slot, uint32_t key, int32_t id) {
                                       if (slot < k) {
                                           ck[slot] = key;
                                           ci[slot] = id;
                                       }
                                   },
                                   sm, gb, eb);
        }
        if (threadIdx.x == 0) a.counts[(size_t)q * a.maxch + c] = min(len, k);
    }
    // last CTA of the query to arrive runs stage B; no CTA waits for another
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&a.tickets[q], 1u);
        s_last = (t == (unsigned)nch - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    int32_t *out = a.ids + (size_t)q * k;
    if (n <= k) {
        emit_all(n, k, out);
    } else {
        // slots c*k + j of every chunk, chunk-major: block order
        uint32_t keys[RB];
        int32_t ids[RB];
        uint32_t valid = 0;
        const uint32_t *qk = a.ckeys + (size_t)q * a.maxch * k;
        const int32_t *qi = a.cids + (size_t)q * a.maxch * k;
        const int32_t *qc = a.counts + (size_t)q * a.maxch;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int s = r * NT + (int)threadIdx.x;
            const int cc = s / k, j = s - cc * k;
            keys[r] = 0u;
            ids[r] = -1;
            if (cc < nch && j < __ldcg(qc + cc)) {
                keys[r] = __ldcg(qk + s);
                ids[r] = __ldcg(qi + s);
                valid |= 1u << r;
            }
        }
        const Threshold th = radix_threshold<NT, RB>(keys, valid, k, sm);
        int gb = 0, eb = 0;
        ordered_emit<NT, RB, 1>(keys, ids, valid, th,
                                [&](int slot, uint32_t, int32_t id) { if (slot < k) out[slot] = id; }, sm, gb, eb);
    }
    if (threadIdx.x == 0) a.tickets[q] = 0u;
}

// ---------------------------------------------------------------------------- launchers

qsa_status launch_topk_register(const TopkArgs &a, cudaStream_t s) {
    if (a.bound <= 1024) {
        topk_register_kernel<256, 1><<<a.nq, 256, 0, s>>>(a);
    } else if (a.bound <= 4096) {
        topk_register_kernel<1024, 1><<<a.nq, 1024, 0, s>>>(a);
    } else if (a.bound <= kRegisterCap) {
        topk_register_kernel<1024, 2><<<a.nq, 1024, 0, s>>>(a);
    } else {
        return fail(QSA_ERR_UNSUPPORTED, "register path holds at most %d blocks per row (bound %d)",
                    kRegisterCap, a.bound);
    }
    return check_cuda(cudaGetLastError(), "topk_register_kernel launch");
}

qsa_status launch_topk_radix(const TopkArgs &a, bool flagged_only, cudaStream_t s) {
    topk_radix_kernel<512><<<a.nq, 512, 0, s>>>(a, flagged_only ? 1 : 0);
    return check_cuda(cudaGetLastError(), "topk_radix_kernel launch");
}

qsa_status launch_topk_sample(const TopkArgs &a, cudaStream_t s) {
    if (a.bound <= 4096) {
        topk_sample_kernel<1024, 1><<<a.nq, 1024, 0, s>>>(a);
    } else {
        topk_sample_kernel<1024, 2><<<a.nq, 1024, 0, s>>>(a);
    }
    qsa_status st = check_cuda(cudaGetLastError(), "topk_sample_kernel launch");
    if (st != QSA_OK) return st;
    return launch_topk_radix(a, true, s);
}

SplitGeom split_geometry(int bound, int nq, int k, int maxch) {
    SplitGeom g{0, 0};
    if (bound <= 0 || nq <= 0) return g;
    const int target_ctas = 2 * num_sms();
    const int per_query = std::max(1, target_ctas / nq);
    int len = (bound + per_query - 1) / per_query;
    len = std::max(len, std::max(kMinChunk, 2 * k));
    len = (len + 3) / 4 * 4;
    int nch = (bound + len - 1) / len;
    while ((long)nch * k > kSplitSlots && len <= kSplitMaxChunk) {
        len *= 2;
        nch = (bound + len - 1) / len;
    }
    if (len > kSplitMaxChunk || (long)nch * k > kSplitSlots || nch > maxch) return g;
    g.chunk_len = len;
    g.nchunks = nch;
    return g;
}

qsa_status launch_topk_split(const TopkArgs &a, const SplitGeom &g, cudaStream_t s) {
    if (g.chunk_len <= 0 || g.chunk_len > kSplitMaxChunk)
        return fail(QSA_ERR_UNSUPPORTED, "split path: no chunk geometry fits (bound %d, k %d)",
                    a.bound, a.k);
    dim3 grid(g.nchunks, a.nq);
    topk_split_kernel<256, kSplitSlots / 256><<<grid, 256, 0, s>>>(a, g.chunk_len);
    return check_cuda(cudaGetLastError(), "topk_split_kernel launch");
}

}  // namespace qsa
