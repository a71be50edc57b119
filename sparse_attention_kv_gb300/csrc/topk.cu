// topk.cu -- block top-k kernels over fp32 score rows.
//
// Five paths, all giving the ids of the rule in qsa_device.cuh.  Every kernel is
// launched as a programmatic dependent of the kernel before it on the stream and
// waits at entry until that kernel has completed (in a chained select its CTAs
// take SMs while the scorer drains).
//  * warp:     k <= 32, rows of up to 8,192 blocks: one CTA per query holds its
//    row in registers (one warp per 1,024-block chunk), bounds the k-th largest
//    score from below with maxima of the whole row, keeps the few scores at or
//    above the bound and ranks them exactly; heavy ties take a per-chunk select
//    and a merge of the chunks' lists (warp_topk.cuh).  The AUTO choice wherever
//    it applies.
//  * register: one CTA per query holds its whole row in registers (<= 8,192
//    blocks: 256 threads x 32) and selects with no re-read -- the "register
//    kernel" the pages name for contexts within its reach (Strata PR #3987,
//    "Problem and result").
//  * sample:   the same kernel with the one-read candidate filter of "#2093 sm_75:
//    the prompt path's top-k with one full read of the scores" (steps 1-4): a
//    lower bound LB = the KS-th largest key among blocks 0, 32, 64, ...
//    (KS = 2k/32 + 16); the blocks with score >= LB go to shared memory; with at
//    least k and at most 4,096 of them the threshold, "above" and the tie budget
//    over the candidates are the row's.  Otherwise the query falls back -- here
//    to a select over the row it already holds on chip, with no second read.
//  * radix:    one CTA per query, multi-pass radix select straight from global
//    memory (four digit passes and the emit); any row length.
//  * split:    stage A, one CTA per (query, chunk), keeps the chunk's top-k
//    candidates in the workspace; the last CTA of a query to finish (atomic
//    ticket, nothing waits) runs stage B over the candidates.  A query's
//    selection restricted to a chunk is a prefix of that chunk's order, so every
//    selected block is among its chunk's candidates (Strata PR #3987,
//    "Approach").
#include <algorithm>
#include <cstddef>
#include <cstdio>
#include <mutex>

#include "qsa_device.cuh"
#include "qsa_internal.h"
#include "warp_topk.cuh"

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

// ---------------------------------------------------------------------------- register / sample

constexpr int kNT = 256;   // threads of the register, sample and split kernels

__device__ __forceinline__ float nan_pad() { return __int_as_float(0x7fffffff); }

// Row values striped over the block: round r, thread t, component e holds
// position r*kNT*4 + t*4 + e.  Positions at or past n read as NaN, which no
// comparison selects.  float4 streaming loads when the row is 16-byte aligned.
template <int R>
__device__ __forceinline__ void load_row_vals(const float *row, int n, float (&x)[R * 4]) {
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int p = r * kNT * 4 + (int)threadIdx.x * 4;
        if (vec && p + 3 < n) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(row + p));
            x[r * 4 + 0] = v.x;
            x[r * 4 + 1] = v.y;
            x[r * 4 + 2] = v.z;
            x[r * 4 + 3] = v.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) x[r * 4 + e] = p + e < n ? __ldcs(row + p + e) : nan_pad();
        }
    }
}

__device__ __forceinline__ int striped_id(int i) { return (i >> 2) * kNT * 4 + (int)threadIdx.x * 4 + (i & 3); }

struct __align__(16) RowSmem {
    CandSmem<kNT> cs;
    // sample path: candidate scores in cand[0, 4096), their ids in cand[4096, 8192);
    // whole-row select: every score of the row, in block order (ids implicit)
    uint32_t cand[kRegisterCap];
    int32_t sel[1024];
};

template <int R, bool SAMPLE>
__global__ void __launch_bounds__(kNT, 2) topk_row_kernel(TopkArgs a) {
    wait_prior_grid();   // the scores may come from the kernel launched just before
    allow_dependent_launch();   // a consumer of the ids (the attention) may launch and wait
    constexpr int KPT = R * 4;
    static_assert(2 * kSampleCap == kRegisterCap, "candidate scores and ids share cand[]");
    __shared__ RowSmem sm;
    float *cval = reinterpret_cast<float *>(sm.cand);
    int32_t *cid = reinterpret_cast<int32_t *>(sm.cand + kSampleCap);
    const int q = blockIdx.x;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, a.flags);
    int32_t *out = a.ids + (size_t)q * k;
    if (n <= k) {
        emit_all(n, k, out);
        return;
    }
    if (n > kNT * KPT) {   // cannot happen: the host sizes R from the bound
        if (threadIdx.x == 0) atomicOr(a.flags, QSA_FLAG_INTERNAL);
        emit_all(0, k, out);
        return;
    }
    const float *row = a.scores + (size_t)q * a.stride;
    cand_smem_init(sm.cs);
    const int ns = (n + 31) / 32;
    const int KS = 2 * k / 32 + 16;
    const bool sampled = SAMPLE && ns >= KS;   // fewer samples than KS: every block is a candidate
    // 1. warp 0 reads the samples (blocks 0, 32, 64, ...) before the row, so the
    //    bound is computed while the rest of the row is still arriving
    uint32_t skey[8];
    if (sampled && threadIdx.x < 32) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = (int)threadIdx.x + 32 * e;
            skey[e] = j < ns ? score_key(__ldg(row + 32 * j)) : 0u;
        }
    }
    float x[KPT];
    load_row_vals<R>(row, n, x);
    if (sampled && threadIdx.x < 32) {
        const uint32_t lbk = warp_kth_largest(skey, KS);
        if (threadIdx.x == 0) sm.cs.misc[4] = (int)lbk;
    }
    __syncthreads();
    const float lb = sampled ? key_float((uint32_t)sm.cs.misc[4]) : -__int_as_float(0x7f800000);

    bool done = false;
    if (SAMPLE || n <= kSampleCap) {
        // 2. one pass over the row held on chip: blocks with score >= LB become
        //    candidates (score, id) in shared memory, in any order
        int c = 0;
        float tmax = -__int_as_float(0x7f800000);
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            c += x[i] >= lb;
            tmax = fmaxf(tmax, x[i]);
        }
        int pos = warp_append(c, &sm.cs.cnt[2]);
#pragma unroll
        for (int i = 0; i < KPT; ++i)
            if (x[i] >= lb) {
                if (pos < kSampleCap) {
                    cval[pos] = x[i];
                    cid[pos] = striped_id(i);
                }
                ++pos;
            }
        uint32_t mn = score_key(lb), mx = score_key(tmax);
        block_minmax<kNT>(mn, mx, sm.cs);
        const int m = sm.cs.cnt[2];
        if (m >= k && m <= kSampleCap) {
            // 3. at least k candidates: the threshold, "above" and the tie budget
            //    over the candidates are the row's
            const Threshold th = smem_threshold<kNT>(
                [&](int i, uint32_t &key) {
                    key = score_key(cval[i]);
                    return true;
                },
                m, k, mn, mx, sm.cs);
            collect_smem<kNT>([&](int i) { return score_key(cval[i]); }, [&](int i) { return cid[i]; }, m, th,
                              nullptr, sm.sel, sm.cs);
            done = true;
        } else if (SAMPLE && threadIdx.x == 0) {
            atomicOr(a.flags, QSA_FLAG_SAMPLE_FALLBACK);
        }
    }
    if (!done) {
        // 4. select over the whole row, still on chip: its scores go to shared
        //    memory in block order
        __syncthreads();   // candidate lists are dead
        float *rowv = reinterpret_cast<float *>(sm.cand);
        uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            if (x[i] == x[i]) {   // not a padding NaN
                const uint32_t key = score_key(x[i]);
                mn = min(mn, key);
                mx = max(mx, key);
                rowv[striped_id(i)] = x[i];
            }
        }
        if (threadIdx.x < 4) sm.cs.cnt[threadIdx.x] = 0;
        block_minmax<kNT>(mn, mx, sm.cs);
        const Threshold th = smem_threshold<kNT>(
            [&](int i, uint32_t &key) {
                key = score_key(rowv[i]);
                return true;
            },
            n, k, mn, mx, sm.cs);
        collect_smem<kNT>([&](int i) { return score_key(rowv[i]); }, [&](int i) { return i; }, n, th, nullptr,
                          sm.sel, sm.cs);
    }
    sort_emit<kNT>(sm.sel, k, k, out);
}

// ---------------------------------------------------------------------------- radix

template <int NT>
__global__ void __launch_bounds__(NT) topk_radix_kernel(TopkArgs a, int flagged_only) {
    wait_prior_grid();   // the scores may come from the kernel launched just before
    allow_dependent_launch();   // a consumer of the ids (the attention) may launch and wait
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

struct __align__(16) SplitSmem {
    CandSmem<kNT> cs;
    uint32_t ck[kSplitSlots];
    int32_t cid[kSplitSlots];
    uint32_t skey[1024];
    int32_t sid[1024];
    int last;
};

__global__ void __launch_bounds__(kNT, 2) topk_split_kernel(TopkArgs a, int chunk_len) {
    wait_prior_grid();   // the scores may come from the kernel launched just before
    allow_dependent_launch();   // a consumer of the ids (the attention) may launch and wait
    __shared__ SplitSmem sm;
    const int q = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int k = a.k;
    const int n = clamp_blocks(a.n_blocks, q, a.bound, c == 0 ? a.flags : nullptr);
    const size_t slot0 = ((size_t)q * a.maxch + c) * k;
    uint32_t *ck = a.ckeys + slot0;
    int32_t *ci = a.cids + slot0;

    // stage A: this chunk's k candidates (key, id), any order
    if (n > k) {
        const int lo = c * chunk_len;
        const int len = max(0, min(chunk_len, n - lo));
        const float *row = a.scores + (size_t)q * a.stride + lo;
        if (len <= k) {
            for (int i = threadIdx.x; i < len; i += kNT) {
                ck[i] = score_key(__ldcs(row + i));
                ci[i] = lo + i;
            }
        } else {
            cand_smem_init(sm.cs);
            uint32_t mn = 0xffffffffu, mx = 0u;
            for (int i = threadIdx.x; i < len; i += kNT) {
                const uint32_t key = score_key(__ldcs(row + i));
                sm.ck[i] = key;
                mn = min(mn, key);
                mx = max(mx, key);
            }
            block_minmax<kNT>(mn, mx, sm.cs);
            const Threshold th = smem_threshold<kNT>(
                [&](int i, uint32_t &key) {
                    key = sm.ck[i];
                    return true;
                },
                len, k, mn, mx, sm.cs);
            collect_smem<kNT>([&](int i) { return sm.ck[i]; }, [&](int i) { return lo + i; }, len, th, sm.skey,
                              sm.sid, sm.cs);
            for (int i = threadIdx.x; i < k; i += kNT) {
                ck[i] = sm.skey[i];
                ci[i] = sm.sid[i];
            }
        }
        if (threadIdx.x == 0) a.counts[(size_t)q * a.maxch + c] = min(len, k);
    }
    // the last CTA of the query to arrive runs stage B; no CTA waits for another
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(&a.tickets[q], 1u);
        sm.last = (t == (unsigned)nch - 1u);
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    int32_t *out = a.ids + (size_t)q * k;
    if (n <= k) {
        emit_all(n, k, out);
    } else {
        cand_smem_init(sm.cs);
        __syncthreads();
        const uint32_t *qk = a.ckeys + (size_t)q * a.maxch * k;
        const int32_t *qi = a.cids + (size_t)q * a.maxch * k;
        const int32_t *qc = a.counts + (size_t)q * a.maxch;
        const int slots = nch * k;
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (int base = 0; base < slots; base += kNT) {
            const int s = base + (int)threadIdx.x;
            const int cc = s / k;
            const bool v = s < slots && (s - cc * k) < __ldcg(qc + cc);
            const int pos = warp_append(v ? 1 : 0, &sm.cs.cnt[2]);
            if (v) {
                const uint32_t key = __ldcg(qk + s);
                sm.ck[pos] = key;
                sm.cid[pos] = __ldcg(qi + s);
                mn = min(mn, key);
                mx = max(mx, key);
            }
        }
        block_minmax<kNT>(mn, mx, sm.cs);
        const int m = sm.cs.cnt[2];
        const Threshold th = smem_threshold<kNT>(
            [&](int i, uint32_t &key) {
                key = sm.ck[i];
                return true;
            },
            m, k, mn, mx, sm.cs);
        collect_smem<kNT>([&](int i) { return sm.ck[i]; }, [&](int i) { return sm.cid[i]; }, m, th, nullptr,
                          sm.sid, sm.cs);
        sort_emit<kNT>(sm.sid, k, k, out);
    }
    if (threadIdx.x == 0) a.tickets[q] = 0u;
}

// ---------------------------------------------------------------------------- warp path
//
// k <= 32, rows of up to NW * 1,024 blocks, one CTA of NW warps per query.  Warp
// w holds blocks [1024 w, 1024 (w + 1)) of the row in registers (one read of
// HBM): lane l the entries 1024 w + 4 (l + 32 t) + c, t < 8, c < 4.
//
// Row bound.  Each lane takes the largest of its 32 scores.  Each warp whose
// chunk fills all 32 lanes takes the r-th largest of its lane maxima, r =
// ceil(k / such warps), and the row bound B is the smallest of those: every such
// warp has r lanes whose maxima (distinct entries) reach B, so at least k
// entries of the row score >= B and every selected block is among them.  On
// continuous scores B sits a little below the row's k-th largest score (about
// 50 entries reach it at 8,125 blocks and k = 32), so one compare per score
// keeps the survivors.  They go to shared memory packed as (key, ~id) -- a
// total order that is exactly the selection order -- and are ranked exactly
// (a few threads per survivor); the k of rank below k are the selection,
// emitted in ascending id order.  This is the one-read candidate filter of
// "#2093 sm_75: the prompt path's top-k with one full read of the scores"
// (steps 2-3) with the bound drawn from maxima of the whole row rather than a
// 1-in-32 sample, so "at least k candidates" holds by construction.
//
// More survivors than the on-chip list holds (heavy ties) take the per-chunk
// path below, which rows of at most one chunk take directly (their bound from
// the lanes' top-2 keys is the tighter one there).

constexpr int kWarpChunk = 1024;   // blocks per warp (CL); 512-block chunks measured slower even for 3 queries
constexpr int kRowCap = 256;       // survivors of the row bound held on chip
constexpr size_t kWarpTwoPerSmBytes = 90 * 1024;   // dynamic shared memory that leaves room for two CTAs per SM

// v[b] for a runtime b < N (N a power of two) without indexing registers: a tree of
// selects on the bits of b.
template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int b) {
    static_assert((N & (N - 1)) == 0 && N >= 2, "power of two");
    float y[N / 2];
#pragma unroll
    for (int j = 0; j < N / 2; ++j) y[j] = (b & 1) ? v[2 * j + 1] : v[2 * j];
    if constexpr (N == 2) {
        return y[0];
    } else {
        return pick<N / 2>(y, b >> 1);
    }
}

template <int NW>
struct __align__(16) WarpPathSmem {
    uint32_t scratch[NW][256];   // per-chunk path: per warp candidates / histogram
    uint64_t lists[NW * 32];     // per-chunk path: each chunk's top k, descending
    uint64_t cand[kRowCap];      // row-bound survivors, packed
    __align__(16) int32_t sel[32];   // selected ids by rank (read as int4)
    uint32_t wbound[8];          // each full warp's r-th largest lane-maximum key
    int cnt;                     // survivors
};

// The per-chunk path.  Warp w bounds its chunk's k-th largest key from below with
// the k-th largest of the lanes' top-2 keys, keeps the entries at or above it (a
// few more than k on continuous scores) and ranks them exactly: its chunk's top
// k, descending, in shared memory.  The chunks' lists are then merged by exact
// ranks (one thread per candidate, binary searches in the other lists).  A
// query's selection restricted to a chunk is a prefix of that chunk's order, so
// every selected block is among its chunk's k (the split of Strata PR #3987,
// section "Approach").  Heavy ties (more than 64 entries at a chunk's bound)
// take the radix warp select for that chunk.  Every thread of the CTA calls it.
template <int NW, int CL>
__device__ __noinline__ void warp_chunk_select(const float *row, int n, int k, int32_t *out, WarpPathSmem<NW> &sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *h = sm.scratch[warp];
    uint64_t *buf = reinterpret_cast<uint64_t *>(h);
    for (int i = lane; i < 256; i += 32) h[i] = 0u;
    __syncwarp();
    const int lo = warp * CL;
    const int len = min(CL, n - lo);
    uint64_t *dst = sm.lists + warp * k;
    if (len > k) {
        const float *r = row + lo;
        const float4 *r4 = reinterpret_cast<const float4 *>(r);
        const bool vec = (reinterpret_cast<uintptr_t>(r) & 15u) == 0;
        auto load1 = [&](int i) { return __ldg(r + i); };   // the few entries that reach the bound, again
        const bool ok =
            vec && len == CL
                ? warp_top_regs<CL / 128, true>([&](int v) { return __ldg(r4 + v); }, load1, len, k, lo, buf, dst)
                : warp_top_regs<CL / 128>(
                      [&](int v) {
                          if (vec && 4 * v + 3 < len) return __ldg(r4 + v);
                          float e[4];
#pragma unroll
                          for (int c = 0; c < 4; ++c) e[c] = 4 * v + c < len ? __ldg(r + 4 * v + c) : 0.0f;
                          return make_float4(e[0], e[1], e[2], e[3]);
                      },
                      load1, len, k, lo, buf, dst);
        if (!ok) {
            for (int i = lane; i < 256; i += 32) h[i] = 0u;
            __syncwarp();
            warp_select([&](int i) { return score_key(__ldg(r + i)); }, len, k, h,
                        [&](int pos, int i) { dst[pos] = pack_cand(score_key(__ldg(r + i)), lo + i); });
            __syncwarp();
            uint64_t v = lane < k ? ~dst[lane] : ~0ull;   // descending, like the other chunks
            __syncwarp();
            warp_sort32_asc(v);
            if (lane < k) dst[lane] = ~v;
        }
    } else if (len > 0) {
        uint64_t v = lane < len ? ~pack_cand(score_key(__ldg(row + lo + lane)), lo + lane) : ~0ull;
        warp_sort32_asc(v);
        if (lane < len) dst[lane] = ~v;
    }
    __syncthreads();
    // Merge: every chunk's list is descending, so a candidate's rank in the whole row
    // is its index in its own list plus, for every other list, the number of entries
    // above it (a binary search); packed values are distinct, so the ranks are a
    // permutation and exactly k candidates rank below k.  One thread per candidate.
    const int nch = (n + CL - 1) / CL;
    auto cnt_of = [&](int c) { return c < nch ? min(k, n - c * CL) : 0; };
    if (lane < cnt_of(warp)) {
        const uint64_t x = sm.lists[warp * k + lane];
        int rank = lane;
#pragma unroll
        for (int b = 0; b < NW; ++b) {
            if (b == warp) continue;
            const int cb = cnt_of(b);
            const uint64_t *lb = sm.lists + b * k;
            int pos = 0;   // entries of list b above x
#pragma unroll
            for (int step = 32; step >= 1; step >>= 1)
                if (pos + step <= cb && lb[pos + step - 1] > x) pos += step;
            rank += pos;
        }
        if (rank < k) sm.sel[rank] = cand_id(x);
    }
    __syncthreads();
    if (warp != 0) return;
    if (lane < k) {   // ascending ids: each id's slot is the number of selected ids below it
        const int32_t id = sm.sel[lane];
        int below = 0;
        for (int t = 0; t < k; ++t) below += sm.sel[t] < id;
        out[below] = id;
    }
}

template <int NW, int CL>
__global__ void __launch_bounds__(NW * 32, 2) topk_warp_kernel(TopkArgs a) {
    wait_prior_grid();   // the scores may come from the kernel launched just before
    allow_dependent_launch();   // a consumer of the ids (the attention) may launch and wait
    static_assert(NW <= 8 && offsetof(WarpPathSmem<NW>, sel) % 16 == 0, "sel is read as int4");
    __shared__ WarpPathSmem<NW> sm;
    const int q = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = a.k;
    int32_t *out = a.ids + (size_t)q * k;
    const float *row = a.scores + (size_t)q * a.stride;
    if constexpr (NW == 1) {
        const int n = clamp_blocks(a.n_blocks, q, a.bound, a.flags);
        if (n <= k) {
            emit_all(n, k, out);
            return;
        }
        warp_chunk_select<NW, CL>(row, n, k, out, sm);
    } else {
        constexpr int NV = CL / 128;   // float4 loads per lane
        constexpr int NT = NW * 32;
        const float kNegInf = __int_as_float(0xff800000);
        // 1. this warp's chunk into registers.  Every entry below the host-visible bound
        //    lies in the caller's row (stride >= bound), so the loads go out together
        //    with the load of n_blocks[q] instead of after it; entries at or past n are
        //    then set to -inf.
        const int lo = warp * CL;
        const int cap = max(0, min(CL, a.bound - lo));
        const float *r = row + lo;
        const float4 *r4 = reinterpret_cast<const float4 *>(r);
        const bool vec = (reinterpret_cast<uintptr_t>(r) & 15u) == 0;
        float x[4 * NV];
        if (vec && cap == CL) {
#pragma unroll
            for (int t = 0; t < NV; ++t) {
                const float4 f = __ldg(r4 + lane + 32 * t);
                x[4 * t + 0] = f.x;
                x[4 * t + 1] = f.y;
                x[4 * t + 2] = f.z;
                x[4 * t + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int t = 0; t < NV; ++t) {
                const int v = lane + 32 * t;
                if (vec && 4 * v + 3 < cap) {
                    const float4 f = __ldg(r4 + v);
                    x[4 * t + 0] = f.x;
                    x[4 * t + 1] = f.y;
                    x[4 * t + 2] = f.z;
                    x[4 * t + 3] = f.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) x[4 * t + c] = 4 * v + c < cap ? __ldg(r + 4 * v + c) : kNegInf;
                }
            }
        }
        const int n = clamp_blocks(a.n_blocks, q, a.bound, a.flags);
        if (n <= k) {
            emit_all(n, k, out);
            return;
        }
        const int len = max(0, min(CL, n - lo));
        if (len < cap) {
#pragma unroll
            for (int t = 0; t < NV; ++t)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (4 * (lane + 32 * t) + c >= len) x[4 * t + c] = kNegInf;
        }
        float m4[NV];
#pragma unroll
        for (int t = 0; t < NV; ++t) m4[t] = fmaxf(fmaxf(x[4 * t], x[4 * t + 1]), fmaxf(x[4 * t + 2], x[4 * t + 3]));
#pragma unroll
        for (int s = 1; s < NV; s <<= 1)
#pragma unroll
            for (int t = 0; t + s < NV; t += 2 * s) m4[t] = fmaxf(m4[t], m4[t + s]);
        const float mx = m4[0];
        // 2. the row bound: warps whose chunk holds >= 128 entries have an entry on every
        //    lane; each takes the r-th largest of its lanes' maxima
        const int nfull = n >= 128 ? min(NW, (n - 128) / CL + 1) : 0;
        if (warp < nfull) {
            const int r_th = (k + nfull - 1) / nfull;
            uint32_t kk = score_key(mx), res = 0u;
            for (int it = 0; it < r_th; ++it) {
                res = __reduce_max_sync(kFull, kk);
                const unsigned win = __ballot_sync(kFull, kk == res);
                if (lane == __ffs(win) - 1) kk = 0u;   // 0 is below every score's key
            }
            if (lane == 0) sm.wbound[warp] = res;
        }
        if (threadIdx.x == 0) sm.cnt = 0;
        __syncthreads();
        uint32_t wb[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) wb[w] = w < nfull ? sm.wbound[w] : 0xffffffffu;
#pragma unroll
        for (int s = 1; s < NW; s <<= 1)
#pragma unroll
            for (int w = 0; w + s < NW; w += 2 * s) wb[w] = min(wb[w], wb[w + s]);
        const uint32_t B = wb[0];
        // with no full warp (n < 128) every entry is a survivor; a bound of -inf (scores
        // of -inf) would also pass the padding, so then entries are tested against len
        const float Bf = nfull > 0 ? key_float(B) : kNegInf;
        const bool guard = !(Bf > kNegInf);
        // 3. survivors, the scores >= B: a bit per entry of the lane (no branches), a
        //    shared atomic for each lane that has any, then each such lane writes its few
        //    survivors, each value picked from the lane's registers by the bits of its
        //    position
        uint32_t sv[4] = {0u, 0u, 0u, 0u};   // four partial masks: short dependency chains
#pragma unroll
        for (int t = 0; t < NV; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (x[4 * t + c] >= Bf) sv[c] |= 1u << (4 * t + c);
        uint32_t surv = (sv[0] | sv[1]) | (sv[2] | sv[3]);
        if (guard) {
#pragma unroll
            for (int t = 0; t < NV; ++t)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (4 * (lane + 32 * t) + c >= len) surv &= ~(1u << (4 * t + c));
        }
        int pos = surv ? atomicAdd(&sm.cnt, __popc(surv)) : 0;
        while (surv) {
            const int bit = __ffs(surv) - 1;
            surv &= surv - 1u;
            const int i = 4 * (lane + 32 * (bit >> 2)) + (bit & 3);
            if (pos < kRowCap) sm.cand[pos] = pack_cand(score_key(pick<4 * NV>(x, bit)), lo + i);
            ++pos;
        }
        __syncthreads();
        const int m = sm.cnt;
        if (m >= k && m <= kRowCap) {
            // 4. exact ranks of the survivors; the k of rank below k are the selection
            rank_survivors<NT>(sm.cand, m, k, sm.sel);
            __syncthreads();
            if (warp == 0 && lane < k) {   // 5. the k ids, ascending: an id's slot is the number below it
                const int32_t id = sm.sel[lane];
                int below = 0;
                const int4 *s4 = reinterpret_cast<const int4 *>(sm.sel);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int4 v = s4[t];
                    below += (4 * t + 0 < k && v.x < id) + (4 * t + 1 < k && v.y < id) +
                             (4 * t + 2 < k && v.z < id) + (4 * t + 3 < k && v.w < id);
                }
                out[below] = id;
            }
            return;
        }
        // heavy ties: more survivors than the list holds
        warp_chunk_select<NW, CL>(row, n, k, out, sm);
    }
}

// ---------------------------------------------------------------------------- launchers

// Every top-k kernel is launched as a programmatic dependent of the kernel before it
// on the stream (the scorer, in a chained select): its CTAs may be scheduled while
// that kernel drains and wait at entry until it has completed.
template <typename... KArgs, typename... Args>
static qsa_status launch_dependent(const char *what, void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                                   size_t dyn_smem, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, kern, args...), what);
}

template <bool SAMPLE>
static qsa_status launch_row(const TopkArgs &a, cudaStream_t s) {
    const char *what = SAMPLE ? "topk_row_kernel<sample> launch" : "topk_row_kernel launch";
    const dim3 grid(a.nq), block(kNT);
    if (a.bound <= 1024) return launch_dependent(what, topk_row_kernel<1, SAMPLE>, grid, block, s, 0, a);
    if (a.bound <= 2048) return launch_dependent(what, topk_row_kernel<2, SAMPLE>, grid, block, s, 0, a);
    if (a.bound <= 4096) return launch_dependent(what, topk_row_kernel<4, SAMPLE>, grid, block, s, 0, a);
    if (a.bound <= kRegisterCap) return launch_dependent(what, topk_row_kernel<8, SAMPLE>, grid, block, s, 0, a);
    return fail(QSA_ERR_UNSUPPORTED, "%s path holds at most %d blocks per row (bound %d)",
                SAMPLE ? "sample" : "register", kRegisterCap, a.bound);
}

qsa_status launch_topk_register(const TopkArgs &a, cudaStream_t s) { return launch_row<false>(a, s); }

qsa_status launch_topk_sample(const TopkArgs &a, cudaStream_t s) { return launch_row<true>(a, s); }

qsa_status launch_topk_warp(const TopkArgs &a, bool behind_scorer, cudaStream_t s) {
    if (a.k > 32)
        return fail(QSA_ERR_UNSUPPORTED, "warp path takes k <= 32 (got %d)", a.k);
    if (a.bound > 8 * kWarpChunk)
        return fail(QSA_ERR_UNSUPPORTED, "warp path holds at most %d blocks per row (bound %d)", 8 * kWarpChunk,
                    a.bound);
    const char *what = "topk_warp_kernel launch";
    const dim3 grid(a.nq);
    if (a.bound <= kWarpChunk) return launch_dependent(what, topk_warp_kernel<1, kWarpChunk>, grid, dim3(32), s, 0, a);
    if (a.bound <= 2 * kWarpChunk)
        return launch_dependent(what, topk_warp_kernel<2, kWarpChunk>, grid, dim3(64), s, 0, a);
    if (a.bound <= 4 * kWarpChunk)
        return launch_dependent(what, topk_warp_kernel<4, kWarpChunk>, grid, dim3(128), s, 0, a);
    if (!behind_scorer) return launch_dependent(what, topk_warp_kernel<8, kWarpChunk>, grid, dim3(256), s, 0, a);
    // Behind the scorer, at most two of these 8-warp CTAs per SM (an otherwise unused
    // shared-memory reservation): the CTAs launched early wait on the SMs the scorer
    // leaves free, and three to such an SM make it finish last (deep prompt select
    // 26.9 us with three, 24.9 with two; the top-k alone prefers three, 12.4 us to 13.7).
    static std::mutex mu;
    static bool opted_in[64] = {false};
    int dev = 0;
    qsa_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != QSA_OK) return st;
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!opted_in[dev]) {
            st = check_cuda(cudaFuncSetAttribute(topk_warp_kernel<8, kWarpChunk>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWarpTwoPerSmBytes),
                            "cudaFuncSetAttribute(topk_warp_kernel)");
            if (st != QSA_OK) return st;
            opted_in[dev] = true;
        }
    }
    return launch_dependent(what, topk_warp_kernel<8, kWarpChunk>, grid, dim3(256), s, kWarpTwoPerSmBytes, a);
}

qsa_status launch_topk_radix(const TopkArgs &a, bool flagged_only, cudaStream_t s) {
    return launch_dependent("topk_radix_kernel launch", topk_radix_kernel<512>, dim3(a.nq), dim3(512), s, 0, a,
                            flagged_only ? 1 : 0);
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
        return fail(QSA_ERR_UNSUPPORTED, "split path: no chunk geometry fits (bound %d, k %d)", a.bound, a.k);
    return launch_dependent("topk_split_kernel launch", topk_split_kernel, dim3(g.nchunks, a.nq), dim3(kNT), s, 0, a,
                            g.chunk_len);
}

}  // namespace qsa
