// qsa_device.cuh -- block-wide building blocks of the block top-k.
//
// The selection rule is the one of "#2093 sm_75: the prompt path's top-k with
// one full read of the scores" (description, step 3): a threshold T = the k-th
// largest key, `above` = the keys strictly greater than T, and a tie budget
// k - above spent on the keys equal to T in block order; the selected cells are
// emitted in block order.  Each radix digit is picked by a parallel scan of its
// bins (Strata PR #3987, section "Approach", last bullet).
#pragma once

#include <cstdint>

namespace qsa {

constexpr unsigned kFull = 0xffffffffu;

// Order-preserving key of an fp32 score: unsigned order of the keys equals the
// float order of the scores, -0 and +0 give the same key.  NaN is not ordered.
__device__ __forceinline__ uint32_t score_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;                      // -0 -> +0
    return u ^ ((u & 0x80000000u) ? 0xffffffffu : 0x80000000u);
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Shared scratch of the block-wide helpers.
struct BlockScratch {
    int warp_sums[32];
    uint32_t hist[256];
    uint32_t red[64];
    int misc[8];
};

// Exclusive scan of v over the NT threads of the block; *total receives the sum.
// Every thread of the block must call it (it holds three barriers).
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, BlockScratch &sm, int &total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = warp_incl_scan(v);
    if (lane == 31) sm.warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = lane < NW ? sm.warp_sums[lane] : 0;
        s = warp_incl_scan(s);
        if (lane < NW) sm.warp_sums[lane] = s;
    }
    __syncthreads();
    const int base = wid == 0 ? 0 : sm.warp_sums[wid - 1];
    total = sm.warp_sums[NW - 1];
    __syncthreads();
    return base + incl - v;
}

// Threshold of a top-k: T is the k-th largest key, above = #keys > T, budget = k - above.
struct Threshold {
    uint32_t T;
    int above;
    int budget;
};

// Radix select of the k-th largest of the valid keys held by the block.
// Each thread holds KPT keys; bit i of `valid` marks keys[i] valid.  Requires
// 1 <= k <= number of valid keys.  The bits that all valid keys share (the common
// prefix of the smallest and largest key) are skipped; the remaining bits are
// taken 8 at a time, most significant first: a 256-bin histogram of the digit
// among the keys that match the prefix so far (warp-aggregated shared atomics),
// then a warp scan of the bins from the top finds the bin holding the k-th key.
template <int NT, int KPT>
__device__ Threshold radix_threshold(const uint32_t (&keys)[KPT], uint32_t valid, int k,
                                     BlockScratch &sm) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    // block min / max of the valid keys
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if (valid >> i & 1u) {
            mn = min(mn, keys[i]);
            mx = max(mx, keys[i]);
        }
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    if (lane == 0) {
        sm.red[wid] = mn;
        sm.red[32 + wid] = mx;
    }
    __syncthreads();
    if (wid == 0) {
        uint32_t a = lane < NW ? sm.red[lane] : 0xffffffffu;
        uint32_t b = lane < NW ? sm.red[32 + lane] : 0u;
        a = __reduce_min_sync(kFull, a);
        b = __reduce_max_sync(kFull, b);
        if (lane == 0) {
            sm.misc[2] = (int)a;
            sm.misc[3] = (int)b;
        }
    }
    __syncthreads();
    mn = (uint32_t)sm.misc[2];
    mx = (uint32_t)sm.misc[3];
    int hi = 32 - __clz((int)(mn ^ mx));   // bits [0, hi) vary; 0 when all keys are equal
    uint32_t prefix = hi == 32 ? 0u : (mx & ~((1u << hi) - 1u));
    int remaining = k;
    while (hi > 0) {
        const int lo = hi > 8 ? hi - 8 : 0;
        const int nbins = 1 << (hi - lo);
        for (int i = threadIdx.x; i < nbins; i += NT) sm.hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            const bool match = (valid >> i & 1u) && (hi == 32 || (keys[i] >> hi) == (prefix >> hi));
            const uint32_t d = match ? (keys[i] >> lo) & (uint32_t)(nbins - 1) : 0xffffffffu;
            const unsigned peers = __match_any_sync(kFull, d);
            if (match && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[d], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (wid == 0) {
            // lane l owns bins nbins-1-8l-j, j = 0..7 (descending)
            uint32_t c[8];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int b = nbins - 1 - 8 * lane - j;
                c[j] = b >= 0 ? sm.hist[b] : 0u;
                sum += (int)c[j];
            }
            const int incl = warp_incl_scan(sum);
            int run = incl - sum;
            if (run < remaining && remaining <= incl) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + (int)c[j] >= remaining) {
                        sm.misc[0] = nbins - 1 - 8 * lane - j;
                        sm.misc[1] = run;
                        break;
                    }
                    run += (int)c[j];
                }
            }
        }
        __syncthreads();
        remaining -= sm.misc[1];
        prefix |= (uint32_t)sm.misc[0] << lo;
        hi = lo;
        __syncthreads();
    }
    Threshold t;
    t.T = prefix;
    t.above = k - remaining;
    t.budget = remaining;
    return t;
}

// Ordered emit.  The block's keys are laid out in R rounds of E consecutive
// elements per thread: element (r, e) of thread t comes at position
// r*NT*E + t*E + e of block order.  An element is selected when key > T, or
// key == T and fewer than `budget` equal keys precede it; it goes to slot
//   #(keys > T before it) + min(#(keys == T before it), budget)
// through sink(slot, key, id).  gt_base / eq_base carry the counts of earlier
// calls, so a row can be emitted tile by tile.
template <int NT, int R, int E, typename Sink>
__device__ void ordered_emit(const uint32_t (&keys)[R * E], const int32_t (&ids)[R * E],
                             uint32_t valid, const Threshold &th, Sink &&sink,
                             BlockScratch &sm, int &gt_base, int &eq_base) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        int gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = r * E + e;
            if (valid >> i & 1u) {
                gt += keys[i] > th.T;
                eq += keys[i] == th.T;
            }
        }
        int total;
        const int excl = block_excl_scan<NT>((gt << 16) | eq, sm, total);
        int g = gt_base + (excl >> 16), q = eq_base + (excl & 0xffff);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = r * E + e;
            if (!(valid >> i & 1u)) continue;
            if (keys[i] > th.T) {
                sink(g + min(q, th.budget), keys[i], ids[i]);
                ++g;
            } else if (keys[i] == th.T) {
                if (q < th.budget) sink(g + q, keys[i], ids[i]);
                ++q;
            }
        }
        gt_base += total >> 16;
        eq_base += total & 0xffff;
    }
}

}  // namespace qsa
