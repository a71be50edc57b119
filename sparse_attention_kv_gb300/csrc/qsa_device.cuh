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
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));   // -0 + 0 = +0; every other score unchanged
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Inverse of score_key (for keys of non-NaN scores; both zeros come back as +0).
__device__ __forceinline__ float key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// Programmatic dependent launch.  wait_prior_grid() blocks until the grid launched
// before this one on the stream has completed and its memory writes are visible; it
// returns at once when this grid was launched without the programmatic attribute.
// allow_dependent_launch() lets a grid launched after this one with that attribute
// start its CTAs (which then wait in wait_prior_grid) once every CTA of this grid
// has executed it or exited.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
struct __align__(16) BlockScratch {
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


// ---------------------------------------------------------------------------
// Selection over candidates held in shared memory (unordered lists).

// Append the calling threads' items to a shared list with one atomic per warp.
// Returns the list slot of this thread's first item.  All 32 lanes call.
__device__ __forceinline__ int warp_append(int count, int *counter) {
    const int lane = threadIdx.x & 31;
    const int incl = warp_incl_scan(count);
    int base = 0;
    if (lane == 31 && incl > 0) base = atomicAdd(counter, incl);
    base = __shfl_sync(kFull, base, 31);
    return base + incl - count;
}

template <int NT>
struct __align__(16) CandSmem {
    static constexpr int NW = NT / 32;
    uint32_t hist[256];   // one digit histogram; zero between passes
    uint32_t wmin[NW], wmax[NW];
    int misc[8];
    int cnt[4];           // list counters
};

template <int NT>
__device__ __forceinline__ void cand_smem_init(CandSmem<NT> &sm) {
    for (int i = threadIdx.x; i < 256; i += NT) sm.hist[i] = 0u;
    if (threadIdx.x < 4) sm.cnt[threadIdx.x] = 0;
}

// Block min and max of per-thread (mn, mx), returned to every thread (one barrier).
template <int NT>
__device__ __forceinline__ void block_minmax(uint32_t &mn, uint32_t &mx, CandSmem<NT> &sm) {
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sm.wmin[wid] = mn;
        sm.wmax[wid] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < CandSmem<NT>::NW; ++w) {
        mn = min(mn, sm.wmin[w]);
        mx = max(mx, sm.wmax[w]);
    }
}

// k-th largest of the keys key_at(i), i < m, for which key_at returns true;
// every such key lies in [mn, mx].  The bits mn and mx share are skipped, the
// rest are taken 8 at a time from the top: a shared histogram of the digit over
// the keys that match the prefix so far, then warp 0 scans the bins from the
// highest down (clearing them) to find the bin of the k-th key.  Two barriers a
// digit; the histogram must be zero on entry and is left zero.
template <int NT, typename KeyAt>
__device__ Threshold smem_threshold(KeyAt &&key_at, int m, int k, uint32_t mn, uint32_t mx,
                                    CandSmem<NT> &sm) {
    const int lane = threadIdx.x & 31;
    int hi = 32 - __clz((int)(mn ^ mx));
    uint32_t prefix = hi == 32 ? 0u : (mx & ~((1u << hi) - 1u));
    int remaining = k;
    while (hi > 0) {
        const int lo = hi > 8 ? hi - 8 : 0;
        const int nbins = 1 << (hi - lo);
        for (int i = threadIdx.x; i < m; i += NT) {
            uint32_t key;
            if (key_at(i, key) && (hi == 32 || (key >> hi) == (prefix >> hi)))
                atomicAdd(&sm.hist[(key >> lo) & (uint32_t)(nbins - 1)], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t c[8];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int b = nbins - 1 - 8 * lane - j;
                c[j] = 0u;
                if (b >= 0) {
                    c[j] = sm.hist[b];
                    sm.hist[b] = 0u;
                }
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
    }
    Threshold t;
    t.T = prefix;
    t.above = k - remaining;
    t.budget = remaining;
    return t;
}

// The k selected candidates i < m: every key > T, and of the keys == T the
// `budget` lowest ids (a second threshold over ~id among the ties when there
// are more ties than budget).  key_at(i) gives candidate i's key, id_at(i) its
// block id.  Appends ids (and keys, when sel_key is not null) to sel_id through
// sm.cnt[0]; uses sm.cnt[1].  Both counters must be zero on entry.  Ends with a
// barrier, after which sm.cnt[0] == k.
template <int NT, typename KeyAt, typename IdAt>
__device__ void collect_smem(KeyAt &&key_at, IdAt &&id_at, int m, const Threshold &th, uint32_t *sel_key,
                             int32_t *sel_id, CandSmem<NT> &sm) {
    int neq = 0;
    for (int base = 0; base < m; base += NT) {
        const int i = base + (int)threadIdx.x;
        const uint32_t key = i < m ? key_at(i) : 0u;
        const bool gt = i < m && key > th.T;
        neq += (i < m && key == th.T);
        const int pos = warp_append(gt ? 1 : 0, &sm.cnt[0]);
        if (gt) {
            if (sel_key) sel_key[pos] = key;
            sel_id[pos] = id_at(i);
        }
    }
    const int wt = (int)__reduce_add_sync(kFull, (unsigned)neq);
    if ((threadIdx.x & 31) == 0 && wt) atomicAdd(&sm.cnt[1], wt);
    __syncthreads();
    const int ntie = sm.cnt[1];
    uint32_t T2 = 0u;   // ties with ~id >= T2 are taken; all of them when T2 == 0
    if (ntie > th.budget) {
        const Threshold t2 = smem_threshold<NT>(
            [&](int i, uint32_t &key) {
                if (key_at(i) != th.T) return false;
                key = ~(uint32_t)id_at(i);
                return true;
            },
            m, th.budget, 0u, 0xffffffffu, sm);
        T2 = t2.T;
    }
    for (int base = 0; base < m; base += NT) {
        const int i = base + (int)threadIdx.x;
        const bool take = i < m && key_at(i) == th.T && ~(uint32_t)id_at(i) >= T2;
        const int pos = warp_append(take ? 1 : 0, &sm.cnt[0]);
        if (take) {
            if (sel_key) sel_key[pos] = th.T;
            sel_id[pos] = id_at(i);
        }
    }
    __syncthreads();
}

// Sort n (<= 1024) ids held in shared memory ascending and write them to out,
// padded with -1 up to k.  n <= 32: warp 0 sorts them in registers (bitonic);
// else a bitonic sort in shared memory over the next power of two (`buf` must
// hold that many ints).  Every thread of the block calls it.
template <int NT>
__device__ void sort_emit(int32_t *buf, int n, int k, int32_t *out) {
    const int lane = threadIdx.x & 31;
    if (n <= 32) {
        if (threadIdx.x < 32) {
            int v = lane < n ? buf[lane] : 0x7fffffff;
#pragma unroll
            for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    const int o = __shfl_xor_sync(kFull, v, stride);
                    const bool up = (lane & size) == 0;
                    const bool lower = (lane & stride) == 0;
                    v = (lower == up) ? min(v, o) : max(v, o);
                }
            }
            if (lane < n) out[lane] = v;
        }
    } else {
        int P = 64;
        while (P < n) P <<= 1;
        for (int i = n + threadIdx.x; i < P; i += NT) buf[i] = 0x7fffffff;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = threadIdx.x; i < P / 2; i += NT) {
                    const int lo = 2 * i - (i & (stride - 1));
                    const int hi = lo + stride;
                    const bool up = (lo & size) == 0;
                    const int a = buf[lo], b = buf[hi];
                    if ((a > b) == up) {
                        buf[lo] = b;
                        buf[hi] = a;
                    }
                }
                __syncthreads();
            }
        }
        for (int i = threadIdx.x; i < n; i += NT) out[i] = buf[i];
    }
    for (int i = n + threadIdx.x; i < k; i += NT) out[i] = -1;
}

// One warp: the r-th largest (1 <= r <= n) of n <= 256 keys, held 8 per lane
// (lane l has v[l + 32e]; absent entries are 0, below every score key).  Each
// lane sorts its 8 keys descending, then r rounds take the warp maximum of the
// lanes' heads and advance the first lane holding it.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t (&x)[8], int r) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int j = 0; j < 7 - i; ++j) {
            const uint32_t a = x[j], b = x[j + 1];
            x[j] = max(a, b);
            x[j + 1] = min(a, b);
        }
    }
    uint32_t res = 0u;
    for (int it = 0; it < r; ++it) {
        res = __reduce_max_sync(kFull, x[0]);
        const unsigned win = __ballot_sync(kFull, x[0] == res);
        if (lane == __ffs(win) - 1) {
#pragma unroll
            for (int j = 0; j < 7; ++j) x[j] = x[j + 1];
            x[7] = 0u;
        }
    }
    return res;
}


// ---------------------------------------------------------------------------
// One warp selecting over a list held in shared memory (no block barriers).

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Warp-wide min / max of 32- and 64-bit keys.
__device__ __forceinline__ uint32_t warp_min(uint32_t x) { return __reduce_min_sync(kFull, x); }
__device__ __forceinline__ uint32_t warp_max(uint32_t x) { return __reduce_max_sync(kFull, x); }
__device__ __forceinline__ uint64_t warp_min(uint64_t x) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const uint64_t o = __shfl_xor_sync(kFull, x, d);
        x = o < x ? o : x;
    }
    return x;
}
__device__ __forceinline__ uint64_t warp_max(uint64_t x) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const uint64_t o = __shfl_xor_sync(kFull, x, d);
        x = o > x ? o : x;
    }
    return x;
}
__device__ __forceinline__ int key_clz(uint32_t x) { return __clz(x); }
__device__ __forceinline__ int key_clz(uint64_t x) { return __clzll(x); }

// One warp: emit, in list order, every entry with key > T and the first `budget`
// entries with key == T; stops once k entries are out.  emit(pos, i) as below.
template <typename K, typename KeyAt, typename Emit>
__device__ __forceinline__ void warp_emit_ordered(KeyAt &&key_at, int n, int k, K T, int budget, Emit &&emit) {
    const int lane = threadIdx.x & 31;
    int taken = 0, ties = 0;
    for (int base = 0; base < n && taken < k; base += 32) {
        const int i = base + lane;
        const K key = i < n ? key_at(i) : K(0);
        const bool gt = i < n && key > T;
        const bool eq = i < n && key == T;
        const unsigned eqm = __ballot_sync(kFull, eq);
        const bool take = gt || (eq && ties + __popc(eqm & lanemask_lt()) < budget);
        const unsigned tm = __ballot_sync(kFull, take);
        if (take) emit(taken + __popc(tm & lanemask_lt()), i);
        taken += __popc(tm);
        ties += __popc(eqm);
    }
}

// The k selected entries of a list i < n (key_at(i) gives a 32- or 64-bit key),
// in list order: every key > T plus, of the keys == T, the first `budget` in list
// order (T = the k-th largest key).  When the list is in ascending block-id order
// the result is the reference selection in ascending id order.  emit(pos, i) is
// called for each selected entry with its output slot pos (0..min(n,k)-1).
// hist: this warp's 256-word shared histogram (zero on entry, left zero).
// All 32 lanes call; no block-wide barrier is used.
template <typename KeyAt, typename Emit>
__device__ void warp_select(KeyAt &&key_at, int n, int k, uint32_t *hist, Emit &&emit) {
    using K = decltype(key_at(0));
    constexpr int kBits = 8 * sizeof(K);
    const int lane = threadIdx.x & 31;
    if (n <= k) {   // everything is selected
        for (int i = lane; i < n; i += 32) emit(i, i);
        return;
    }
    K mn = ~K(0), mx = K(0);
    for (int i = lane; i < n; i += 32) {
        const K key = key_at(i);
        mn = min(mn, key);
        mx = max(mx, key);
    }
    mn = warp_min(mn);
    mx = warp_max(mx);
    int hi = kBits - key_clz(mn ^ mx);
    K prefix = hi == kBits ? K(0) : (mx & ~((K(1) << hi) - K(1)));
    int remaining = k;
    while (hi > 0) {
        const int lo = hi > 8 ? hi - 8 : 0;
        const int nbins = 1 << (hi - lo);
        for (int i = lane; i < n; i += 32) {
            const K key = key_at(i);
            if (hi == kBits || (key >> hi) == (prefix >> hi))
                atomicAdd(&hist[static_cast<uint32_t>(key >> lo) & (uint32_t)(nbins - 1)], 1u);
        }
        __syncwarp();
        uint32_t c[8];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int b = nbins - 1 - 8 * lane - j;
            c[j] = 0u;
            if (b >= 0) {
                c[j] = hist[b];
                hist[b] = 0u;
            }
            sum += (int)c[j];
        }
        const int incl = warp_incl_scan(sum);
        int run = incl - sum;
        int digit = 0, above = 0;
        const bool mine = run < remaining && remaining <= incl;
        if (mine) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (run + (int)c[j] >= remaining) {
                    digit = nbins - 1 - 8 * lane - j;
                    above = run;
                    break;
                }
                run += (int)c[j];
            }
        }
        const int src = __ffs(__ballot_sync(kFull, mine)) - 1;
        digit = __shfl_sync(kFull, digit, src);
        above = __shfl_sync(kFull, above, src);
        remaining -= above;
        prefix |= static_cast<K>(digit) << lo;
        hi = lo;
        __syncwarp();
    }
    warp_emit_ordered(key_at, n, k, prefix, remaining, emit);
}


// ---------------------------------------------------------------------------
// Packed candidates and warp sorting networks.
//
// A candidate (key, block id) packs into (key << 32) | ~id.  Block ids are
// distinct and non-negative, so packed values are distinct, never 0, and a larger
// packed value is a larger key or, on equal keys, a lower block id: the order in
// which the selection takes blocks.

__device__ __forceinline__ uint64_t pack_cand(uint32_t key, int32_t id) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~id);
}
__device__ __forceinline__ uint32_t cand_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ int32_t cand_id(uint64_t c) { return ~static_cast<int32_t>(static_cast<uint32_t>(c)); }

// Bitonic sort of 64 values held two per lane (element 2 * lane + s is v_s),
// descending: afterwards element r is the (r+1)-th largest.  21 compare-exchange
// steps, 15 of them across lanes.
template <typename T>
__device__ __forceinline__ void warp_sort64_desc(T &v0, T &v1) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1) {
        const bool desc = ((2 * lane) & size) == 0;
#pragma unroll
        for (int stride = size >> 1; stride >= 1; stride >>= 1) {
            if (stride == 1) {
                const T hi = v0 > v1 ? v0 : v1, lo = v0 > v1 ? v1 : v0;
                v0 = desc ? hi : lo;
                v1 = desc ? lo : hi;
            } else {
                const int d = stride >> 1;   // partner lane distance
                const bool keep_max = ((lane & d) == 0) == desc;
                const T o0 = __shfl_xor_sync(kFull, v0, d), o1 = __shfl_xor_sync(kFull, v1, d);
                v0 = keep_max ? (v0 > o0 ? v0 : o0) : (v0 > o0 ? o0 : v0);
                v1 = keep_max ? (v1 > o1 ? v1 : o1) : (v1 > o1 ? o1 : v1);
            }
        }
    }
}

// Bitonic sort of 32 values, one per lane, ascending by lane.
template <typename T>
__device__ __forceinline__ void warp_sort32_asc(T &v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
        const bool asc = (lane & size) == 0;
#pragma unroll
        for (int stride = size >> 1; stride >= 1; stride >>= 1) {
            const T o = __shfl_xor_sync(kFull, v, stride);
            const bool keep_min = ((lane & stride) == 0) == asc;
            v = keep_min ? (v < o ? v : o) : (v < o ? o : v);
        }
    }
}

// The k-th largest (1 <= k <= 32) of the 64 values held two per lane: a lower
// bound of a list's k-th largest key when each lane holds the two largest keys of
// its own share of the list (distinct entries; 0 where a share has fewer than
// two), since then k distinct entries reach it.
__device__ __forceinline__ uint32_t warp_bound_from_top2(uint32_t m1, uint32_t m2, int k) {
    warp_sort64_desc(m1, m2);
    const int r = k - 1;
    return __shfl_sync(kFull, (r & 1) ? m2 : m1, r >> 1);
}

// The top k of m <= 64 distinct packed candidates buf[0..m) (k <= m): emit(r, c)
// for the candidate c of rank r < k (rank 0 the largest).  Each lane ranks
// entries lane and lane + 32 against all m by shared-memory broadcast reads, so
// there is no shuffle chain.  buf needs 16-byte alignment and room for 64.
template <typename Emit>
__device__ __forceinline__ void warp_rank_top(uint64_t *buf, int m, int k, Emit &&emit) {
    const int lane = threadIdx.x & 31;
    if (lane == 0 && (m & 1)) buf[m] = 0ull;   // pad to pairs: 0 is below every candidate
    __syncwarp();
    const uint64_t v0 = lane < m ? buf[lane] : 0ull;
    const uint64_t v1 = lane + 32 < m ? buf[lane + 32] : 0ull;
    int r0 = 0, r1 = 0;
    const ulonglong2 *b2 = reinterpret_cast<const ulonglong2 *>(buf);
#pragma unroll 4
    for (int j = 0; j < (m + 1) >> 1; ++j) {
        const ulonglong2 pr = b2[j];
        r0 += (pr.x > v0) + (pr.y > v0);
        r1 += (pr.x > v1) + (pr.y > v1);
    }
    if (lane < m && r0 < k) emit(r0, v0);
    if (lane + 32 < m && r1 < k) emit(r1, v1);
    __syncwarp();
}

// Exact ranks of m distinct packed candidates cand[0..m) (rank 0 = the largest):
// sel[r] = the id of the candidate of rank r, for r < k (exactly k rank below k when
// m >= k).  A rank is the number of candidates above; P threads per candidate (a
// power of two dividing the warp) share the count.  Every thread of the NT-thread
// block calls it.
template <int NT>
__device__ __forceinline__ void rank_survivors(const uint64_t *cand, int m, int k, int32_t *sel) {
    if (m <= 64) {   // the common case: every compare unrolled, P fixed
        constexpr int P = NT / 64;
        const int i = (int)threadIdx.x / P, sub = (int)threadIdx.x % P;
        const uint64_t c = i < m ? cand[i] : 0ull;
        int rk = 0;
#pragma unroll
        for (int t = 0; t < 64 / P; ++t) {
            const int j = sub + P * t;
            rk += j < m && cand[j] > c;
        }
#pragma unroll
        for (int o = 1; o < P; o <<= 1) rk += __shfl_xor_sync(kFull, rk, o);
        if (sub == 0 && i < m && rk < k) sel[rk] = cand_id(c);
        return;
    }
    int lp = 0;   // P = 1 << lp <= 8, as many as the block holds
    while (lp < 3 && (2 * m << lp) <= NT) ++lp;
    const int P = 1 << lp;
    for (int b0 = 0; b0 < m * P; b0 += NT) {
        const int e = b0 + (int)threadIdx.x;
        const int i = e >> lp, sub = e & (P - 1);
        const uint64_t c = i < m ? cand[i] : 0ull;
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        int j = sub;
        for (; j + 3 * P < m; j += 4 * P) {
            r0 += cand[j] > c;
            r1 += cand[j + P] > c;
            r2 += cand[j + 2 * P] > c;
            r3 += cand[j + 3 * P] > c;
        }
        for (; j < m; j += P) r0 += cand[j] > c;
        int rk = (r0 + r1) + (r2 + r3);
        for (int o = 1; o < P; o <<= 1) rk += __shfl_xor_sync(kFull, rk, o);
        if (sub == 0 && i < m && rk < k) sel[rk] = cand_id(c);
    }
}

}  // namespace qsa
