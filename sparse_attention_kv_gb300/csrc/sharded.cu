// sharded.cu -- selection over KV blocks split into shards (one per GPU, or any
// partition of a query's blocks): stage A keeps each shard's k best blocks as
// candidates (score and global block id), stage B merges every shard's candidates
// into the selection.
//
// A query's selection restricted to a subset of its blocks is a prefix of that
// subset's order, score descending then block id ascending (Strata PR #3987,
// section "Approach": the chunks of the split each keep their top k and one CTA
// per query selects over the union).  So every selected block is among its
// shard's k best, and selecting over the union of the shards' candidates in the
// same order gives exactly the blocks of one selection over all blocks.
#include <cstdint>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kMergeNT = 256;   // threads of the merge kernel (one CTA per query)

// Stage A, after the shard's top-k has written its (local, ascending) ids: the
// candidates' scores, and the ids moved to the global numbering.  Slots with no
// block (id -1) keep id -1.
__global__ void __launch_bounds__(256) candidates_kernel(const float *__restrict__ scores, int64_t stride,
                                                         int32_t *__restrict__ ids, float *__restrict__ cand_scores,
                                                         int nq, int k, int32_t offset) {
    wait_prior_grid();   // the ids come from the top-k launched just before
    allow_dependent_launch();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)nq * k) return;
    const int q = (int)(e / k);
    const int32_t id = ids[e];
    if (id >= 0) {
        cand_scores[e] = scores[(size_t)q * stride + id];
        ids[e] = id + offset;
    } else {
        cand_scores[e] = __int_as_float(0xff800000);   // -inf; the slot is empty (id -1)
    }
}

struct __align__(16) MergeSmem {
    CandSmem<kMergeNT> cs;
    uint32_t key[kMergeCap];
    int32_t id[kMergeCap];
    int32_t sel[1024];
    uint64_t cand[kMergeNT];   // k <= 32: the candidates at or above the bound, packed
    uint32_t wb[kMergeNT / 32];
    int nsurv;
};

// Stage B: one CTA per query.  The query's candidates of every shard (id >= 0; with
// counts, the first counts[q * counts_stride + g] of shard g) go to shared memory as
// (key, id); the threshold T (the k-th largest key), the keys above it and, of the
// keys equal to it, the lowest ids give the k selected blocks (the rule of "#2093
// sm_75: the prompt path's top-k with one full read of the scores", step 3),
// emitted in ascending id order and -1 padded.  Shard g's candidates of query q
// start at ((g nq) + q) kslot.
__global__ void __launch_bounds__(kMergeNT) merge_kernel(const float *__restrict__ cand_scores,
                                                         const int32_t *__restrict__ cand_ids,
                                                         const int32_t *__restrict__ counts, int counts_stride,
                                                         int n_shards, int nq, int kslot, int k,
                                                         int32_t *__restrict__ out_ids) {
    wait_prior_grid();   // the candidates may come from the kernel launched just before
    allow_dependent_launch();
    __shared__ MergeSmem sm;
    const int q = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    cand_smem_init(sm.cs);
    if (threadIdx.x == 0) sm.nsurv = 0;
    // the lengths of this thread's lists first, then the loads of every slot of this
    // thread that holds a candidate (slots t, t + 256, ... of the shard-major list) at
    // once, so that they are all in flight together
    constexpr int PER = kMergeCap / kMergeNT;
    const int total = n_shards * kslot;   // <= kMergeCap
    float sc[PER];
    int32_t cid[PER], len[PER], slot[PER];
    size_t off[PER];
    // slot e = r * 256 + t is slot i of list g; one division, then steps of 256 slots
    const int step_g = kMergeNT / kslot, step_i = kMergeNT - step_g * kslot;
    int g = (int)threadIdx.x / kslot, i = (int)threadIdx.x - g * kslot;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const bool in = r * kMergeNT + (int)threadIdx.x < total;
        off[r] = ((size_t)g * nq + q) * kslot + i;
        slot[r] = in ? i : kslot;   // kslot: at or past every list's length
        len[r] = min(g, n_shards - 1);   // the slot's list for now; its length below
        g += step_g;
        i += step_i;
        if (i >= kslot) {
            i -= kslot;
            ++g;
        }
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) len[r] = counts ? counts[(size_t)q * counts_stride + len[r]] : kslot;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const bool v = slot[r] < len[r];
        cid[r] = v ? cand_ids[off[r]] : -1;
        sc[r] = v ? cand_scores[off[r]] : 0.0f;
    }
    __syncthreads();   // the counters above are set
    int nv = 0;
#pragma unroll
    for (int r = 0; r < PER; ++r) nv += cid[r] >= 0;
    int pos = warp_append(nv, &sm.cs.cnt[2]);
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int r = 0; r < PER; ++r)
        if (cid[r] >= 0) {
            const uint32_t key = score_key(sc[r]);
            sm.key[pos] = key;
            sm.id[pos] = cid[r];
            ++pos;
            mn = min(mn, key);
            mx = max(mx, key);
        }
    block_minmax<kMergeNT>(mn, mx, sm.cs);
    const int m = sm.cs.cnt[2];
    int32_t *out = out_ids + (size_t)q * k;
    if (m <= k) {   // every candidate is selected
        for (int i = threadIdx.x; i < m; i += kMergeNT) sm.sel[i] = sm.id[i];
        __syncthreads();
        sort_emit<kMergeNT>(sm.sel, m, k, out);
        return;
    }
    if (k <= 32) {
        // A bound first, as in the warp top-k: thread t's candidates are t, t + 256, ...;
        // each warp takes the r-th largest of its threads' maxima (r = ceil(k / 8)) and
        // the bound is the smallest of those, so at least k candidates reach it.  The few
        // that do are ranked exactly on (key, ~id), the selection order.  Fewer than 256
        // candidates: all of them are ranked.
        if (m <= kMergeNT) {
            for (int i = threadIdx.x; i < m; i += kMergeNT) sm.cand[i] = pack_cand(sm.key[i], sm.id[i]);
            if (threadIdx.x == 0) sm.nsurv = m;
        } else {
            uint32_t tm = 0u;   // every thread holds a candidate (m > 256)
            for (int i = threadIdx.x; i < m; i += kMergeNT) tm = max(tm, sm.key[i]);
            const int r = (k + kMergeNT / 32 - 1) / (kMergeNT / 32);
            uint32_t res = 0u;
            for (int it = 0; it < r; ++it) {
                res = __reduce_max_sync(kFull, tm);
                const unsigned win = __ballot_sync(kFull, tm == res);
                if (lane == __ffs(win) - 1) tm = 0u;   // 0 is below every score's key
            }
            if (lane == 0) sm.wb[warp] = res;
            __syncthreads();
            uint32_t B = 0xffffffffu;
#pragma unroll
            for (int w = 0; w < kMergeNT / 32; ++w) B = min(B, sm.wb[w]);
            for (int i = threadIdx.x; i < m; i += kMergeNT)
                if (sm.key[i] >= B) {
                    const int p = atomicAdd(&sm.nsurv, 1);
                    if (p < kMergeNT) sm.cand[p] = pack_cand(sm.key[i], sm.id[i]);
                }
        }
        __syncthreads();
        const int m2 = sm.nsurv;
        if (m2 <= kMergeNT) {
            rank_survivors<kMergeNT>(sm.cand, m2, k, sm.sel);
            __syncthreads();
            if (warp == 0) {
                int v = lane < k ? sm.sel[lane] : 0x7fffffff;
                warp_sort32_asc(v);
                if (lane < k) out[lane] = v;
            }
            return;
        }
        // heavy ties at the bound: the exact select below
    }
    const Threshold th = smem_threshold<kMergeNT>(
        [&](int i, uint32_t &key) {
            key = sm.key[i];
            return true;
        },
        m, k, mn, mx, sm.cs);
    collect_smem<kMergeNT>([&](int i) { return sm.key[i]; }, [&](int i) { return sm.id[i]; }, m, th, nullptr,
                           sm.sel, sm.cs);
    sort_emit<kMergeNT>(sm.sel, k, k, out);
}

template <typename... KArgs, typename... Args>
qsa_status launch_pdl(const char *what, void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                      Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, kern, args...), what);
}

}  // namespace

qsa_status launch_candidates(const float *scores, int64_t stride, int32_t *ids, float *cand_scores, int nq, int k,
                             int32_t offset, cudaStream_t s) {
    const int64_t n = (int64_t)nq * k;
    const dim3 grid((unsigned)((n + 255) / 256));
    return launch_pdl("candidates_kernel launch", candidates_kernel, grid, dim3(256), s, scores, stride, ids,
                      cand_scores, nq, k, offset);
}

qsa_status launch_merge(const float *cand_scores, const int32_t *cand_ids, const int32_t *counts, int counts_stride,
                        int n_shards, int nq, int kslot, int k, int32_t *ids, cudaStream_t s) {
    return launch_pdl("merge_kernel launch", merge_kernel, dim3(nq), dim3(kMergeNT), s, cand_scores, cand_ids,
                      counts, counts_stride, n_shards, nq, kslot, k, ids);
}

}  // namespace qsa
