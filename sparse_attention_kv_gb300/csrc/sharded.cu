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
};

// Stage B: one CTA per query.  The query's candidates of every shard (id >= 0) go
// to shared memory as (key, id); the threshold T (the k-th largest key), the keys
// above it and, of the keys equal to it, the lowest ids give the k selected
// blocks (the rule of "#2093 sm_75: the prompt path's top-k with one full read of
// the scores", step 3), emitted in ascending id order and -1 padded.
__global__ void __launch_bounds__(kMergeNT) merge_kernel(const float *__restrict__ cand_scores,
                                                         const int32_t *__restrict__ cand_ids, int n_shards, int nq,
                                                         int k, int32_t *__restrict__ out_ids) {
    wait_prior_grid();   // the candidates may come from the kernel launched just before
    allow_dependent_launch();
    __shared__ MergeSmem sm;
    const int q = blockIdx.x;
    cand_smem_init(sm.cs);
    __syncthreads();
    const int total = n_shards * k;
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int base = 0; base < total; base += kMergeNT) {
        const int e = base + (int)threadIdx.x;
        const int g = e / k, i = e - (e / k) * k;
        const size_t off = ((size_t)g * nq + q) * k + i;
        const int32_t id = e < total ? cand_ids[off] : -1;
        const bool v = id >= 0;
        const int pos = warp_append(v ? 1 : 0, &sm.cs.cnt[2]);
        if (v) {
            const uint32_t key = score_key(cand_scores[off]);
            sm.key[pos] = key;
            sm.id[pos] = id;
            mn = min(mn, key);
            mx = max(mx, key);
        }
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

qsa_status launch_merge(const float *cand_scores, const int32_t *cand_ids, int n_shards, int nq, int k, int32_t *ids,
                        cudaStream_t s) {
    return launch_pdl("merge_kernel launch", merge_kernel, dim3(nq), dim3(kMergeNT), s, cand_scores, cand_ids,
                      n_shards, nq, k, ids);
}

}  // namespace qsa
