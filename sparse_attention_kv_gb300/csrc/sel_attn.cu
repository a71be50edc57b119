// sel_attn.cu -- selection attention, forward, over the blocks each query selected.
//
//   o[q][h][:] = sum_t p_t V[g][t][:] / sum_t p_t,  p_t = exp(scale * (s_t - m)),
//   s_t = dot(qa[q][h][:], K[g][t][:]),  m = max_t s_t,  g = h / 16,
//
// over the tokens t of the distinct selected blocks ids[q][*] (64 tokens each)
// that lie below n_tokens[q].  This is the consumer of the block selection set
// out in "[wave] NSA: LDS optimization for block-gather in selection attention"
// (section "Problem": a query reads the tokens of its selected blocks, which are
// scattered in memory; strategy 1: each block's K and V are staged on chip once
// and read there by every head of the GQA group).
//
// One CTA per (query, KV head); the 16 heads of the group are the N side of
// every MMA.  Two passes over on-chip data keep the softmax exact without
// rescaling:
//   1. S^T = K_pair . Q^T on tcgen05 (M = 128 tokens of two blocks, N = 16
//      heads, K = 128), one TMEM tile per pair of blocks; all of a query's
//      logits stay in TMEM (k <= 64 blocks -> at most 512 columns).
//   2. Four softmax warps (one TMEM lane = one token each) take the per-head
//      maximum over every visible token, then write p = exp2((s - m) * scale *
//      log2 e) rounded to the inputs' 16-bit format into a shared-memory ring and
//      sum the rounded values, so the output is an exact convex combination of
//      the weights used.
//   3. O^T += V_b^T . P_b^T on tcgen05 (M = 128 head dims, N = 16 heads, K = 64
//      tokens per block) accumulates in TMEM over the columns of the first
//      logit tile, which is consumed first.
// The V cache holds every 64-token block dimension-major ([128][64]), so both
// operands of both products are K-major under the 128-byte swizzle that TMA
// writes (q, K and V in bf16 or fp16; the weights in the same format).  Warp 0
// issues TMA loads (K pairs, then V pairs, through one ring), warp 1 owns TMEM
// and issues the MMAs, warps 2-5 run the softmax and the epilogue.  The kernel
// is launched as a programmatic dependent of the work before it and reads
// nothing the caller wrote until that work has completed.
//
// When the (query, KV head) units are too few to fill the GPU (a decode
// window), each unit's pairs are split over a thread-block cluster of 2, 4 or 8
// CTAs.  Each CTA keeps its slice's unnormalised output, per-head maximum and
// weight sum; after a cluster barrier it stores them through distributed shared
// memory into the CTA that combines each head, and after a second barrier every
// CTA combines its share of the group's heads from local memory (weights
// 2^((m_r - M) scale log2 e), M the largest partial maximum).
//
// Every wait is bounded; on expiry the CTA raises QSA_FLAG_WAIT_TIMEOUT, drains
// its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "qsa_device.cuh"
#include "tc_ptx.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kG = 16;                  // heads per GQA group (MMA N)
constexpr int kMaxSel = 64;             // blocks per query
constexpr int kStages = 3;              // K/V ring stages
constexpr int kStageBytes = 32768;      // two blocks of K (two 64-column halves) or of V^T
constexpr int kPStages = 2;             // P ring stages
constexpr int kPBytes = 4096;           // two blocks x 16 heads x 64 tokens bf16
constexpr int kThreads = 192;           // TMA warp, MMA warp, four softmax warps
constexpr int kSoft = 128;
// instruction-descriptor A/B formats of kind::f16
constexpr uint32_t kFmtF16 = 0, kFmtBF16 = 1;

constexpr int kOffQ = 0;                                  // 2 halves x 16 rows x 128 B
constexpr int kOffKV = 4096;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffCtrl = kOffP + kPStages * kPBytes;

struct AttnCtrl {
    uint64_t qfull;
    uint64_t full[kStages], empty[kStages];
    uint64_t sfull;                      // every logit tile written
    uint64_t pfull[kPStages], pempty[kPStages];
    uint64_t tailbar;                    // the V block holding the end of the context landed
    uint64_t ofull;                      // the output accumulator complete
    uint64_t done;                       // every MMA complete (teardown)
    uint32_t tmem_base;
    int abort;
    int nsel;
    int ntok;
    int32_t raw[kMaxSel];
    int32_t sel[kMaxSel];                // the distinct valid ids, in slot order
    float red[4][kG];
    float m[kG];                         // per-head maximum logit (unscaled)
    float l[kG];                         // per-head sum of the rounded weights
};
constexpr int kSmemBytes = kOffCtrl + (int)sizeof(AttnCtrl) + 1024;   // + alignment slack
// more than half of an SM's shared memory: one CTA per SM, for queries whose
// logits take all 512 TMEM columns
constexpr int kSmemOneBytes = 120 * 1024;
static_assert(kSmemBytes <= kSmemOneBytes, "attention shared memory");

struct AttnParams {
    const int32_t *ids;
    const int32_t *n_tokens;
    float *out;
    float *lse;
    uint32_t *flags;
    int n_heads, n_kv, k, capacity, nb_cap;
    int split;                           // CTAs per (query, KV head): 1, or a cluster of 2, 4 or 8
    float scale, scale_log2;
};
constexpr int kMaxSplit = 8;

__device__ __forceinline__ void soft_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Every lane of the calling warp learns whether lane 0's bounded wait succeeded.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
    return __shfl_sync(kFull, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Barrier over every thread of the cluster; release/acquire orders shared-memory
// writes before it with reads by other CTAs after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store to the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *local, int rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}
__device__ __forceinline__ void st_cluster(float4 *local, int rank, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr(local, rank)), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_cluster(float2 *local, int rank, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(cluster_addr(local, rank)), "f"(v.x), "f"(v.y)
                 : "memory");
}

// Byte offset of (row, col) of a bf16 tile with 128-byte rows under the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2);
}

// Zero tokens r..63 of a 64-token V^T block ([128 dims][64 tokens], swizzled), one
// warp.
__device__ __forceinline__ void clear_tail(uint8_t *blk, int r) {
    const int lane = threadIdx.x & 31;
    for (int d = lane; d < 128; d += 32)
        for (int c = r >> 3; c < 8; ++c) {
            uint8_t *chunk = blk + swz(d, 8 * c);
            if (8 * c >= r) {
                *reinterpret_cast<uint4 *>(chunk) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                uint16_t *e = reinterpret_cast<uint16_t *>(chunk);
                for (int t = r - 8 * c; t < 8; ++t) e[t] = 0;
            }
        }
}

// The weights of the P.V product in the inputs' 16-bit format, and their value.
template <bool F16>
__device__ __forceinline__ float store_weight(uint8_t *dst, float e) {
    if constexpr (F16) {
        const __half eh = __float2half_rn(e);
        *reinterpret_cast<__half *>(dst) = eh;
        return __half2float(eh);
    } else {
        const __nv_bfloat16 eb = __float2bfloat16_rn(e);
        *reinterpret_cast<__nv_bfloat16 *>(dst) = eb;
        return __bfloat162float(eb);
    }
}

// F16: q, K and V (and so the weights) are fp16; otherwise bf16.
template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    sel_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sKV = smem + kOffKV;
    uint8_t *sP = smem + kOffP;
    AttnCtrl &ct = *reinterpret_cast<AttnCtrl *>(smem + kOffCtrl);
    volatile int *abort_flag = &ct.abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = p.split;                       // CTAs (one cluster) per (query, KV head)
    const int rank = split > 1 ? (int)cluster_ctarank() : 0;
    const int unit = blockIdx.x / split;
    const int qi = unit / p.n_kv, g = unit % p.n_kv;
    const int head0 = g * kG;

    if (tid == 32) {
        mbar_init(&ct.qfull, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ct.full[s], 2);   // the producer's expect-tx arrival and its release arrival
            mbar_init(&ct.empty[s], 1);
        }
        mbar_init(&ct.tailbar, 1);
        mbar_init(&ct.sfull, 1);
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&ct.pfull[s], kSoft);
            mbar_init(&ct.pempty[s], 1);
        }
        mbar_init(&ct.ofull, 1);
        mbar_init(&ct.done, 1);
        ct.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    }
    __syncthreads();
    // The kernel may be launched as a programmatic dependent of the one that wrote the
    // ids (a top-k): nothing the caller wrote is read before this wait.
    wait_prior_grid();
    if (tid == 0) {   // the group's 16 query rows, two 64-column halves
        mbar_expect_tx(&ct.qfull, 2 * kG * 128);
        for (int hh = 0; hh < 2; ++hh)
            tma_load_2d(sQ + hh * kG * 128, &tm_q, &ct.qfull, hh * 64, qi * p.n_heads + head0);
    }
    if (warp == 2) {
        // the query's distinct ids inside its context, in slot order (both loads in
        // flight before either is used)
        const int32_t *row_ids = p.ids + (size_t)qi * p.k;
        const int32_t r0 = lane < p.k ? row_ids[lane] : -1;
        const int32_t r1 = lane + 32 < p.k ? row_ids[lane + 32] : -1;
        int ntok = p.n_tokens[qi];
        if (ntok < 0 || ntok > p.capacity) {
            if (lane == 0 && g == 0 && rank == 0 && p.flags) atomicOr(p.flags, QSA_FLAG_NBLOCKS_CLAMPED);
            ntok = ntok < 0 ? 0 : p.capacity;
        }
        const int nb = (ntok + 63) >> 6;
        ct.raw[lane] = r0;
        ct.raw[lane + 32] = r1;
        __syncwarp();
        int cnt = 0;
        bool bad = false;
        for (int j0 = 0; j0 < p.k; j0 += 32) {
            const int j = j0 + lane;
            const int32_t b = j < p.k ? ct.raw[j] : -1;
            bool take = b >= 0 && b < nb;
            bad |= j < p.k && b != -1 && !take;
            for (int i = 0; take && i < j; ++i) take = ct.raw[i] != b;
            const unsigned m = __ballot_sync(kFull, take);
            if (take) ct.sel[cnt + __popc(m & ((1u << lane) - 1u))] = b;
            cnt += __popc(m);
        }
        if (__any_sync(kFull, bad) && lane == 0 && rank == 0 && p.flags) atomicOr(p.flags, QSA_FLAG_BAD_ID);
        if (lane == 0) {
            ct.nsel = cnt;
            ct.ntok = ntok;
        }
    }
    __syncthreads();
    const int nsel = ct.nsel, ntok = ct.ntok;
    // this CTA's pair tiles: all of them, or a slice of a cluster's split
    const int T = (nsel + 1) >> 1;
    const int p0 = rank * T / split, p1 = (rank + 1) * T / split;
    const int tl = p1 - p0;
    const int b0 = 2 * p0;                          // first block of the slice (index into sel)
    const int nloc = min(nsel, 2 * p1) - b0;        // blocks of the slice
    float *out = p.out + ((size_t)qi * p.n_heads + head0) * 128;
    float *lse = p.lse ? p.lse + (size_t)qi * p.n_heads + head0 : nullptr;
    float *part = reinterpret_cast<float *>(sKV);   // split: this CTA's unnormalised output [16][128]

    if (nloc > 0) {
    uint32_t ncols = 32;
    while ((int)ncols < tl * 16) ncols <<= 1;
    if (warp == 1) {
        tmem_alloc(&ct.tmem_base, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ct.tmem_base;

    if (warp == 0) {
        // ---------------- producer: K pairs 0..tl-1, then V pairs 0..tl-1.  Lane 0
        // issues; the whole warp clears the V tokens past the context of the block
        // that holds its end, after that block lands and before the stage is
        // released to the MMA (its weights are 0, but 0 x NaN would not be).
        int issued = 0;
        bool tail_issued = false;
        for (int i = 0; i < 2 * tl; ++i) {
            const int s = i % kStages;
            if (!warp_wait(&ct.empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort_flag)) break;
            const int tile = i < tl ? i : i - tl;
            const int nb_t = min(2, nloc - 2 * tile);
            const int32_t *blk = ct.sel + b0 + 2 * tile;
            uint8_t *st = sKV + s * kStageBytes;
            int tail_j = -1;
            if (i >= tl)
                for (int j = 0; j < nb_t; ++j)
                    if ((blk[j] + 1) * 64 > ntok) tail_j = j;
            if (lane == 0) {
                mbar_expect_tx(&ct.full[s], (uint32_t)((nb_t - (tail_j >= 0 ? 1 : 0)) * 16384));   // arrival 1
                if (tail_j >= 0) mbar_expect_tx(&ct.tailbar, 16384u);
                for (int j = 0; j < nb_t; ++j) {
                    if (i < tl) {   // 64 token rows, two 64-column halves of 16 KB regions
                        const int y = g * p.capacity + blk[j] * 64;
                        tma_load_2d(st + j * 8192, &tm_k, &ct.full[s], 0, y);
                        tma_load_2d(st + 16384 + j * 8192, &tm_k, &ct.full[s], 64, y);
                    } else {        // 128 dimension rows of 64 tokens
                        tma_load_2d(st + j * 16384, &tm_v, j == tail_j ? &ct.tailbar : &ct.full[s], 0,
                                    (g * p.nb_cap + blk[j]) * 128);
                    }
                }
            }
            if (tail_j >= 0) {   // at most one block per query holds the end of its context
                tail_issued = true;
                if (warp_wait(&ct.tailbar, 0, abort_flag)) clear_tail(st + tail_j * 16384, ntok - blk[tail_j] * 64);
                fence_proxy_async();
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&ct.full[s]);   // arrival 2
            ++issued;
        }
        if (lane == 0) {
            for (int j = max(0, issued - kStages); j < issued; ++j)
                mbar_drain(&ct.full[j % kStages], (uint32_t)(j / kStages) & 1u);
            if (tail_issued) mbar_drain(&ct.tailbar, 0);
            mbar_drain(&ct.qfull, 0);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t id = idesc(F16 ? kFmtF16 : kFmtBF16, 128, kG);
            bool ok = mbar_wait(&ct.qfull, 0, abort_flag);
            tc_fence_after();
            const uint32_t q0 = smem_u32(sQ);
            for (int i = 0; ok && i < tl; ++i) {   // logits of pair i -> columns 16 i
                const int s = i % kStages;
                if (!(ok = mbar_wait(&ct.full[s], (uint32_t)(i / kStages) & 1u, abort_flag))) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sKV + s * kStageBytes);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma<MmaKind::f16>(tmem + (uint32_t)(i * 16), sdesc(a0 + (kk >> 2) * 16384 + (kk & 3) * 32),
                               sdesc(q0 + (kk >> 2) * (kG * 128) + (kk & 3) * 32), id, kk > 0 ? 1u : 0u);
                mma_commit(&ct.empty[s]);
            }
            if (ok) mma_commit(&ct.sfull);
            for (int i = 0; ok && i < tl; ++i) {   // output: columns 0..15, after pair 0 is consumed
                const int r = tl + i, s = r % kStages, ps = i % kPStages;
                if (!(ok = mbar_wait(&ct.full[s], (uint32_t)(r / kStages) & 1u, abort_flag))) break;
                if (!(ok = mbar_wait(&ct.pfull[ps], (uint32_t)(i / kPStages) & 1u, abort_flag))) break;
                tc_fence_after();
                const int nb_t = min(2, nloc - 2 * i);
                const uint32_t a0 = smem_u32(sKV + s * kStageBytes), bp = smem_u32(sP + ps * kPBytes);
                for (int j = 0; j < nb_t; ++j)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma<MmaKind::f16>(tmem, sdesc(a0 + j * 16384 + kk * 32), sdesc(bp + j * 2048 + kk * 32), id,
                                   (i | j | kk) != 0 ? 1u : 0u);
                mma_commit(&ct.empty[s]);
                mma_commit(&ct.pempty[ps]);
            }
            if (ok) mma_commit(&ct.ofull);
            mma_commit(&ct.done);
            mbar_drain(&ct.done, 0);
        }
    } else {
        // ---------------- softmax and epilogue: one TMEM lane (a token of a pair,
        // later a head dimension) per thread.  Every thread reaches every named
        // barrier, whatever the waits returned.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int half = row >> 6, tok = row & 63;
        const int sw = warp - 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        auto visible = [&](int i) {
            const int j = 2 * i + half;
            return j < nloc && ct.sel[b0 + j] * 64 + tok < ntok;
        };
        bool ok = warp_wait(&ct.sfull, 0, abort_flag);
        tc_fence_after();
        float mx[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) mx[h] = -INFINITY;
        if (ok) {
            for (int i0 = 0; i0 < tl; i0 += 4) {
                uint32_t v[4][16];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (i0 + u < tl) tmem_ld16_nowait(lane_addr + (uint32_t)((i0 + u) * 16), v[u]);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    reg_fence(v[u]);
                    if (i0 + u < tl && visible(i0 + u))
#pragma unroll
                        for (int h = 0; h < kG; ++h) mx[h] = fmaxf(mx[h], __uint_as_float(v[u][h]));
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kG; ++h) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], o));
        }
        if (lane == 0)
#pragma unroll
            for (int h = 0; h < kG; ++h) ct.red[sw][h] = mx[h];
        soft_barrier();
        float mc[kG];   // m * scale * log2(e)
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            const float m = fmaxf(fmaxf(ct.red[0][h], ct.red[1][h]), fmaxf(ct.red[2][h], ct.red[3][h]));
            mc[h] = m * p.scale_log2;
            if (row == 0) ct.m[h] = m;
        }
        float l[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) l[h] = 0.0f;
        for (int i = 0; ok && i < tl; ++i) {
            const int ps = i % kPStages;
            if (i >= kPStages && !(ok = warp_wait(&ct.pempty[ps], (uint32_t)((i / kPStages) - 1) & 1u, abort_flag)))
                break;
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16_nowait(lane_addr + (uint32_t)(i * 16), v);
            tmem_wait_ld();
            reg_fence(v);
            if (2 * i + half < nloc) {   // this row's block exists: write its weights (0 past the context)
                const bool vis = visible(i);
                uint8_t *pb = sP + ps * kPBytes + half * 2048;
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    const float e = vis ? exp2f(fmaf(__uint_as_float(v[h]), p.scale_log2, -mc[h])) : 0.0f;
                    l[h] += store_weight<F16>(pb + swz(h, tok), e);
                }
            }
            fence_proxy_async();   // the weights are read by the tensor core
            tc_fence_before();
            mbar_arrive(&ct.pfull[ps]);
        }
#pragma unroll
        for (int h = 0; h < kG; ++h) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l[h] += __shfl_xor_sync(kFull, l[h], o);
        }
        soft_barrier();   // every warp has read ct.red
        if (lane == 0)
#pragma unroll
            for (int h = 0; h < kG; ++h) ct.red[sw][h] = l[h];
        soft_barrier();
        if (row < kG) ct.l[row] = (ct.red[0][row] + ct.red[1][row]) + (ct.red[2][row] + ct.red[3][row]);
        soft_barrier();
        ok = ok && warp_wait(&ct.ofull, 0, abort_flag);
        tc_fence_after();
        if (ok) {
            uint32_t o[16];
            tmem_ld16_nowait(lane_addr, o);
            tmem_wait_ld();
            reg_fence(o);
            // row = head dimension d; a warp's stores for one head are 32 consecutive floats
            if (split == 1) {
#pragma unroll
                for (int h = 0; h < kG; ++h) out[h * 128 + row] = __uint_as_float(o[h]) / ct.l[h];
                if (lse && row < kG) lse[row] = p.scale * ct.m[row] + logf(ct.l[row]);
            } else {   // the ring is idle once the output is complete
#pragma unroll
                for (int h = 0; h < kG; ++h) part[h * 128 + row] = __uint_as_float(o[h]);
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
    } else {   // no visible token in this CTA's slice
        if (split == 1 && warp >= 2) {   // o = 0, lse = -inf
            for (int i = tid - 64; i < kG * 128; i += kSoft) out[i] = 0.0f;
            if (lse && tid - 64 < kG) lse[tid - 64] = -INFINITY;
        }
        if (tid < kG) {
            ct.m[tid] = -INFINITY;
            ct.l[tid] = 0.0f;
        }
        if (tid == 0) mbar_drain(&ct.qfull, 0);
    }
    if (tid == 0 && ct.abort && p.flags) atomicOr(p.flags, QSA_FLAG_WAIT_TIMEOUT);
    if (split > 1) {
        // Every CTA of the cluster is past its last MMA and copy, so every ring is
        // idle.  Each CTA sends its partial (m, l and the unnormalised output of each
        // head) to the CTA that combines that head, into the second ring stage of the
        // receiver; after the second barrier every combine reads local memory only.
        const int nh = kG / split;                                   // heads combined per CTA
        float *recv = reinterpret_cast<float *>(sKV + kStageBytes);  // [split][nh][128]
        float *recv_ml = recv + kG * 128;                            // [split][nh][2]
        cluster_sync();
        for (int e = tid; e < kG * 32; e += kThreads) {              // float4 e of part: head e / 32
            const int h = e >> 5, d4 = e & 31;
            const float4 v = reinterpret_cast<const float4 *>(part)[e];
            st_cluster(reinterpret_cast<float4 *>(recv + ((rank * nh + h % nh) * 128)) + d4, h / nh, v);
        }
        if (tid < kG) {
            const float2 ml = make_float2(ct.m[tid], ct.l[tid]);
            st_cluster(reinterpret_cast<float2 *>(recv_ml) + rank * nh + tid % nh, tid / nh, ml);
        }
        cluster_sync();
        for (int e = tid; e < nh * 128; e += kThreads) {
            const int hh = e >> 7, d = e & 127;
            const float2 *ml = reinterpret_cast<const float2 *>(recv_ml);
            float M = -INFINITY;
            for (int r = 0; r < split; ++r) M = fmaxf(M, ml[r * nh + hh].x);
            float L = 0.0f, acc = 0.0f;
            for (int r = 0; r < split; ++r) {
                const float2 v = ml[r * nh + hh];
                if (v.y > 0.0f) {   // a partial with no visible token has l = 0 and is skipped
                    const float f = exp2f((v.x - M) * p.scale_log2);
                    L = fmaf(f, v.y, L);
                    acc = fmaf(f, recv[(r * nh + hh) * 128 + d], acc);
                }
            }
            const int h = rank * nh + hh;
            out[h * 128 + d] = L > 0.0f ? acc / L : 0.0f;
            if (lse && d == 0) lse[h] = L > 0.0f ? p.scale * M + logf(L) : -INFINITY;
        }
    }
}

template <int Bytes, bool F16>
qsa_status launch_with(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const AttnParams &ap,
                       int grid, cudaStream_t s) {
    static std::mutex mu;
    static bool opted_in[64] = {false};
    int dev = 0;
    qsa_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != QSA_OK) return st;
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!opted_in[dev]) {
            st = check_cuda(cudaFuncSetAttribute(sel_attn_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemOneBytes),
                            "cudaFuncSetAttribute(selection attention)");
            if (st != QSA_OK) return st;
            opted_in[dev] = true;
        }
    }
    // Always a programmatic dependent: behind a top-k that allows it, the CTAs launch
    // while the top-k finishes and wait at entry; behind any other work they launch when
    // it completes, as without the attribute.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)ap.split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ap.split > 1 ? 2 : 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, sel_attn_kernel<F16>, mq, mk, mv, ap), "sel_attn_kernel launch");
}

}  // namespace

qsa_status launch_select_attention(const AttnArgs &a, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    qsa_status st = get_map(&mq, a.qa, 2, QSA_HEAD_DIM, (uint64_t)a.nq * a.n_heads, kG);
    if (st != QSA_OK) return st;
    st = get_map(&mk, a.kcache, 2, QSA_HEAD_DIM, (uint64_t)a.n_kv_heads * a.capacity, 64);
    if (st != QSA_OK) return st;
    st = get_map(&mv, a.vcache_t, 2, 64, (uint64_t)a.n_kv_heads * a.capacity * 2, 128);
    if (st != QSA_OK) return st;
    AttnParams ap{};
    ap.ids = a.ids;
    ap.n_tokens = a.n_tokens;
    ap.out = a.out;
    ap.lse = a.lse;
    ap.flags = a.flags;
    ap.n_heads = a.n_heads;
    ap.n_kv = a.n_kv_heads;
    ap.k = a.k;
    ap.capacity = a.capacity;
    ap.nb_cap = a.capacity / 64;
    ap.scale = a.scale;
    ap.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
    // Few (query, KV head) units (a decode window): split each unit's pairs over a
    // cluster of up to 8 CTAs, doubling while the grid stays within two CTAs per SM
    // (clusters of 16, measured on the 3-query decode window, start further apart and
    // finish later).
    const int units = a.nq * a.n_kv_heads;
    const int pairs = (a.k + 1) / 2;
    ap.split = 1;
    while (ap.split < kMaxSplit && ap.split * 2 <= pairs && (long)units * ap.split * 2 <= 2L * num_sms())
        ap.split *= 2;
    const int grid = units * ap.split;
    // more than 32 blocks in one CTA can take all 512 TMEM columns: one CTA per SM
    const bool alone = a.k > 32 && ap.split == 1;
    if (a.dt == QSA_F16)
        return alone ? launch_with<kSmemOneBytes, true>(mq, mk, mv, ap, grid, s)
                     : launch_with<kSmemBytes, true>(mq, mk, mv, ap, grid, s);
    return alone ? launch_with<kSmemOneBytes, false>(mq, mk, mv, ap, grid, s)
                 : launch_with<kSmemBytes, false>(mq, mk, mv, ap, grid, s);
}

}  // namespace qsa
