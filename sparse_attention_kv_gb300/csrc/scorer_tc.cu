// scorer_tc.cu -- indexer block scorer on the 5th-generation tensor cores.
//
//   score[q][b] = sum_h w[q][h] * relu(dot(q[q][h][:], kblk[b][:]))
//
// The contraction is the GEMM of "#1091 qsa_select: FP32 tiled block scores
// below sm_80" (section "What": rows = query x indexer head, K = 128, the ReLU
// of each head summed per block), laid out for tcgen05: the MMA's M side is 128
// KV blocks (one TMEM lane each), its N side is a group of queries x heads
// (<= 256 columns), K = 128.  One thread of the epilogue owns one block row of
// the accumulator, so the ReLU and the head-weighted sum stay in its registers
// and the score stores of a warp are 32 consecutive blocks.
//
// Per CTA (192 threads): warp 0 issues TMA loads (kblk tiles through a ring of
// shared-memory stages, the query-group tile once), warp 1 owns TMEM and issues
// tcgen05.mma from one thread, warps 2-5 drain the double-buffered accumulator
// (tcgen05.ld) and write the scores.  bf16 inputs use kind::f16 (bf16 x bf16 ->
// fp32); fp8 e4m3 inputs use kind::f8f6f4 (e4m3 x e4m3 -> fp32, the 128 elements
// of K in one 128-byte swizzle atom).  fp32 inputs use kind::tf32 on a three-term split a = a_hi + a_lo
// (a_hi = a with the low 13 mantissa bits cleared): a_hi*b_hi + a_hi*b_lo +
// a_lo*b_hi, which keeps the product error near 2^-20 relative.
//
// The partial tail block of a context is a key row like any other; rows at or
// past n_blocks[q] are computed but not stored, rows past the capacity are
// zero-filled by TMA.  Every wait on an mbarrier is bounded; on expiry the CTA
// raises QSA_FLAG_WAIT_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "qsa_device.cuh"
#include "tc_ptx.cuh"
#include "warp_topk.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kBM = 128;       // KV blocks per tile (MMA M = TMEM lanes)
constexpr int kEpiParts = 4;                  // epilogue warps per TMEM lane quarter
constexpr int kEpi = 128 * kEpiParts;         // epilogue threads
constexpr int kThreads = 64 + kEpi;           // + one TMA warp and one MMA warp
constexpr int kMaxChunks = (16 + kEpiParts - 1) / kEpiParts;  // 16-column chunks per thread
constexpr int kFusedMaxQ = 16;                // queries per group of the fused kernel (scores kept on chip)

template <int DT>
struct Cfg;
template <>
struct Cfg<QSA_BF16> {  // bf16 -> kind::f16
    static constexpr int kEsize = 2, kEPA = 64, kAtoms = 2, kStages = 4, kMaxBN = 256;
    static constexpr uint32_t kFmt = 1;
    static constexpr MmaKind kKind = MmaKind::f16;
};
template <>
struct Cfg<QSA_F32> {  // fp32 -> kind::tf32, three-term split
    static constexpr int kEsize = 4, kEPA = 32, kAtoms = 4, kStages = 1, kMaxBN = 64;
    static constexpr uint32_t kFmt = 2;
    static constexpr MmaKind kKind = MmaKind::tf32;
};
template <>
struct Cfg<QSA_E4M3> {  // fp8 e4m3 -> kind::f8f6f4, K = 128 in one 128-byte atom
    static constexpr int kEsize = 1, kEPA = 128, kAtoms = 1, kStages = 4, kMaxBN = 256;
    static constexpr uint32_t kFmt = 0;
    static constexpr MmaKind kKind = MmaKind::f8f6f4;
};

// One 128-byte swizzle atom of a tile holds rows x 128 bytes (kEPA elements of K).
constexpr int kAtomA = kBM * 128;  // 16 KB

// The fused kernel keeps each CTA's scores on chip (kSbuf bytes) and gives each
// epilogue warp a 256-bin histogram; it pays for them with fewer kblk stages.
template <int DT, bool FUSED>
struct Layout {
    using C = Cfg<DT>;
    static constexpr bool kF32 = DT == QSA_F32;
    static constexpr int kStages = (FUSED && !kF32) ? 2 : C::kStages;
    static constexpr int kB = C::kAtoms * C::kMaxBN * 128;
    static constexpr int kAStage = C::kAtoms * kAtomA;
    static constexpr int offB = 0;
    static constexpr int offBlo = offB + kB;
    static constexpr int offA = offBlo + (kF32 ? kB : 0);
    static constexpr int offAlo = offA + kStages * kAStage;
    static constexpr int offCtrl = offAlo + (kF32 ? kStages * kAStage : 0);
};
constexpr int kHistBytes = (kEpi / 32) * 256 * 4;   // one 256-bin histogram per epilogue warp

struct Ctrl {
    uint64_t full[4], empty[4], split[4];
    uint64_t bfull, bsplit, done;
    uint64_t tfull[2], tempty[2];
    uint32_t tmem_base;
    int abort;
    int last;
    __align__(16) float w[256];
    int nb[256];
    uint64_t top[kEpi / 32][32];   // fused form: an epilogue warp's exact top k (k <= 32)
};

template <int DT, bool FUSED>
constexpr int sbuf_bytes() {
    return FUSED ? (227 * 1024 - 1024 - Layout<DT, FUSED>::offCtrl - (int)sizeof(Ctrl) - kHistBytes) / 1024 * 1024 : 0;
}
template <int DT, bool FUSED>
constexpr int smem_bytes() {
    return Layout<DT, FUSED>::offCtrl + (int)sizeof(Ctrl) + (FUSED ? kHistBytes + sbuf_bytes<DT, FUSED>() : 0) + 1024;
}

struct KParams {
    const float *w;
    const int32_t *n_blocks;
    float *scores;
    int64_t stride;
    uint32_t *flags;
    int nq, bound, qg, bn, tiles_per_cta, tiles_total, tmem_cols;
    // fused score-then-select only: each CTA's candidate lists, [cpg][nq][kslot] scores and
    // global ids, and their lengths counts[q * maxch + CTA]
    int k;
    float *cand_scores;
    int32_t *cand_ids;
    int32_t *counts;
    int kslot;
    int maxch;
    int sb_stride;     // scores per query in the on-chip buffer (tiles_per_cta * 128)
};

// sum_h w[h] * relu(acc[h]) for one query, in fp32: ReLU per head, then the
// products added in two interleaved partial sums (packed two-wide FMA) that
// are combined at the end.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
template <int H>
__device__ __forceinline__ float head_sum(const float *w, const uint32_t *acc) {
    if constexpr (H >= 4) {
        uint64_t s = 0;   // (0.0f, 0.0f)
#pragma unroll
        for (int h = 0; h < H; h += 4) {
            const float4 wv = *reinterpret_cast<const float4 *>(w + h);
            const float r0 = fmaxf(__uint_as_float(acc[h + 0]), 0.0f);
            const float r1 = fmaxf(__uint_as_float(acc[h + 1]), 0.0f);
            const float r2 = fmaxf(__uint_as_float(acc[h + 2]), 0.0f);
            const float r3 = fmaxf(__uint_as_float(acc[h + 3]), 0.0f);
            s = fma2(pack2(wv.x, wv.y), pack2(r0, r1), s);
            s = fma2(pack2(wv.z, wv.w), pack2(r2, r3), s);
        }
        float a, b;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(s));
        return a + b;
    } else {
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < H; ++h) s = fmaf(w[h], fmaxf(__uint_as_float(acc[h]), 0.0f), s);
        return s;
    }
}


// a = hi + lo with hi = a truncated to tf32 (exact split), in place for hi.
__device__ __forceinline__ void split_tf32(uint8_t *buf, uint8_t *lo, int bytes, int tid, int nthreads) {
    uint4 *p = reinterpret_cast<uint4 *>(buf);
    uint4 *l = reinterpret_cast<uint4 *>(lo);
    for (int i = tid; i < bytes / 16; i += nthreads) {
        uint4 x = p[i], h, r;
        h.x = x.x & 0xFFFFE000u;
        h.y = x.y & 0xFFFFE000u;
        h.z = x.z & 0xFFFFE000u;
        h.w = x.w & 0xFFFFE000u;
        r.x = __float_as_uint(__uint_as_float(x.x) - __uint_as_float(h.x));
        r.y = __float_as_uint(__uint_as_float(x.y) - __uint_as_float(h.y));
        r.z = __float_as_uint(__uint_as_float(x.z) - __uint_as_float(h.z));
        r.w = __float_as_uint(__uint_as_float(x.w) - __uint_as_float(h.w));
        p[i] = h;
        l[i] = r;
    }
}

// ---------------------------------------------------------------- fused select

// The selection step of the fused kernel, stage A.  For each query j of the group
// (epilogue warp j, j + 16, ...), this CTA's blocks of it are on chip; they are
// reduced to a list that holds every block of the query's selection among them,
// written to the workspace as (score, global id) with its length.  The merge kernel
// launched after this one selects over every CTA's lists.  A query's selection
// restricted to one CTA's blocks is a prefix of that range's order (the split of
// Strata PR #3987, section "Approach"), so a list holding the range's k best is
// enough:
//  * at most kslot blocks: all of them;
//  * k <= 32: the scores at or above the k-th largest of the lanes' maxima (k
//    distinct entries reach it; about 120 of 1,024 on continuous scores), unranked --
//    the one-read filter of "#2093 sm_75: the prompt path's top-k with one full
//    read of the scores" (steps 2-3) with the bound taken from the chunk itself;
//  * more survivors than kslot (heavy ties), or k > 32: the range's exact top k.
__device__ __noinline__ void fused_stage_a(const KParams &p, Ctrl &ct, float *sbuf, uint32_t *hist, int q0, int qv,
                                           int t_begin, int ntiles) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ew = warp - 2;   // epilogue warp index
    if (ew < 0) return;        // the TMA and MMA warps have no part here
    constexpr int nw = kEpi / 32;
    const int c = blockIdx.x;
    // the parameters live in memory that the stores below could alias: read them once
    const int k = p.k, kslot = p.kslot, nq = p.nq, sb_stride = p.sb_stride, maxch = p.maxch;
    float *const __restrict__ cs = p.cand_scores;
    int32_t *const __restrict__ ci = p.cand_ids;
    int32_t *const __restrict__ counts = p.counts;
    uint32_t *h = hist + ew * 256;                        // 1 KB: 64-entry rank buffer or a histogram
    uint64_t *buf = reinterpret_cast<uint64_t *>(h);
    uint64_t *top = ct.top[ew];
    const float ninf = __int_as_float(0xff800000);
    const int lo = t_begin * kBM;
    for (int j = ew; j < qv; j += nw) {
        const int q = q0 + j;
        const int nloc = max(0, min(ntiles * kBM, ct.nb[j] - lo));
        const size_t base = ((size_t)c * nq + q) * kslot;
        float *row = sbuf + (size_t)j * sb_stride;   // this CTA's blocks of query j
        int count = -1;
        if (nloc <= kslot) {
            for (int i = lane; i < nloc; i += 32) {
                cs[base + i] = row[i];
                ci[base + i] = lo + i;
            }
            count = nloc;
        } else if (k <= 32 && nloc <= 1024) {
            // lane l holds entries l + 32 t; at least k lanes hold one (nloc > kslot >= k),
            // the others read -inf
            float x[32];
            float mx = ninf;
#pragma unroll
            for (int t = 0; t < 32; ++t) x[t] = row[min(lane + 32 * t, nloc - 1)];   // nloc > kslot >= 1
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                if (lane + 32 * t >= nloc) x[t] = ninf;
                mx = fmaxf(mx, x[t]);
            }
            uint32_t kk = score_key(mx), bk;
            if (k == 32) {
                bk = __reduce_min_sync(kFull, kk);
            } else {
                bk = 0u;
                for (int it = 0; it < k; ++it) {
                    bk = __reduce_max_sync(kFull, kk);
                    const unsigned win = __ballot_sync(kFull, kk == bk);
                    if (lane == __ffs(win) - 1) kk = 0u;   // 0 is below every score's key
                }
            }
            // each lane counts its survivors, a scan over the lanes places them, and
            // each lane writes its own run (no vote inside the loop)
            const float bf = key_float(bk);
            int cnt = 0;
#pragma unroll
            for (int t = 0; t < 32; ++t) cnt += (lane + 32 * t < nloc && x[t] >= bf) ? 1 : 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += v;
            }
            const int total = __shfl_sync(kFull, incl, 31);
            if (total <= kslot) {
                int at = incl - cnt;
                if (2 * total <= sb_stride) {
                    // the row is in registers: its shared copy holds the list (scores,
                    // then ids), written to the workspace in whole lines
                    float *st = row;
                    int32_t *sti = reinterpret_cast<int32_t *>(row + total);
                    __syncwarp();
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int i = lane + 32 * t;
                        if (i < nloc && x[t] >= bf) {
                            st[at] = x[t];
                            sti[at] = lo + i;
                            ++at;
                        }
                    }
                    __syncwarp();
                    for (int e = lane; e < total; e += 32) {
                        cs[base + e] = st[e];
                        ci[base + e] = sti[e];
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int i = lane + 32 * t;
                        if (i < nloc && x[t] >= bf) {
                            cs[base + at] = x[t];
                            ci[base + at] = lo + i;
                            ++at;
                        }
                    }
                }
                count = total;
            }
        }
        if (count < 0) {   // the range's exact top k
            bool ok = false;
            if (k <= 32) {
                if (nloc <= 128) ok = stage_a_regs<1>(row, nloc, k, lo, buf, top);
                else if (nloc <= 256) ok = stage_a_regs<2>(row, nloc, k, lo, buf, top);
                else if (nloc <= 512) ok = stage_a_regs<4>(row, nloc, k, lo, buf, top);
                else if (nloc <= 1024) ok = stage_a_regs<8>(row, nloc, k, lo, buf, top);
                else ok = stage_a_smem(row, nloc, k, lo, buf, top);
                if (ok) {
                    __syncwarp();
                    if (lane < k) {
                        cs[base + lane] = key_float(cand_key(top[lane]));
                        ci[base + lane] = cand_id(top[lane]);
                    }
                }
            }
            if (!ok) {   // heavy ties, or k > 32: the radix warp select over the range
                for (int i = lane; i < 256; i += 32) h[i] = 0u;
                __syncwarp();
                warp_select([&](int i) { return score_key(row[i]); }, nloc, k, h, [&](int at, int i) {
                    cs[base + at] = row[i];
                    ci[base + at] = lo + i;
                });
            }
            count = k;
        }
        __syncwarp();
        if (lane == 0) counts[(size_t)q * maxch + c] = count;
    }
}

// ---------------------------------------------------------------- kernel

template <int DT, int H, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    scorer_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const KParams p) {
    using C = Cfg<DT>;
    using L = Layout<DT, FUSED>;
    constexpr bool F32 = DT == QSA_F32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sB = smem + L::offB;
    uint8_t *sBlo = smem + L::offBlo;
    uint8_t *sA = smem + L::offA;
    uint8_t *sAlo = smem + L::offAlo;
    Ctrl &ct = *reinterpret_cast<Ctrl *>(smem + L::offCtrl);
    volatile int *abort_flag = &ct.abort;
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + L::offCtrl + sizeof(Ctrl));       // FUSED only
    float *sbuf = reinterpret_cast<float *>(smem + L::offCtrl + sizeof(Ctrl) + kHistBytes);  // FUSED only

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A dependent grid (the top-k of a chained select) launches once every CTA of this
    // grid has executed this or exited, so no scorer CTA is still waiting for an SM
    // when top-k CTAs take free ones; they wait at entry until this grid completes.
    // This grid is itself launched as a programmatic dependent of the work before it:
    // its CTAs may be scheduled while that work drains, and each waits here, before it
    // takes tensor memory or reads or writes anything, until that work has completed.
    allow_dependent_launch();
    wait_prior_grid();
    const int g = blockIdx.y;
    const int q0 = g * p.qg;
    const int qv = min(p.qg, p.nq - q0);  // queries of this group
    const int bn = p.bn;

    const int t_begin = blockIdx.x * p.tiles_per_cta;
    const int t_cap = min(p.tiles_per_cta, p.tiles_total - t_begin);  // tiles under the bound

    // TMEM first (warp 1), while the barriers are set up: nothing the MMA warp needs
    // waits for the reads of w and n_blocks, which only the epilogue uses
    if (warp == 1 && t_cap > 0) {
        tmem_alloc(&ct.tmem_base, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&ct.full[s], 1);
            mbar_init(&ct.empty[s], 1);
            mbar_init(&ct.split[s], kEpi);
        }
        mbar_init(&ct.bfull, 1);
        mbar_init(&ct.bsplit, kEpi);
        mbar_init(&ct.done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ct.tfull[b], 1);
            mbar_init(&ct.tempty[b], kEpi / 32);
        }
        ct.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The query tile and the first stages are requested at once.  The tiles run to the
    // host-visible bound: the TMA and MMA warps never wait for n_blocks, and the
    // epilogue stores only the rows below each query's count.
    const int ntiles = t_cap;
    int issued = 0;
    if (tid == 0 && ntiles > 0) {
        mbar_expect_tx(&ct.bfull, (uint32_t)(C::kAtoms * bn * 128));
        for (int a = 0; a < C::kAtoms; ++a)
            tma_load_2d(sB + a * bn * 128, &tm_q, &ct.bfull, a * C::kEPA, q0 * H);
        const int pre = min(L::kStages, ntiles);
        for (int i = 0; i < pre; ++i) {
            mbar_expect_tx(&ct.full[i], (uint32_t)(C::kAtoms * kAtomA));
            for (int a = 0; a < C::kAtoms; ++a)
                tma_load_2d(sA + i * L::kAStage + a * kAtomA, &tm_k, &ct.full[i], a * C::kEPA, (t_begin + i) * kBM);
        }
        issued = pre;
    }
    if (ntiles <= 0) {
        // no tile under the bound (fused form, empty contexts): the block counts for its
        // selection step
        for (int j = tid; j < qv; j += kThreads) {
            int n = p.n_blocks[q0 + j];
            if (n < 0 || n > p.bound) {
                if (p.flags && blockIdx.x == 0) atomicOr(p.flags, QSA_FLAG_NBLOCKS_CLAMPED);
                n = n < 0 ? 0 : p.bound;
            }
            ct.nb[j] = n;
        }
        __syncthreads();
    } else {
    const uint32_t tmem = ct.tmem_base;
    const int buf_cols = p.tmem_cols / 2;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer (tiles after the early ones)
            for (int i = issued; i < ntiles; ++i) {
                const int s = i % L::kStages;
                const uint32_t ph = (uint32_t)(i / L::kStages) & 1u;
                if (!mbar_wait(&ct.empty[s], ph ^ 1u, abort_flag)) break;
                mbar_expect_tx(&ct.full[s], (uint32_t)(C::kAtoms * kAtomA));
                const int row = (t_begin + i) * kBM;
                for (int a = 0; a < C::kAtoms; ++a)
                    tma_load_2d(sA + s * L::kAStage + a * kAtomA, &tm_k, &ct.full[s], a * C::kEPA, row);
                ++issued;
            }
            // drain: the latest load of every stage and the query tile
            for (int j = max(0, issued - L::kStages); j < issued; ++j)
                mbar_drain(&ct.full[j % L::kStages], (uint32_t)(j / L::kStages) & 1u);
            mbar_drain(&ct.bfull, 0);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t id = idesc(C::kFmt, kBM, bn);
            // Every descriptor is its stage's or the query tile's base plus a constant
            // (start addresses in 16-byte units, all below 2^14): this warp shares its
            // scheduler with busy epilogue warps, so each MMA costs it a few integer adds.
            uint64_t db[C::kAtoms * 4], dbl[F32 ? C::kAtoms * 4 : 1];
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    db[a * 4 + kk] = sdesc(smem_u32(sB) + (uint32_t)(a * bn * 128 + kk * 32));
                    if constexpr (F32) dbl[a * 4 + kk] = sdesc(smem_u32(sBlo) + (uint32_t)(a * bn * 128 + kk * 32));
                }
            bool ok = mbar_wait(F32 ? &ct.bsplit : &ct.bfull, 0, abort_flag);
            tc_fence_after();
            for (int i = 0; ok && i < ntiles; ++i) {
                const int s = i % L::kStages;
                const uint32_t ph = (uint32_t)(i / L::kStages) & 1u;
                const int b = i & 1;
                const uint32_t tph = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(&ct.tempty[b], tph ^ 1u, abort_flag)) break;
                if (!mbar_wait(F32 ? &ct.split[s] : &ct.full[s], ph, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * buf_cols);
                const uint64_t da = sdesc(smem_u32(sA + s * L::kAStage));
                const uint64_t dal = F32 ? sdesc(smem_u32(sAlo + s * L::kAStage)) : 0ull;
#pragma unroll
                for (int a = 0; a < C::kAtoms; ++a) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t aoff = (uint64_t)((a * kAtomA + kk * 32) >> 4);
                        const uint32_t acc = (a | kk) != 0 ? 1u : 0u;
                        mma<C::kKind>(d, da + aoff, db[a * 4 + kk], id, acc);
                        if constexpr (F32) {
                            mma<C::kKind>(d, da + aoff, dbl[a * 4 + kk], id, 1u);
                            mma<C::kKind>(d, dal + aoff, db[a * 4 + kk], id, 1u);
                        }
                    }
                }
                mma_commit(&ct.empty[s]);
                mma_commit(&ct.tfull[b]);
            }
            // every MMA issued so far has completed once this arrives
            mma_commit(&ct.done);
            mbar_drain(&ct.done, 0);
        }
    } else {
        // ---------------- epilogue: warps 2.., one accumulator row per thread.
        // The kEpiParts warps of a TMEM lane quarter (warp % 4) split the tile's
        // 16-column chunks (16/H queries each) between them.
        const int et = tid - 64;                 // 0..511
        // the group's weights and block counts (clamped), for the epilogue warps only
        for (int i = et; i < qv * H; i += kEpi) ct.w[i] = p.w[(size_t)q0 * H + i];
        for (int j = et; j < qv; j += kEpi) {
            int n = p.n_blocks[q0 + j];
            if (n < 0 || n > p.bound) {
                if (p.flags && blockIdx.x == 0) atomicOr(p.flags, QSA_FLAG_NBLOCKS_CLAMPED);
                n = n < 0 ? 0 : p.bound;
            }
            ct.nb[j] = n;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory");
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int part = (warp - 2) >> 2;        // 0..kEpiParts-1
        const int row = quarter * 32 + lane;
        const int nchunk = (qv * H + 15) / 16;   // <= 16
        const int c_begin = part * nchunk / kEpiParts;
        const int c_end = (part + 1) * nchunk / kEpiParts;
        bool ok = true;
        if constexpr (F32) {
            ok = __all_sync(0xffffffffu, mbar_wait(&ct.bfull, 0, abort_flag));
            if (ok) split_tf32(sB, sBlo, C::kAtoms * bn * 128, et, kEpi);
            fence_proxy_async();
            mbar_arrive(&ct.bsplit);
        }
        for (int i = 0; ok && i < ntiles; ++i) {
            if constexpr (F32) {
                const int s = i % L::kStages;
                const uint32_t ph = (uint32_t)(i / L::kStages) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&ct.full[s], ph, abort_flag))) break;
                split_tf32(sA + s * L::kAStage, sAlo + s * L::kAStage, L::kAStage, et, kEpi);
                fence_proxy_async();
                mbar_arrive(&ct.split[s]);
            }
            const int b = i & 1;
            const uint32_t tph = (uint32_t)(i >> 1) & 1u;
            // Lane 0 of each warp waits for the accumulator (a suspending try-wait)
            // and the warp goes on by itself: no epilogue-wide barrier per tile, so a
            // slow warp delays only its own share.
            int acc_ok = 0;
            if (lane == 0) acc_ok = mbar_wait(&ct.tfull[b], tph, abort_flag) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, acc_ok, 0)) break;
            tc_fence_after();
            const int blk = (t_begin + i) * kBM + row;
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * buf_cols);
            // every column chunk of this thread's part in flight at once, one wait; a
            // full part (64 columns) in one load, which reads TMEM faster than four
            const int nc = c_end - c_begin;   // <= kMaxChunks
            uint32_t v[kMaxChunks][16];
            static_assert(kMaxChunks == 4, "one 64-column load per full part");
            if (nc == kMaxChunks) {
                tmem_ld64_nowait(taddr + (uint32_t)(c_begin * 16), v);
            } else {
#pragma unroll
                for (int cc = 0; cc < kMaxChunks; ++cc)
                    if (cc < nc) tmem_ld16_nowait(taddr + (uint32_t)((c_begin + cc) * 16), v[cc]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < kMaxChunks; ++cc)
                if (cc < nc) reg_fence(v[cc]);
            // the accumulators are in registers: the buffer goes back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ct.tempty[b]);
#pragma unroll
            for (int cc = 0; cc < kMaxChunks; ++cc) {
                if (cc < nc) {
#pragma unroll
                    for (int jj = 0; jj < 16 / H; ++jj) {
                        const int j = (c_begin + cc) * (16 / H) + jj;
                        if (j < qv) {
                            const float sc = head_sum<H>(&ct.w[j * H], &v[cc][jj * H]);
                            if (FUSED) sbuf[j * p.sb_stride + i * kBM + row] = sc;
                            if ((!FUSED || p.scores) && blk < ct.nb[j])
                                p.scores[(size_t)(q0 + j) * p.stride + blk] = sc;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
    }
    }  // ntiles > 0
    if (tid == 0 && ct.abort && p.flags) atomicOr(p.flags, QSA_FLAG_WAIT_TIMEOUT);
    if constexpr (FUSED) fused_stage_a(p, ct, sbuf, hist, q0, qv, t_begin, max(ntiles, 0));
}

// ---------------------------------------------------------------- host side

template <int DT, int H, bool FUSED>
qsa_status launch_typed(const CUtensorMap &mk, const CUtensorMap &mq, const KParams &kp, dim3 grid,
                        cudaStream_t s) {
    constexpr int bytes = smem_bytes<DT, FUSED>();
    static_assert(bytes <= 227 * 1024, "scorer shared memory");
    // the shared-memory opt-in is a per-device property of the function: set it once on
    // every device this instantiation launches on
    static std::mutex mu;
    static bool opted_in[64] = {false};
    int dev = 0;
    qsa_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != QSA_OK) return st;
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!opted_in[dev]) {
            st = check_cuda(cudaFuncSetAttribute(scorer_tc_kernel<DT, H, FUSED>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                            "cudaFuncSetAttribute(scorer)");
            if (st != QSA_OK) return st;
            opted_in[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, scorer_tc_kernel<DT, H, FUSED>, mk, mq, kp),
                      FUSED ? "fused scorer+select launch" : "scorer_tc_kernel launch");
}

template <int DT, bool FUSED>
qsa_status launch_heads(int H, const CUtensorMap &mk, const CUtensorMap &mq, const KParams &kp, dim3 grid,
                        cudaStream_t s) {
    switch (H) {
    case 1: return launch_typed<DT, 1, FUSED>(mk, mq, kp, grid, s);
    case 2: return launch_typed<DT, 2, FUSED>(mk, mq, kp, grid, s);
    case 4: return launch_typed<DT, 4, FUSED>(mk, mq, kp, grid, s);
    case 8: return launch_typed<DT, 8, FUSED>(mk, mq, kp, grid, s);
    case 16: return launch_typed<DT, 16, FUSED>(mk, mq, kp, grid, s);
    default: return fail(QSA_ERR_INVALID_ARG, "n_heads %d", H);
    }
}

}  // namespace

qsa_status launch_scorer(const ScorerArgs &a, cudaStream_t s) {
    const int dt = a.dt;
    const int H = a.n_heads;
    const int max_bn = dt == QSA_F32 ? Cfg<QSA_F32>::kMaxBN : dt == QSA_E4M3 ? Cfg<QSA_E4M3>::kMaxBN : Cfg<QSA_BF16>::kMaxBN;
    const int tiles = (a.bound + kBM - 1) / kBM;
    if (tiles == 0 && !a.fused) return QSA_OK;   // no block can be valid
    const int sms = num_sms();
    const int t1 = std::max(tiles, 1);
    // queries per group: as many as fill the MMA's N side; the fused kernel keeps at
    // most 16 on chip and fewer when their scores would not fit.  Its CTAs' candidate
    // lists (kslot slots each) share the workspace's candidate arrays, and the merge
    // holds the cpg lists of a query on chip.
    int qg = std::min(a.nq, std::max(1, a.fused ? std::min(max_bn / H, kFusedMaxQ) : max_bn / H));
    int groups = 0, cpg = 0, tpc = 0, kslot = 0;
    for (;; qg = (qg + 1) / 2) {
        groups = (a.nq + qg - 1) / qg;
        cpg = std::max(1, std::min(t1, sms / groups));
        tpc = (t1 + cpg - 1) / cpg;
        if (!a.fused) break;
        const int sbuf = dt == QSA_F32    ? sbuf_bytes<QSA_F32, true>()
                         : dt == QSA_E4M3 ? sbuf_bytes<QSA_E4M3, true>()
                                          : sbuf_bytes<QSA_BF16, true>();
        const int tpc_max = sbuf / (qg * kBM * 4);
        bool fits = tpc_max >= 1;
        if (fits) {
            tpc = std::min(tpc, tpc_max);
            cpg = (t1 + tpc - 1) / tpc;
            if ((long)cpg * a.k > kMergeCap) {   // fewer CTAs per group, more tiles each
                tpc = (t1 + std::max(1, kMergeCap / a.k) - 1) / std::max(1, kMergeCap / a.k);
                cpg = (t1 + tpc - 1) / tpc;
                fits = tpc <= tpc_max;
            }
            kslot = kMergeCap / cpg;   // the fused workspace holds kMergeCap candidates per query
            fits = fits && kslot >= a.k;
        }
        if (fits) break;
        if (qg == 1)
            return fail(QSA_ERR_UNSUPPORTED,
                        "fused select: the per-CTA scores do not fit on chip, or %d CTAs x k = %d candidates exceed "
                        "the merge's %d; use the chained form", cpg, a.k, kMergeCap);
    }
    cpg = (t1 + tpc - 1) / tpc;
    const int bn = (qg * H + 15) / 16 * 16;
    int tmem_cols = 32;
    while (tmem_cols < 2 * bn) tmem_cols *= 2;

    CUtensorMap mk, mq;
    const int esize = dt == QSA_F32 ? 4 : dt == QSA_E4M3 ? 1 : 2;
    qsa_status st = get_map(&mk, a.kblk, esize, QSA_HEAD_DIM, (uint64_t)a.max_blocks, kBM);
    if (st != QSA_OK) return st;
    st = get_map(&mq, a.q, esize, QSA_HEAD_DIM, (uint64_t)a.nq * H, (uint32_t)bn);
    if (st != QSA_OK) return st;

    KParams kp{};
    kp.w = a.w;
    kp.n_blocks = a.n_blocks;
    kp.scores = a.scores;
    kp.stride = a.stride;
    kp.flags = a.flags;
    kp.nq = a.nq;
    kp.bound = a.bound;
    kp.qg = qg;
    kp.bn = bn;
    kp.tiles_per_cta = tpc;
    kp.tiles_total = tiles;
    kp.tmem_cols = tmem_cols;
    kp.k = a.k;
    kp.maxch = a.maxch;
    kp.sb_stride = tpc * kBM;
    kp.cand_scores = a.cand_scores;
    kp.cand_ids = a.cand_ids;
    kp.counts = a.counts;
    kp.kslot = kslot;
    const dim3 grid(cpg, groups);
    switch (dt) {
    case QSA_F32:
        st = a.fused ? launch_heads<QSA_F32, true>(H, mk, mq, kp, grid, s)
                     : launch_heads<QSA_F32, false>(H, mk, mq, kp, grid, s);
        break;
    case QSA_E4M3:
        st = a.fused ? launch_heads<QSA_E4M3, true>(H, mk, mq, kp, grid, s)
                     : launch_heads<QSA_E4M3, false>(H, mk, mq, kp, grid, s);
        break;
    default:
        st = a.fused ? launch_heads<QSA_BF16, true>(H, mk, mq, kp, grid, s)
                     : launch_heads<QSA_BF16, false>(H, mk, mq, kp, grid, s);
        break;
    }
    if (st != QSA_OK || !a.fused) return st;
    // the fused form's last step: one CTA per query selects over its CTAs' lists,
    // launched as a programmatic dependent (its launch overlaps the scorer's work)
    return launch_merge(a.cand_scores, a.cand_ids, a.counts, a.maxch, cpg, a.nq, kslot, a.k, a.ids, s);
}

}  // namespace qsa
