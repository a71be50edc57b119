// topk_static.cu -- the block top-k for callers that cannot allocate device memory.
//
// Some callers of this library have no way to call cudaMalloc at the point where
// they select blocks: code running inside a pre-planned memory arena that may not
// grow, plug-ins handed only the input and output buffers, or environments where a
// device allocation on the serving path is forbidden.  qsa_block_topk needs a
// caller-owned workspace; qsa_block_topk_static instead uses a fixed scratch
// array compiled into the library, so its callers pass only inputs and outputs.
//
// The scratch is a file-scope device array of kStaticScratchBytes bytes; every
// GPU that loads the library holds it until the process exits.  Host code cannot
// hand the array's name to a kernel (on the host it is only a stand-in for the
// device symbol), so the first call on each device looks the device address up
// with cudaGetSymbolAddress, with that device current, and caches it (again after
// the device's context has been replaced, e.g. by cudaDeviceReset).  That first
// call therefore makes a runtime query and should come before any stream
// capture.  Every call shares the one array and leaves its contents behind; the
// parts that must start at zero are cleared on the caller's stream at the start
// of each call, and calls that can overlap on the GPU (two streams, or two host
// threads) race on the array.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    });
    return fn;
}

// Device address of g_static_scratch on the current device, looked up once per
// device and context: a context that replaced the one of the cached address (after
// cudaDeviceReset, say) has the module loaded elsewhere, so it is looked up again.
qsa_status static_scratch(void **out) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    static CUcontext ctx_of[64] = {nullptr};
    int dev = 0;
    qsa_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != QSA_OK) return st;
    if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    auto get_ctx = ctx_get_current();
    if (!get_ctx) return fail(QSA_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
    // null while this thread has no current context yet: then the symbol query below
    // sets the runtime's context up and the address is looked up again
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !ctx || ctx_of[dev] != ctx) {
        void *p = nullptr;
        st = check_cuda(cudaGetSymbolAddress(&p, g_static_scratch), "cudaGetSymbolAddress(static scratch)");
        if (st != QSA_OK) return st;
        if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return QSA_OK;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" qsa_status qsa_block_topk_static(const float *scores, int64_t scores_stride, const int32_t *n_blocks,
                                            int nq, int max_blocks, int active_blocks, int k, int32_t *ids,
                                            qsa_path path, qsa_stream stream) {
    // every argument is checked before the shared scratch is touched: a rejected call
    // enqueues nothing, not even the clear
    if (nq < 1 || max_blocks < 1 || max_blocks > QSA_MAX_BLOCKS || k < 1 || k > QSA_MAX_K)
        return fail(QSA_ERR_INVALID_ARG, "bad sizes (nq %d, max_blocks %d, k %d)", nq, max_blocks, k);
    if (active_blocks < -1)
        return fail(QSA_ERR_INVALID_ARG, "active_blocks must be -1 or >= 0 (got %d)", active_blocks);
    if (!scores || !n_blocks || !ids) return fail(QSA_ERR_INVALID_ARG, "NULL scores, n_blocks or ids");
    if (scores_stride < max_blocks)
        return fail(QSA_ERR_INVALID_ARG, "scores_stride %lld < max_blocks %d", (long long)scores_stride,
                    max_blocks);
    if (path < QSA_PATH_AUTO || path > QSA_PATH_WARP) return fail(QSA_ERR_INVALID_ARG, "bad path %d", (int)path);
    const WsLayout L = ws_layout(nq, max_blocks, k);
    if (L.total > kStaticScratchBytes)
        return fail(QSA_ERR_WORKSPACE,
                    "nq %d, max_blocks %d, k %d need %zu bytes of scratch; the static scratch holds %zu "
                    "(use qsa_block_topk with a workspace)",
                    nq, max_blocks, k, L.total, kStaticScratchBytes);
    void *ws = nullptr;
    qsa_status st = static_scratch(&ws);
    if (st != QSA_OK) return st;
    // flags word and last-CTA tickets must start at zero; the rest is written before it is read
    st = check_cuda(cudaMemsetAsync(ws, 0, L.qflags, static_cast<cudaStream_t>(stream)),
                    "cudaMemsetAsync(static scratch)");
    if (st != QSA_OK) return st;
    return qsa_block_topk(scores, scores_stride, n_blocks, nq, max_blocks, active_blocks, k, ids, ws,
                          kStaticScratchBytes, path, stream);
}
