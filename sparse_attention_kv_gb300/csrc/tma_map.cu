// tma_map.cu -- host side of the TMA tensor loads: 2-D tensor maps of fp32, bf16
// or 8-bit elements with a 128-byte swizzle (the shared-memory layout the tcgen05
// descriptors expect), encoded through the driver entry point and cached per
// (pointer, shape, element size, device).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qsa_internal.h"

namespace qsa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct MapKey {
    const void *ptr;
    uint32_t inner;
    uint64_t rows;
    uint32_t box_rows;
    int esize;
    int dev;
    bool operator==(const MapKey &o) const {
        return ptr == o.ptr && inner == o.inner && rows == o.rows && box_rows == o.box_rows && esize == o.esize &&
               dev == o.dev;
    }
};

}  // namespace

// Small cache of encoded tensor maps (a map is 128 bytes of host data).
qsa_status get_map(CUtensorMap *out, const void *ptr, int esize, uint32_t inner, uint64_t rows, uint32_t box_rows) {
    static std::mutex mu;
    static MapKey keys[32];
    static CUtensorMap maps[32];
    static int used = 0, next = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const MapKey key{ptr, inner, rows, box_rows, esize, dev};
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (keys[i] == key) {
                *out = maps[i];
                return QSA_OK;
            }
    }
    auto fn = encode_fn();
    if (!fn) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    if (esize != 1 && esize != 2 && esize != 4) return fail(QSA_ERR_INVALID_ARG, "element size %d", esize);
    const cuuint64_t strides[1] = {(cuuint64_t)inner * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / esize), box_rows};
    const CUtensorMapDataType dtype = esize == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                      : esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    const CUresult r = fn(&m, dtype, 2,
                          const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    {
        std::lock_guard<std::mutex> lock(mu);
        keys[next] = key;
        maps[next] = m;
        next = (next + 1) % 32;
        if (used < 32) ++used;
    }
    *out = m;
    return QSA_OK;
}

}  // namespace qsa
