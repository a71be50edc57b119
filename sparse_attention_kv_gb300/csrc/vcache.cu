// vcache.cu -- the V cache layout of the selection attention: each 64-token block
// of a KV head stored dimension-major ([128 dims][64 tokens]), converted from the
// token-row layout ([tokens][128]) one block at a time.
//
// One CTA per (KV head, block): 256 threads read the block's 64 x 128 16-bit
// values as 16-byte vectors (rows of 256 contiguous bytes), hold them in shared
// memory with a padded row pitch, and write the 128 x 64 transpose as 16-byte
// vectors (rows of 128 contiguous bytes).  The values are copied bit for bit.
#include <cstdint>

#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int kTok = 64, kDim = 128;
constexpr int kPitch = kDim + 2;   // 16-bit elements per staged row: the column reads spread over the banks

__global__ void __launch_bounds__(256) vcache_transpose_kernel(const uint16_t *__restrict__ v,
                                                              uint16_t *__restrict__ vt, int capacity,
                                                              int first_block, int n_blocks) {
    __shared__ uint16_t tile[kTok * kPitch];
    const int g = blockIdx.y;
    const int b = first_block + blockIdx.x;
    const int nb_cap = capacity / kTok;
    const uint16_t *src = v + ((size_t)g * capacity + (size_t)b * kTok) * kDim;
    uint16_t *dst = vt + ((size_t)g * nb_cap + b) * (size_t)(kDim * kTok);
    // 64 rows x 16 vectors of 8 values
    for (int e = threadIdx.x; e < kTok * (kDim / 8); e += blockDim.x) {
        const int t = e / (kDim / 8), c = e % (kDim / 8);
        const uint4 x = reinterpret_cast<const uint4 *>(src + (size_t)t * kDim)[c];
        const uint16_t w[8] = {(uint16_t)(x.x & 0xFFFF), (uint16_t)(x.x >> 16), (uint16_t)(x.y & 0xFFFF),
                               (uint16_t)(x.y >> 16),    (uint16_t)(x.z & 0xFFFF), (uint16_t)(x.z >> 16),
                               (uint16_t)(x.w & 0xFFFF), (uint16_t)(x.w >> 16)};
#pragma unroll
        for (int i = 0; i < 8; ++i) tile[t * kPitch + c * 8 + i] = w[i];
    }
    __syncthreads();
    // 128 rows (dims) x 8 vectors of 8 tokens
    for (int e = threadIdx.x; e < kDim * (kTok / 8); e += blockDim.x) {
        const int d = e / (kTok / 8), c = e % (kTok / 8);
        uint16_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = tile[(c * 8 + i) * kPitch + d];
        uint4 x;
        x.x = (uint32_t)w[0] | ((uint32_t)w[1] << 16);
        x.y = (uint32_t)w[2] | ((uint32_t)w[3] << 16);
        x.z = (uint32_t)w[4] | ((uint32_t)w[5] << 16);
        x.w = (uint32_t)w[6] | ((uint32_t)w[7] << 16);
        reinterpret_cast<uint4 *>(dst + (size_t)d * kTok)[c] = x;
    }
}

}  // namespace

qsa_status launch_vcache_transpose(const void *v, void *vcache_t, int n_kv_heads, int capacity, int first_block,
                                   int n_blocks, cudaStream_t s) {
    if (n_blocks == 0) return QSA_OK;
    const dim3 grid((unsigned)n_blocks, (unsigned)n_kv_heads);
    vcache_transpose_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t *>(v), static_cast<uint16_t *>(vcache_t),
                                                capacity, first_block, n_blocks);
    return check_cuda(cudaGetLastError(), "vcache_transpose_kernel launch");
}

}  // namespace qsa
