// copy_blocks.cu -- the device half of copy-on-write: copy whole physical blocks (every KV
// head, K and V) from src to dst so a sequence can write into its own copy of a block it
// shared with others (yangyu.win blog #54, section 5 question 2).
//
// A block of the [num_blocks, Hkv, bs, d] pool is Hkv * bs * d contiguous 16-bit words; each
// thread moves 16-byte vectors, so reads and writes are fully coalesced; each thread has four K and
// four V vectors in flight.
#include "pa_device.cuh"

namespace pa {

constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;                                // K and V vectors in flight per thread
constexpr int COPY_CHUNK = COPY_THREADS * COPY_UNROLL;        // vectors of one work item (16 KB of K, of V)

// Work item = (pair c, chunk k of COPY_CHUNK vectors of its blocks); the grid strides over items.
// Each thread loads its COPY_UNROLL K and V vectors of the item before storing any.
__global__ void __launch_bounds__(COPY_THREADS) copy_blocks_kernel(const int32_t *pairs, int32_t n, uint4 *k_cache,
                                                                   uint4 *v_cache, int64_t vec_per_block,
                                                                   int32_t num_blocks, int *status) {
    const int chunks = (int)((vec_per_block + COPY_CHUNK - 1) / COPY_CHUNK);
    const int64_t items = (int64_t)n * chunks;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int c = (int)(item / chunks);
        const int k = (int)(item - (int64_t)c * chunks);
        const int32_t src = __ldg(pairs + 2 * c), dst = __ldg(pairs + 2 * c + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (k == 0 && threadIdx.x == 0) set_status(status, STATUS_BOUNDS);
            continue;
        }
        const uint4 *ks = k_cache + (int64_t)src * vec_per_block, *vs = v_cache + (int64_t)src * vec_per_block;
        uint4 *kd = k_cache + (int64_t)dst * vec_per_block, *vd = v_cache + (int64_t)dst * vec_per_block;
        const int64_t v0 = (int64_t)k * COPY_CHUNK + threadIdx.x;
        uint4 a[COPY_UNROLL], b[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const int64_t v = v0 + u * COPY_THREADS;
            if (v < vec_per_block) {
                a[u] = ks[v];
                b[u] = vs[v];
            }
        }
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const int64_t v = v0 + u * COPY_THREADS;
            if (v < vec_per_block) {
                kd[v] = a[u];
                vd[v] = b[u];
            }
        }
    }
}

cudaError_t launch_copy_blocks(const int32_t *pairs, int32_t n, void *k_cache, void *v_cache, int64_t vec_per_block,
                               int32_t num_blocks, int *status, int sm_count, cudaStream_t stream) {
    if (n == 0 || vec_per_block == 0) return cudaSuccess;
    const int64_t items = (int64_t)n * ((vec_per_block + COPY_CHUNK - 1) / COPY_CHUNK);
    int64_t blocks = items;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    copy_blocks_kernel<<<(unsigned)blocks, COPY_THREADS, 0, stream>>>(pairs, n, static_cast<uint4 *>(k_cache),
                                                                      static_cast<uint4 *>(v_cache), vec_per_block,
                                                                      num_blocks, status);
    return cudaGetLastError();
}

}  // namespace pa
