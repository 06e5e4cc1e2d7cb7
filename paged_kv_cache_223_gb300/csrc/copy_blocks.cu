// copy_blocks.cu -- the device half of copy-on-write: copy whole physical blocks (every KV
// head, K and V) from src to dst so a sequence can write into its own copy of a block it
// shared with others (yangyu.win blog #54, section 5 question 2).
//
// A block of the [num_blocks, Hkv, bs, d] pool is Hkv * bs * d contiguous 16-bit words; each
// thread moves 16-byte vectors, so reads and writes are fully coalesced.
#include "pa_device.cuh"

namespace pa {

__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t *pairs, int32_t n, uint4 *k_cache,
                                                          uint4 *v_cache, int64_t vec_per_block, int32_t num_blocks,
                                                          int *status) {
    const int64_t total = (int64_t)n * vec_per_block;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = i / vec_per_block;
        const int64_t v = i - c * vec_per_block;
        const int32_t src = __ldg(pairs + 2 * c), dst = __ldg(pairs + 2 * c + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (v == 0) set_status(status, STATUS_BOUNDS);
            continue;
        }
        k_cache[(int64_t)dst * vec_per_block + v] = k_cache[(int64_t)src * vec_per_block + v];
        v_cache[(int64_t)dst * vec_per_block + v] = v_cache[(int64_t)src * vec_per_block + v];
    }
}

cudaError_t launch_copy_blocks(const int32_t *pairs, int32_t n, void *k_cache, void *v_cache, int64_t vec_per_block,
                               int32_t num_blocks, int *status, int sm_count, cudaStream_t stream) {
    const int64_t total = (int64_t)n * vec_per_block;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    copy_blocks_kernel<<<(unsigned)blocks, 256, 0, stream>>>(pairs, n, static_cast<uint4 *>(k_cache),
                                                             static_cast<uint4 *>(v_cache), vec_per_block, num_blocks,
                                                             status);
    return cudaGetLastError();
}

}  // namespace pa
