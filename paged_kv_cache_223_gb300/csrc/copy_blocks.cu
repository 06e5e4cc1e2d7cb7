// copy_blocks.cu -- the device half of copy-on-write: copy whole physical blocks (every KV
// head, K and V) from src to dst so a sequence can write into its own copy of a block it
// shared with others (yangyu.win blog #54, section 5 question 2).
//
// A block of the [num_blocks, Hkv, bs, d] pool is Hkv * bs * d contiguous 16-bit words; each
// thread moves 16-byte vectors, so reads and writes are fully coalesced; each thread has four K and
// four V vectors of one item in flight while it stores those of the item before.
#include "pa_device.cuh"

namespace pa {

constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;                                // K and V vectors in flight per thread
constexpr int COPY_CHUNK = COPY_THREADS * COPY_UNROLL;        // vectors of one work item (16 KB of K, of V)

// Work item = (pair c, chunk k of COPY_CHUNK vectors of its blocks); the grid strides over items.
// Each thread loads its COPY_UNROLL K and V vectors of the next item (and that item's pair) before it
// stores those of the current one, so its loads never wait for its stores. Against loading each item
// only after storing the one before (48 registers, 5 CTAs per SM; now 107 and 2): 0.0974 -> 0.0937 ms
// on 4096 pairs of 32 KB blocks, same box, three rounds.
__global__ void __launch_bounds__(COPY_THREADS) copy_blocks_kernel(const int32_t *pairs, int32_t n, uint4 *k_cache,
                                                                   uint4 *v_cache, int64_t vec_per_block,
                                                                   int32_t num_blocks, int *status) {
    const int chunks = (int)((vec_per_block + COPY_CHUNK - 1) / COPY_CHUNK);
    const int64_t items = (int64_t)n * chunks;
    // two register sets: slot s holds an item's vectors, its destination block offset and first vector
    uint4 a[2][COPY_UNROLL], b[2][COPY_UNROLL];
    int64_t dst_off[2], v0[2];
    bool ok[2];
    auto load = [&](int64_t item, int s) {
        const int c = (int)(item / chunks);
        const int k = (int)(item - (int64_t)c * chunks);
        const int32_t src = __ldg(pairs + 2 * c), dst = __ldg(pairs + 2 * c + 1);
        ok[s] = src >= 0 && src < num_blocks && dst >= 0 && dst < num_blocks;
        if (!ok[s]) {
            if (k == 0 && threadIdx.x == 0) set_status(status, STATUS_BOUNDS);
            return;
        }
        const uint4 *ks = k_cache + (int64_t)src * vec_per_block, *vs = v_cache + (int64_t)src * vec_per_block;
        dst_off[s] = (int64_t)dst * vec_per_block;
        v0[s] = (int64_t)k * COPY_CHUNK + threadIdx.x;
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const int64_t v = v0[s] + u * COPY_THREADS;
            if (v < vec_per_block) {
                a[s][u] = ks[v];
                b[s][u] = vs[v];
            }
        }
    };
    auto store = [&](int s) {
        if (!ok[s]) return;
        uint4 *kd = k_cache + dst_off[s], *vd = v_cache + dst_off[s];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const int64_t v = v0[s] + u * COPY_THREADS;
            if (v < vec_per_block) {
                kd[v] = a[s][u];
                vd[v] = b[s][u];
            }
        }
    };
    int64_t item = blockIdx.x;
    if (item >= items) return;
    load(item, 0);
    // two items per trip, so that each register set keeps a fixed slot
    for (;;) {
        const int64_t next = item + gridDim.x;
        if (next < items) load(next, 1);
        store(0);
        if (next >= items) break;
        const int64_t after = next + gridDim.x;
        if (after < items) load(after, 0);
        store(1);
        if (after >= items) break;
        item = after;
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
