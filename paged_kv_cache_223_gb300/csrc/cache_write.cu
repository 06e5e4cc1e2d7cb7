// cache_write.cu -- scatter the new tokens' K and V rows into their pool slots.
//
// Each new token i owns slot s = slot_mapping[i]; row (i, h) of k goes to
// K[s / bs][h][s % bs][:], likewise v (a sequence that crosses a block boundary
// gets a fresh physical block from the free pool: yangyu.win blog #54, section 5
// question 2). The copy is of raw 16-bit words, one 16-byte vector per thread:
// loads of a token's rows are contiguous, and each (token, head) row lands as
// head_dim * 2 contiguous bytes, so both sides are fully coalesced.
#include "pa_device.cuh"

namespace pa {

__global__ void __launch_bounds__(256) cache_write_kernel(const CacheWriteParams p) {
    const int64_t per_tok = (int64_t)p.Hkv * p.vec_per_row;
    const int64_t total = p.num_tokens * per_tok;
    const int64_t slot_limit = p.num_blocks * p.bs;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tok = i / per_tok;
        const int64_t rem = i - tok * per_tok;            // h * vec_per_row + vec
        const int64_t s = __ldg(p.slots + tok);
        if (s < 0) continue;                              // padding token
        if (s >= slot_limit) {                            // outside the pool: skip, flag
            set_status(p.status, STATUS_BOUNDS);
            continue;
        }
        const int64_t blk = s / p.bs;
        const int64_t off = s - blk * p.bs;
        const int64_t h = rem / p.vec_per_row;
        const int64_t vec = rem - h * p.vec_per_row;
        const int64_t dst = ((blk * p.Hkv + h) * p.bs + off) * p.vec_per_row + vec;
        const uint4 kv = __ldg(p.k + i);
        const uint4 vv = __ldg(p.v + i);
        p.k_cache[dst] = kv;
        p.v_cache[dst] = vv;
    }
}

cudaError_t launch_cache_write(const CacheWriteParams &p, int sm_count, cudaStream_t stream) {
    const int64_t total = p.num_tokens * p.Hkv * p.vec_per_row;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count * 8;
    if (blocks > cap) blocks = cap;
    cache_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
