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

// ---------------------------------------------------------------- FP8 pools
//
// Quantising cache write for FP8 E4M3 pools (head_dim 128). A cache buffer holds the codes
// [num_blocks, Hkv, bs, 128] followed by one float32 scale per (slot, head). One warp per
// (token, head) row: scale = amax|x| / 448 (1 when amax is 0), codes = e4m3(x / scale) rounded
// to nearest even and saturated, so the row's largest magnitude maps to the largest finite code
// (the quantisation section of learn.tanhdev.com part 8: FP8 E4M3 halves the KV cache, with care
// against overflow from outliers). Each lane converts 4 values; the row's 128 codes are one
// coalesced 128-byte store.
namespace pa {

template <typename T>
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(const T *k, const T *v, const int64_t *slots,
                                                               int64_t num_tokens, int Hkv, int bs, int64_t num_blocks,
                                                               uint8_t *k_cache, uint8_t *v_cache, int *status) {
    constexpr int D = 128;
    const int lane = threadIdx.x & 31;
    const int64_t rows = num_tokens * Hkv;
    const int64_t slot_limit = num_blocks * bs;
    const int64_t codes = num_blocks * Hkv * bs * D;
    for (int64_t r = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t tok = r / Hkv;
        const int h = (int)(r - tok * Hkv);
        const int64_t s = __ldg(slots + tok);
        if (s < 0) continue;
        if (s >= slot_limit) {
            if (lane == 0) set_status(status, STATUS_BOUNDS);
            continue;
        }
        const int64_t blk = s / bs, off = s - (s / bs) * bs;
        const int64_t srow = (blk * Hkv + h) * bs + off;          // slot row of this head
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const T *src = (which ? v : k) + r * D + lane * 4;
            uint8_t *pool = which ? v_cache : k_cache;
            const uint2 raw = *reinterpret_cast<const uint2 *>(src);
            const T *e = reinterpret_cast<const T *>(&raw);
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = (float)e[i];
            float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
            const __nv_fp8x2_storage_t c01 =
                __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)), __NV_SATFINITE,
                                         __NV_E4M3);
            const __nv_fp8x2_storage_t c23 =
                __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)), __NV_SATFINITE,
                                         __NV_E4M3);
            *reinterpret_cast<uint32_t *>(pool + srow * D + lane * 4) = (uint32_t)c01 | ((uint32_t)c23 << 16);
            if (lane == 0) reinterpret_cast<float *>(pool + codes)[srow] = scale;
        }
    }
}

cudaError_t launch_cache_write_fp8(const void *k, const void *v, const int64_t *slots, int64_t num_tokens, int Hkv,
                                   int bs, int64_t num_blocks, int dtype, uint8_t *k_cache, uint8_t *v_cache,
                                   int *status, int sm_count, cudaStream_t stream) {
    const int64_t rows = num_tokens * Hkv;
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows * 32 + 255) / 256;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    if (dtype == PA_FP16)
        cache_write_fp8_kernel<__half><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const __half *>(k), static_cast<const __half *>(v), slots, num_tokens, Hkv, bs, num_blocks,
            k_cache, v_cache, status);
    else
        cache_write_fp8_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), slots, num_tokens, Hkv, bs,
            num_blocks, k_cache, v_cache, status);
    return cudaGetLastError();
}

}  // namespace pa
