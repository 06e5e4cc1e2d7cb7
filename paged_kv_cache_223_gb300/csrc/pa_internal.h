// pa_internal.h -- types shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// Bits of the device status word (read by pa_pool_check).
constexpr int STATUS_BOUNDS = 1;   // block id, slot or context length outside what the pool/table holds
constexpr int STATUS_TIMEOUT = 2;  // a bounded wait on a TMA copy ran out

constexpr int TILE_TOKENS = 16;    // tokens per staged K/V tile (one m16 MMA tile of keys)
constexpr int DECODE_WARPS = 4;    // warps per decode CTA (each runs its own copy pipeline)
constexpr int MAX_ROWS = 32;       // query rows per (sequence, KV head): q_len * (Hq / Hkv)

struct DecodeParams {
    const void *q;
    void *out;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const float *k_scales;  // FP8 pools: per (slot, head) scales of K and V, [num_blocks, Hkv, bs]
    const float *v_scales;
    float *part_o;       // [num_seqs, q_len, Hq, max_parts, D] unnormalised partition outputs
    float2 *part_ml;     // [num_seqs, q_len, Hq, max_parts] (running max in log2 units, sum)
    int *status;
    int64_t stride;      // block-table row stride (entries)
    int num_seqs;
    int Hq;
    int Hkv;
    int G;               // Hq / Hkv
    int q_len;
    int rows;            // q_len * G
    int bs;              // block size (16 or 32)
    int num_blocks;
    int part_tokens;     // partition length (multiple of bs)
    int max_parts;       // partitions launched per (sequence, KV head)
    int max_ctx;         // longest context the launch covers (max_parts * part_tokens, <= stride * bs)
    float scale_log2;    // scale * log2(e)
    uint64_t wait_ns;    // bounded-wait limit
    int part0 = 0;       // shared-prefix decode: partitions below part0 (the prefix) come from the prefix
                         // kernel; the decode covers [part0, max_parts)
    int pchunk = 1;      // prefix partitions per prefix-kernel CTA (their combined state goes to the first)
    int merge_splits = 1;  // merge CTAs per (sequence, query position, KV head): each takes a share of
                           // the (row, 4-dim) columns, so small batches still fill the GPU
    int vf_ctas = 0;       // tensor-core verify kernel: persistent CTAs (0 = one per SM of the device)
    int *vf_work = nullptr;  // tensor-core verify kernel: [next item, CTAs finished], both 0 between launches
    bool allow_verify = true;  // may route 9..32 rows to the tensor-core verify kernel
};

struct CacheWriteParams {
    const uint4 *k;
    const uint4 *v;
    const int64_t *slots;
    uint4 *k_cache;
    uint4 *v_cache;
    int *status;
    int64_t num_tokens;
    int Hkv;
    int vec_per_row;     // head_dim / 8
    int bs;
    int64_t num_blocks;
};

// A kernel launch with programmatic stream serialization: the kernel may be launched while the one ahead
// of it in the stream is still running, and waits for it (pdl_wait) before touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_maybe_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args &&...args) {
    if (pdl) return launch_pdl(kernel, grid, block, smem, stream, static_cast<Args &&>(args)...);
    kernel<<<grid, block, smem, stream>>>(static_cast<Args &&>(args)...);
    return cudaGetLastError();
}

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_cache_write(const CacheWriteParams &p, int sm_count, cudaStream_t stream);
// FP8 pools: k, v hold 16-bit rows of the model dtype; caches are codes followed by scales.
cudaError_t launch_cache_write_fp8(const void *k, const void *v, const int64_t *slots, int64_t num_tokens, int Hkv,
                                   int bs, int64_t num_blocks, int dtype, uint8_t *k_cache, uint8_t *v_cache,
                                   int *status, int sm_count, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &p, int dtype, int head_dim, const CUtensorMap &tmk,
                          const CUtensorMap &tmv, cudaStream_t stream, bool kv8 = false);
// pdl: launched with programmatic serialization behind the decode kernel that writes the partitions' states
// (false when other work is ordered in between, e.g. an event wait)
cudaError_t launch_merge(const DecodeParams &p, int dtype, int head_dim, cudaStream_t stream, bool pdl = true);
cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                               int B, int K, int64_t V, int32_t *out, int32_t *n_out, int *status,
                               cudaStream_t stream);
cudaError_t launch_copy_blocks(const int32_t *pairs, int32_t n, void *k_cache, void *v_cache, int64_t vec_per_block,
                               int32_t num_blocks, int *status, int sm_count, cudaStream_t stream);
cudaError_t launch_prefill(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           cudaStream_t stream);
// Shared-prefix attention: every query row of every sequence against prefix partitions [0, part0)
// (blocks from sequence 0's table), written as partition partials for the merge.
cudaError_t launch_prefix(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          cudaStream_t stream);
// Tensor-core decode of 9..32 query rows per KV head (16-bit pools, head_dim 128): persistent, at most
// max_ctas CTAs (one per SM).
cudaError_t launch_verify(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          int max_ctas, cudaStream_t stream);
bool decode_uses_verify(int head_dim, int rows, bool kv8);
size_t decode_smem_bytes(int head_dim, int nt);
size_t verify_smem_bytes();
size_t prefill_smem_bytes();
size_t merge_smem_bytes(int G, int max_parts, int head_dim, int splits = 1);
int merge_splits_for(int64_t units, int G, int head_dim, int sm_count);
constexpr size_t MAX_SMEM_PER_CTA = 227 * 1024;

}  // namespace pa
