// pa_api.cu -- the C ABI declared in include/pagedattn.h: pool lifecycle, argument
// validation, TMA descriptor encoding and kernel launches. No computation happens
// here; every step of the path runs in the kernels of cache_write.cu and decode.cu.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <unordered_map>

#include "pa_internal.h"

using namespace pa;

struct pa_pool {
    pa_pool_config cfg;
    void *k_cache = nullptr;
    void *v_cache = nullptr;
    bool owns_caches = false;
    uint64_t cache_bytes = 0;
    float *part_o = nullptr;
    float2 *part_ml = nullptr;
    int64_t ws_slots = 0;        // (output row, partition) pairs the workspace holds
    int *status = nullptr;
    int *work = nullptr;         // tensor-core decode's item counters (in the status allocation; reset by each launch)
    int sm_count = 0;
    int part_tokens = 512;
    uint64_t wait_ns = 2000000000ull;
    // shared-prefix decode: the prefix kernel runs on this stream beside the caller's decode
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    std::mutex mu;
    std::unordered_map<const void *, CUtensorMap> maps;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The pool seen as a 2-D tensor: rows = num_blocks * Hkv * block_size key rows of head_dim
// elements. Boxes are 16 rows x 64 elements (128 bytes), swizzled 128B in shared memory.
pa_status tensor_map(pa_pool *pool, const void *cache, CUtensorMap *out) {
    std::lock_guard<std::mutex> lk(pool->mu);
    auto it = pool->maps.find(cache);
    if (it != pool->maps.end()) {
        *out = it->second;
        return PA_OK;
    }
    auto fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    const pa_pool_config &c = pool->cfg;
    CUtensorMap m;
    const bool kv8 = c.kv_format == PA_KV_FP8_E4M3;
    cuuint64_t dims[2] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size};
    cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * (kv8 ? 1 : 2)};
    cuuint32_t box[2] = {kv8 ? 128u : 64u, (cuuint32_t)TILE_TOKENS};   // 128-byte-wide boxes either way
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : (c.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    CUresult r = fn(&m, ty, 2, const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ERR_CUDA;
    if (pool->maps.size() > 4096) pool->maps.clear();
    pool->maps.emplace(cache, m);
    *out = m;
    return PA_OK;
}

void free_pool(pa_pool *p) {
    if (!p) return;
    DeviceGuard g(p->cfg.device);
    if (p->owns_caches) {
        cudaFree(p->k_cache);
        cudaFree(p->v_cache);
    }
    cudaFree(p->part_o);
    cudaFree(p->part_ml);
    cudaFree(p->status);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->side) cudaStreamDestroy(p->side);
    delete p;
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_OOM: return "out of device memory";
        case PA_ERR_DEVICE_BOUNDS: return "device saw an out-of-range block id, slot or context length";
        case PA_ERR_TIMEOUT: return "device gave up waiting on a copy";
    }
    return "unknown status";
}

pa_status pa_pool_create(const pa_pool_config *config, pa_pool **out) {
    if (!config || !out) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_pool_config c = *config;
    if (c.num_blocks <= 0 || c.num_kv_heads <= 0 || c.max_seqs <= 0 || c.max_q_heads <= 0 || c.max_q_len < 1 ||
        c.max_q_len > 8 || c.max_context_len < 1 || c.device < 0)
        return PA_ERR_INVALID_ARG;
    if (c.block_size != 16 && c.block_size != 32) return PA_ERR_UNSUPPORTED;
    if (c.head_dim != 64 && c.head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (c.dtype != PA_FP16 && c.dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (c.kv_format != PA_KV_16BIT && c.kv_format != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
    if (c.kv_format == PA_KV_FP8_E4M3 && c.head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (c.partition_tokens == 0) c.partition_tokens = 512;
    if (c.partition_tokens < 0 || c.partition_tokens % c.block_size != 0 || c.partition_tokens > 16384)
        return PA_ERR_INVALID_ARG;
    if ((c.k_cache == nullptr) != (c.v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    if ((c.k_cache && !aligned16(c.k_cache)) || (c.v_cache && !aligned16(c.v_cache))) return PA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)c.num_blocks * c.num_kv_heads * c.block_size;
    if (rows >= (int64_t)1 << 31) return PA_ERR_UNSUPPORTED;

    DeviceGuard g(c.device);
    if (!g.ok) return PA_ERR_CUDA;
    pa_pool *p = new pa_pool();
    p->cfg = c;
    p->part_tokens = c.partition_tokens;
    p->cache_bytes = c.kv_format == PA_KV_FP8_E4M3 ? (uint64_t)rows * (c.head_dim + 4) : (uint64_t)rows * c.head_dim * 2;
    if (cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess) {
        delete p;
        return PA_ERR_CUDA;
    }
    if (c.k_cache) {
        p->k_cache = c.k_cache;
        p->v_cache = c.v_cache;
    } else {
        p->owns_caches = true;
        if (cudaMalloc(&p->k_cache, p->cache_bytes) != cudaSuccess ||
            cudaMalloc(&p->v_cache, p->cache_bytes) != cudaSuccess) {
            cudaGetLastError();
            free_pool(p);
            return PA_ERR_OOM;
        }
    }
    const int64_t max_parts = (c.max_context_len + c.partition_tokens - 1) / c.partition_tokens;
    p->ws_slots = (int64_t)c.max_seqs * c.max_q_len * c.max_q_heads * max_parts;
    if (max_parts > 1) {
        if (cudaMalloc(&p->part_o, (size_t)p->ws_slots * c.head_dim * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&p->part_ml, (size_t)p->ws_slots * sizeof(float2)) != cudaSuccess) {
            cudaGetLastError();
            free_pool(p);
            return PA_ERR_OOM;
        }
    }
    if (cudaMalloc(&p->status, 64) != cudaSuccess || cudaMemset(p->status, 0, 64) != cudaSuccess) {
        cudaGetLastError();
        free_pool(p);
        return PA_ERR_OOM;
    }
    p->work = p->status + 8;
    if (cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        free_pool(p);
        return PA_ERR_CUDA;
    }
    *out = p;
    return PA_OK;
}

void pa_destroy(pa_pool *pool) { free_pool(pool); }

pa_status pa_pool_caches(const pa_pool *pool, void **k_cache, void **v_cache, uint64_t *bytes_each) {
    if (!pool) return PA_ERR_INVALID_ARG;
    if (k_cache) *k_cache = pool->k_cache;
    if (v_cache) *v_cache = pool->v_cache;
    if (bytes_each) *bytes_each = pool->cache_bytes;
    return PA_OK;
}

pa_status pa_cache_write(pa_pool *pool, const void *k, const void *v, const int64_t *slot_mapping,
                         int32_t num_tokens, void *k_cache, void *v_cache, void *stream) {
    if (!pool || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    if (!k_cache) {
        k_cache = pool->k_cache;
        v_cache = pool->v_cache;
    }
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    const pa_pool_config &c = pool->cfg;
    DeviceGuard g(c.device);
    if (!g.ok) return PA_ERR_CUDA;
    if (c.kv_format == PA_KV_FP8_E4M3)
        return launch_cache_write_fp8(k, v, slot_mapping, num_tokens, c.num_kv_heads, c.block_size, c.num_blocks,
                                      c.dtype, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
                                      pool->status, pool->sm_count, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? PA_OK
                   : PA_ERR_CUDA;
    CacheWriteParams p;
    p.k = static_cast<const uint4 *>(k);
    p.v = static_cast<const uint4 *>(v);
    p.slots = slot_mapping;
    p.k_cache = static_cast<uint4 *>(k_cache);
    p.v_cache = static_cast<uint4 *>(v_cache);
    p.status = pool->status;
    p.num_tokens = num_tokens;
    p.Hkv = c.num_kv_heads;
    p.vec_per_row = c.head_dim / 8;
    p.bs = c.block_size;
    p.num_blocks = c.num_blocks;
    return launch_cache_write(p, pool->sm_count, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                                     : PA_ERR_CUDA;
}

static pa_status decode_params(const pa_pool *pool, int32_t stride, int32_t num_seqs, int32_t num_q_heads,
                               int32_t q_len, DecodeParams &p) {
    const pa_pool_config &c = pool->cfg;
    if (stride < 1 || num_seqs < 1 || num_seqs > c.max_seqs || num_q_heads < 1 || num_q_heads > c.max_q_heads ||
        num_q_heads % c.num_kv_heads != 0 || q_len < 1 || q_len > c.max_q_len)
        return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / c.num_kv_heads;
    if (G * q_len > MAX_ROWS) return PA_ERR_UNSUPPORTED;
    int64_t max_ctx = (int64_t)stride * c.block_size;
    if (max_ctx > c.max_context_len) max_ctx = c.max_context_len;
    const int64_t max_parts = (max_ctx + pool->part_tokens - 1) / pool->part_tokens;
    if (max_parts > 1 && (int64_t)num_seqs * q_len * num_q_heads * max_parts > pool->ws_slots) return PA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * c.num_kv_heads * max_parts >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    if (max_parts > 1 && merge_smem_bytes(G, (int)max_parts, c.head_dim) > MAX_SMEM_PER_CTA) return PA_ERR_UNSUPPORTED;
    p.stride = stride;
    p.num_seqs = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = c.num_kv_heads;
    p.G = G;
    p.q_len = q_len;
    p.rows = G * q_len;
    p.bs = c.block_size;
    p.num_blocks = c.num_blocks;
    p.part_tokens = pool->part_tokens;
    p.max_parts = (int)max_parts;
    p.max_ctx = (int)max_ctx;
    p.wait_ns = pool->wait_ns;
    p.part_o = pool->part_o;
    p.part_ml = pool->part_ml;
    p.status = pool->status;
    return PA_OK;
}

// Partitions per CTA, chosen at launch: all of them when the (sequence, KV head) units alone fill
// three waves and contexts span at most 4 partitions; else the largest power of two that still
// leaves at least 8 waves of CTAs (2 per SM) for the longest context. Fewer, longer partitions
// write and merge fewer partial states and spread each CTA's fixed costs over more tiles. The
// persistent tensor-core kernel (one CTA per SM walking its items) needs only about 4 items per SM
// for balance, and each item ends with an epilogue, so it takes the coarsest split that keeps those.
static void coarsen_partitions(const pa_pool *pool, DecodeParams &p) {
    const int64_t units = (int64_t)p.num_seqs * p.Hkv;
    if (p.max_parts <= 1) return;
    const bool persistent = decode_uses_verify(pool->cfg.head_dim, p.rows, pool->cfg.kv_format == PA_KV_FP8_E4M3);
    if (p.max_parts <= 4 && units >= 6LL * pool->sm_count) {
        p.part_tokens = p.max_parts * p.part_tokens;
        p.max_parts = 1;
        return;
    }
    const int64_t want = persistent ? 4LL * pool->sm_count : 8LL * 2 * pool->sm_count;
    int k = 1;
    while (2 * k <= p.max_parts && units * ((p.max_parts + 2 * k - 1) / (2 * k)) >= want) k *= 2;
    if (k > 1) {
        p.part_tokens *= k;
        p.max_parts = (p.max_parts + k - 1) / k;
    }
}

int32_t pa_decode_launches(const pa_pool *pool, int32_t block_table_stride, int32_t num_seqs, int32_t num_q_heads,
                           int32_t q_len) {
    if (!pool) return -1;
    DecodeParams p;
    if (decode_params(pool, block_table_stride, num_seqs, num_q_heads, q_len, p) != PA_OK) return -1;
    coarsen_partitions(pool, p);
    return p.max_parts > 1 ? 2 : 1;
}

pa_status pa_decode(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                    int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale, void *out, void *stream) {
    if (!pool || !q || !out || !block_tables || !context_lens || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    if (!k_cache) {
        k_cache = pool->k_cache;
        v_cache = pool->v_cache;
    }
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    DecodeParams p;
    pa_status st = decode_params(pool, block_table_stride, num_seqs, num_q_heads, q_len, p);
    if (st != PA_OK) return st;
    coarsen_partitions(pool, p);
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = scale * 1.4426950408889634f;
    const bool kv8 = pool->cfg.kv_format == PA_KV_FP8_E4M3;
    const int64_t code_bytes = (int64_t)pool->cfg.num_blocks * pool->cfg.num_kv_heads * pool->cfg.block_size *
                               pool->cfg.head_dim;
    p.k_scales = kv8 ? reinterpret_cast<const float *>(static_cast<const uint8_t *>(k_cache) + code_bytes) : nullptr;
    p.v_scales = kv8 ? reinterpret_cast<const float *>(static_cast<const uint8_t *>(v_cache) + code_bytes) : nullptr;
    DeviceGuard g(pool->cfg.device);
    if (!g.ok) return PA_ERR_CUDA;
    CUtensorMap tmk, tmv;
    if ((st = tensor_map(pool, k_cache, &tmk)) != PA_OK) return st;
    if ((st = tensor_map(pool, v_cache, &tmv)) != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.merge_splits = merge_splits_for((int64_t)num_seqs * q_len * p.Hkv, p.G, pool->cfg.head_dim, pool->sm_count);
    p.vf_ctas = pool->sm_count;
    p.vf_work = pool->work;
    if (launch_decode(p, pool->cfg.dtype, pool->cfg.head_dim, tmk, tmv, s, kv8) != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_parts > 1 && launch_merge(p, pool->cfg.dtype, pool->cfg.head_dim, s) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

pa_status pa_decode_shared_prefix(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale,
                                  int32_t prefix_tokens, void *out, void *stream) {
    if (!pool || !q || !out || !block_tables || !context_lens || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    const pa_pool_config &c = pool->cfg;
    if (c.kv_format != PA_KV_16BIT || c.head_dim != 128 || pool->part_tokens % 128 != 0) return PA_ERR_UNSUPPORTED;
    if (!k_cache) {
        k_cache = pool->k_cache;
        v_cache = pool->v_cache;
    }
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    DecodeParams p;
    pa_status st = decode_params(pool, block_table_stride, num_seqs, num_q_heads, q_len, p);
    if (st != PA_OK) return st;
    if (prefix_tokens <= 0 || prefix_tokens % pool->part_tokens != 0 || prefix_tokens / pool->part_tokens >= p.max_parts)
        return PA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * p.rows > ((int64_t)1 << 24)) return PA_ERR_UNSUPPORTED;
    p.part0 = prefix_tokens / pool->part_tokens;
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_scales = p.v_scales = nullptr;
    DeviceGuard g(c.device);
    if (!g.ok) return PA_ERR_CUDA;
    CUtensorMap tmk, tmv;
    if ((st = tensor_map(pool, k_cache, &tmk)) != PA_OK) return st;
    if ((st = tensor_map(pool, v_cache, &tmv)) != PA_OK) return st;
    // prefix partitions per prefix CTA: the fewest waves of (partitions per CTA + 2 tiles of start-up)
    {
        const int64_t ctiles = (((int64_t)num_seqs * p.rows + 127) / 128 + 1) / 2;
        const int tiles_per_part = pool->part_tokens / 128;
        int64_t best = -1;
        for (int k = 1; k <= p.part0; ++k) {
            const int64_t ctas = ctiles * p.Hkv * ((p.part0 + k - 1) / k);
            const int64_t cost = ((ctas + pool->sm_count - 1) / pool->sm_count) * (k * tiles_per_part + 2);
            if (best < 0 || cost < best) {
                best = cost;
                p.pchunk = k;
            }
        }
    }
    // the suffix decode keeps the many-CTA kernel of decode.cu: its items are short (the prefix is done by the
    // prefix kernel), and the persistent tensor-core kernel's per-item costs outweigh its gain there
    // (shared-prefix verify workload: 0.075 vs 0.065 ms per call)
    p.allow_verify = false;
    p.vf_ctas = pool->sm_count;
    p.vf_work = pool->work;
    // the prefix kernel (tensor cores, one CTA per SM) goes first, straight onto the caller's stream, so
    // that its CTAs take whole SMs before the suffix decode (bandwidth, many small CTAs, on the pool's
    // side stream) fills the rest; the merge waits for both
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lk(pool->mu);
    if (cudaEventRecord(pool->ev_fork, s) != cudaSuccess || cudaStreamWaitEvent(pool->side, pool->ev_fork, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    if (launch_prefix(p, c.dtype, tmk, tmv, s) != cudaSuccess) return PA_ERR_CUDA;
    if (launch_decode(p, c.dtype, c.head_dim, tmk, tmv, pool->side, false) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaEventRecord(pool->ev_join, pool->side) != cudaSuccess || cudaStreamWaitEvent(s, pool->ev_join, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    p.merge_splits = merge_splits_for((int64_t)num_seqs * q_len * p.Hkv, p.G, c.head_dim, pool->sm_count);
    if (launch_merge(p, c.dtype, c.head_dim, s, false) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

pa_status pa_prefill(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                     int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale, void *out, void *stream) {
    if (!pool || !q || !out || !block_tables || !context_lens || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    const pa_pool_config &c = pool->cfg;
    if (c.kv_format != PA_KV_16BIT || c.head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!k_cache) {
        k_cache = pool->k_cache;
        v_cache = pool->v_cache;
    }
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    if (block_table_stride < 1 || num_seqs < 1 || num_q_heads < 1 || num_q_heads % c.num_kv_heads != 0 || q_len < 1 ||
        q_len > PA_PREFILL_MAX_Q_LEN)
        return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / c.num_kv_heads;
    const int64_t rows = (int64_t)G * q_len;
    if (rows > ((int64_t)1 << 24) || (int64_t)num_seqs * c.num_kv_heads * ((rows + 127) / 128) >= ((int64_t)1 << 31))
        return PA_ERR_UNSUPPORTED;
    int64_t max_ctx = (int64_t)block_table_stride * c.block_size;
    if (max_ctx > c.max_context_len) max_ctx = c.max_context_len;
    DecodeParams p = {};
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = pool->status;
    p.stride = block_table_stride;
    p.num_seqs = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = c.num_kv_heads;
    p.G = G;
    p.q_len = q_len;
    p.rows = (int)rows;
    p.bs = c.block_size;
    p.num_blocks = c.num_blocks;
    p.max_ctx = (int)max_ctx;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_ns = pool->wait_ns;
    DeviceGuard g(c.device);
    if (!g.ok) return PA_ERR_CUDA;
    CUtensorMap tmk, tmv;
    pa_status st;
    if ((st = tensor_map(pool, k_cache, &tmk)) != PA_OK) return st;
    if ((st = tensor_map(pool, v_cache, &tmv)) != PA_OK) return st;
    return launch_prefill(p, c.dtype, tmk, tmv, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                                 : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(pa_pool *pool, const int32_t *pairs, int32_t n, void *k_cache, void *v_cache,
                         void *stream) {
    if (!pool || n < 0) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 3u)) return PA_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return PA_ERR_INVALID_ARG;
    if (!k_cache) {
        k_cache = pool->k_cache;
        v_cache = pool->v_cache;
    }
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    const pa_pool_config &c = pool->cfg;
    DeviceGuard g(c.device);
    if (!g.ok) return PA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c.kv_format == PA_KV_FP8_E4M3) {
        // codes of a block, then its scales in the scale region
        const int64_t code_vec = (int64_t)c.num_kv_heads * c.block_size * c.head_dim / 16;
        const int64_t scale_vec = (int64_t)c.num_kv_heads * c.block_size * 4 / 16;
        const int64_t code_bytes = (int64_t)c.num_blocks * c.num_kv_heads * c.block_size * c.head_dim;
        uint8_t *kc = static_cast<uint8_t *>(k_cache), *vc = static_cast<uint8_t *>(v_cache);
        if (launch_copy_blocks(pairs, n, kc, vc, code_vec, c.num_blocks, pool->status, pool->sm_count, s) !=
                cudaSuccess ||
            launch_copy_blocks(pairs, n, kc + code_bytes, vc + code_bytes, scale_vec, c.num_blocks, pool->status,
                               pool->sm_count, s) != cudaSuccess)
            return PA_ERR_CUDA;
        return PA_OK;
    }
    const int64_t vec_per_block = (int64_t)c.num_kv_heads * c.block_size * c.head_dim / 8;
    return launch_copy_blocks(pairs, n, k_cache, v_cache, vec_per_block, c.num_blocks, pool->status, pool->sm_count,
                              s) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                         int32_t num_seqs, int32_t num_draft, int64_t vocab, int32_t *out, int32_t *n_out,
                         void *stream) {
    if (num_seqs < 0 || num_draft < 0 || num_draft > 64 || vocab < 1 || vocab >= ((int64_t)1 << 31))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!p || !v || !out || !n_out || (num_draft > 0 && (!q || !draft || !u))) return PA_ERR_INVALID_ARG;
    const void *ptrs[] = {p, q, draft, u, v, out, n_out};
    for (const void *x : ptrs)
        if (reinterpret_cast<uintptr_t>(x) & 3u) return PA_ERR_INVALID_ARG;
    return launch_spec_verify(p, q, draft, u, v, num_seqs, num_draft, vocab, out, n_out, nullptr,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_pool_selftest_wait(pa_pool *pool, uint64_t limit_ns, void *stream) {
    if (!pool || limit_ns > 10ull * 1000000000ull) return PA_ERR_INVALID_ARG;
    DeviceGuard g(pool->cfg.device);
    if (!g.ok) return PA_ERR_CUDA;
    return launch_wait_selftest(pool->status, limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                                          : PA_ERR_CUDA;
}

pa_status pa_pool_check(pa_pool *pool, void *stream) {
    if (!pool) return PA_ERR_INVALID_ARG;
    DeviceGuard g(pool->cfg.device);
    if (!g.ok) return PA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, pool->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess || cudaMemsetAsync(pool->status, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (h & STATUS_TIMEOUT) return PA_ERR_TIMEOUT;
    if (h & STATUS_BOUNDS) return PA_ERR_DEVICE_BOUNDS;
    return PA_OK;
}

}  // extern "C"
