// decode_noalloc.cu -- pa_decode_noalloc: the paged decode for callers that cannot allocate
// device memory (see include/pagedattn.h). Its only scratch is the file-scope array below.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pa_internal.h"

using namespace pa;

namespace {

constexpr size_t SCRATCH_BYTES = PA_NOALLOC_SCRATCH_BYTES;
constexpr size_t STATUS_BYTES = 256;   // the call's status word (offset 0) and item counters (offset 128), padded

// The call's status word (bytes 0..3), then the split pass's workspace: partition outputs followed by
// the (max, sum) pairs. Every call clears the status word and writes each partial slot it later reads.
static __device__ __align__(256) unsigned char g_scratch[SCRATCH_BYTES];

// Driver entry points (through the runtime, so the library needs no -lcuda).
template <typename F>
F driver_fn(const char *name, unsigned version) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
    static PFN_cuCtxGetCurrent_v4000 fn = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
    return fn;
}

PFN_cuCtxGetId_v12000 ctx_id_fn() {
    static PFN_cuCtxGetId_v12000 fn = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    return fn;
}

// Unique id of the calling thread's current context (false if there is none yet).
bool current_ctx_id(unsigned long long *id) {
    auto cur = ctx_current_fn();
    auto gid = ctx_id_fn();
    CUcontext c = nullptr;
    if (!cur || !gid || cur(&c) != CUDA_SUCCESS || !c) return false;
    return gid(c, id) == CUDA_SUCCESS;
}

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
struct ScratchAddr {
    void *ptr = nullptr;
    unsigned long long ctx = 0;
};
ScratchAddr g_addr[MAX_DEVICES];

// Device address of g_scratch in the current context of `device` (the current device). In host
// code the name g_scratch is only a host-side stand-in, so it is never passed to a kernel. The
// address is looked up on the first call in a context and again whenever the context changes
// (after cudaDeviceReset the module is loaded anew and the array may sit elsewhere).
cudaError_t scratch_address(int device, void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    ScratchAddr &a = g_addr[device];
    if (!a.ptr || !have_id || a.ctx != id) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);   // makes the primary context current if needed
        if (e != cudaSuccess) return e;
        if (!current_ctx_id(&id)) return cudaErrorContextIsDestroyed;
        a.ptr = p;
        a.ctx = id;
    }
    *out = a.ptr;
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn =
        driver_fn<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled", 12000);
    return fn;
}

bool encode(const void *cache, int num_blocks, int Hkv, int bs, int D, int dtype, CUtensorMap *m) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_blocks * Hkv * bs};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)TILE_TOKENS};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// With no status word to hand back, a call whose kernels flagged anything (a copy wait that ran
// out, which leaves outputs unwritten, or an out-of-range block id or context length) marks its
// whole output as NaN (the all-ones 16-bit word is a NaN in fp16 and in bf16).
__global__ void poison_on_error_kernel(const int *status, uint4 *out, int64_t nvec) {
    if (__ldcg(status) == 0) return;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, int32_t num_blocks,
                                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                                       const int32_t *block_tables, int32_t block_table_stride,
                                       const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t q_len, float scale, int32_t partition_tokens, void *out,
                                       void *stream) {
    // ---- host-side validation (nothing launched on error)
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || num_kv_heads <= 0 || block_table_stride < 1 || num_seqs < 1 || q_len < 1 || q_len > 8 ||
        num_q_heads < 1 || num_q_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (dtype != PA_FP16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (partition_tokens == 0) partition_tokens = 512;
    if (partition_tokens < 0 || partition_tokens % block_size != 0 || partition_tokens > 16384)
        return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (G * q_len > MAX_ROWS) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * num_kv_heads * block_size >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    const int64_t max_ctx = (int64_t)block_table_stride * block_size;
    if (max_ctx >= ((int64_t)1 << 31)) return PA_ERR_INVALID_ARG;
    const int64_t max_parts = (max_ctx + partition_tokens - 1) / partition_tokens;
    if ((int64_t)num_seqs * num_kv_heads * max_parts >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    if (max_parts > 1 && merge_smem_bytes(G, (int)max_parts, head_dim) > MAX_SMEM_PER_CTA) return PA_ERR_UNSUPPORTED;
    // scratch needed: the status word, then per (output row, partition) head_dim floats plus one (max, sum) pair
    const int64_t slots = (int64_t)num_seqs * q_len * num_q_heads * max_parts;
    const int64_t o_bytes = ((slots * head_dim * 4 + 255) / 256) * 256;
    const int64_t need = (int64_t)STATUS_BYTES + (max_parts > 1 ? o_bytes + slots * 8 : 0);
    if (need > (int64_t)SCRATCH_BYTES) return PA_ERR_INVALID_ARG;   // beyond PA_NOALLOC_SCRATCH_BYTES

    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= MAX_DEVICES) return PA_ERR_CUDA;
    void *scratch = nullptr;
    if (scratch_address(device, &scratch) != cudaSuccess) return PA_ERR_CUDA;
    CUtensorMap tmk, tmv;
    if (!encode(k_cache, num_blocks, num_kv_heads, block_size, head_dim, dtype, &tmk) ||
        !encode(v_cache, num_blocks, num_kv_heads, block_size, head_dim, dtype, &tmv))
        return PA_ERR_CUDA;

    unsigned char *sbase = static_cast<unsigned char *>(scratch);
    DecodeParams p;
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.k_scales = p.v_scales = nullptr;
    p.status = reinterpret_cast<int *>(sbase);
    p.vf_work = reinterpret_cast<int *>(sbase + 128);   // tensor-core decode's item counters (each launch resets them)
    p.part_o = reinterpret_cast<float *>(sbase + STATUS_BYTES);
    p.part_ml = reinterpret_cast<float2 *>(sbase + STATUS_BYTES + o_bytes);
    p.stride = block_table_stride;
    p.num_seqs = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = num_kv_heads;
    p.G = G;
    p.q_len = q_len;
    p.rows = G * q_len;
    p.bs = block_size;
    p.num_blocks = num_blocks;
    p.part_tokens = partition_tokens;
    p.max_parts = (int)max_parts;
    p.max_ctx = (int)max_ctx;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_ns = 2000000000ull;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.status, 0, sizeof(int), s) != cudaSuccess) return PA_ERR_CUDA;
    if (launch_decode(p, dtype, head_dim, tmk, tmv, s) != cudaSuccess) return PA_ERR_CUDA;
    if (max_parts > 1 && launch_merge(p, dtype, head_dim, s) != cudaSuccess) return PA_ERR_CUDA;
    const int64_t nvec = (int64_t)num_seqs * q_len * num_q_heads * head_dim * 2 / 16;
    const int64_t blocks = (nvec + 255) / 256;
    poison_on_error_kernel<<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0, s>>>(p.status,
                                                                                     static_cast<uint4 *>(out), nvec);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
