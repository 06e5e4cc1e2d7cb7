// synth.cu -- device-side copy of the seeded input generator in synth/__init__.py.
//
// Test and benchmark infrastructure: it fills buffers with the same 16-bit words the
// host generator produces (SplitMix64 counter hash; Irwin-Hall sum of twelve 16-bit
// fields; float32 scale; round to nearest even to fp16/bf16), so workloads of many GB
// can be created on the GPU while the oracle regenerates any part of them on the host.
// It holds none of the attention arithmetic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace {

__host__ __device__ __forceinline__ uint64_t mix(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t value16(uint64_t base, uint64_t idx, int dtype, float sigma, float mean) {
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) {   // h(3i), h(3i+1), h(3i+2): twelve 16-bit fields
        const uint64_t h = mix(base + 3 * idx + j);
        s += (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) + (uint32_t)((h >> 32) & 0xFFFF) +
             (uint32_t)(h >> 48);
    }
    const float num = (float)(2 * (int32_t)s - 786420);           // exact
    float z = __fmul_rn(num, 0x1p-17f);                            // exact: a power of two
    z = __fmul_rn(z, sigma);
    z = __fadd_rn(z, mean);
    if (dtype == 0) return __half_as_ushort(__float2half_rn(z));
    return __bfloat16_as_ushort(__float2bfloat16_rn(z));
}

// dst[r][c] = value(rows[r] * row_len + c) for r < nrows, c < row_len
__global__ void fill_rows_kernel(uint16_t *dst, const int64_t *rows, int64_t nrows, int64_t row_len, uint64_t base,
                                 int dtype, float sigma, float mean) {
    const int64_t total = nrows * row_len;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / row_len;
        const int64_t c = i - r * row_len;
        const int64_t src = (rows ? rows[r] : r) * row_len + c;
        dst[i] = value16(base, (uint64_t)src, dtype, sigma, mean);
    }
}

__global__ void fill_word_kernel(uint16_t *dst, int64_t n, uint16_t w) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = w;
}

}  // namespace

extern "C" {

// base = mix(seed ^ (stream * 0xD1B54A32D192ED03)), as on the host.
uint64_t synth_stream_base(uint64_t seed, uint64_t stream) { return mix(seed ^ (stream * 0xD1B54A32D192ED03ull)); }

// rows: device int64 [nrows] of counter rows, or NULL for rows 0..nrows-1. Returns a cudaError_t.
int synth_fill_rows(void *dst, const int64_t *rows, int64_t nrows, int64_t row_len, uint64_t seed, uint64_t stream,
                    int dtype, float sigma, float mean, void *cuda_stream) {
    const int64_t total = nrows * row_len;
    if (total <= 0) return 0;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    fill_rows_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(
        (uint16_t *)dst, rows, nrows, row_len, synth_stream_base(seed, stream), dtype, sigma, mean);
    return (int)cudaGetLastError();
}

int synth_fill_word(void *dst, int64_t n, uint16_t word, void *cuda_stream) {
    if (n <= 0) return 0;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    fill_word_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>((uint16_t *)dst, n, word);
    return (int)cudaGetLastError();
}

}  // extern "C"
