/*
 * synth_host.c -- host-side, multithreaded copy of the seeded input generator defined in
 * synth/__init__.py (SplitMix64 counter hash; Irwin-Hall sum of twelve 16-bit fields;
 * float32 scale; round to nearest even to fp16/bf16). Test and benchmark infrastructure:
 * it exists because the numpy statement of the recipe is too slow for multi-GB inputs.
 * It holds none of the attention arithmetic.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_host_stream_base(uint64_t seed, uint64_t stream) { return mix(seed ^ (stream * 0xD1B54A32D192ED03ull)); }

static uint16_t to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static uint16_t to_f16(float x) {
    _Float16 h = (_Float16)x;   /* IEEE conversion, round to nearest even */
    uint16_t w;
    memcpy(&w, &h, 2);
    return w;
}

static uint16_t value16(uint64_t base, uint64_t idx, int dtype, float sigma, float mean) {
    uint32_t s = 0;
    for (int j = 0; j < 3; ++j) { /* h(3i), h(3i+1), h(3i+2): twelve 16-bit fields */
        const uint64_t h = mix(base + 3 * idx + (uint64_t)j);
        s += (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) + (uint32_t)((h >> 32) & 0xFFFF) +
             (uint32_t)(h >> 48);
    }
    const float num = (float)(2 * (int32_t)s - 786420);   /* exact */
    /* three separately rounded float32 operations (built with -ffp-contract=off); the first is exact */
    float z = num * 0x1p-17f;
    z = z * sigma;
    z = z + mean;
    return dtype == 0 ? to_f16(z) : to_bf16(z);
}

typedef struct {
    uint16_t *dst;
    const int64_t *rows;
    int64_t nrows, row_len;
    uint64_t base;
    int dtype;
    float sigma, mean;
    int64_t r0, r1;
} job_t;

static void *work(void *arg) {
    job_t *J = (job_t *)arg;
    for (int64_t r = J->r0; r < J->r1; ++r) {
        const int64_t src = (J->rows ? J->rows[r] : r) * J->row_len;
        uint16_t *d = J->dst + r * J->row_len;
        for (int64_t c = 0; c < J->row_len; ++c) d[c] = value16(J->base, (uint64_t)(src + c), J->dtype, J->sigma, J->mean);
    }
    return NULL;
}

/* dst[r][c] = value(rows[r] * row_len + c); rows NULL means r. */
int synth_host_fill_rows(uint16_t *dst, const int64_t *rows, int64_t nrows, int64_t row_len, uint64_t seed,
                         uint64_t stream, int dtype, float sigma, float mean, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if (nrows < nthreads) nthreads = nrows > 0 ? (int)nrows : 1;
    pthread_t th[64];
    job_t jobs[64];
    const uint64_t base = synth_host_stream_base(seed, stream);
    for (int i = 0; i < nthreads; ++i) {
        job_t j = {dst, rows, nrows, row_len, base, dtype, sigma, mean, nrows * i / nthreads, nrows * (i + 1) / nthreads};
        jobs[i] = j;
        pthread_create(&th[i], NULL, work, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    return 0;
}
