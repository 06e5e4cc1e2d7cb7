/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged-attention decode library.
 *
 * The KV cache is one pool of fixed-size physical blocks (16 or 32 tokens);
 * each sequence's block table maps its logical token blocks to physical block
 * ids, and the attention kernel looks the table up itself (itimpress.au
 * "PagedAttention, speculative decoding, MoE and Blackwell", section 1;
 * yangyu.win blog #54 section 2.2; learn.tanhdev.com "Part 8: Inference
 * optimization with vLLM", section on executing the kernel math in CUDA).
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must point to memory of the pool's
 *    device, 16-byte aligned, owned by the caller (the library never frees
 *    them). The library owns only what pa_pool_create allocated.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Work is enqueued asynchronously; no call synchronises except
 *    pa_pool_check.
 *  - Argument errors are detected on the host and returned before anything is
 *    launched. Data errors that only the device can see (a block id outside the
 *    pool, a context length the table cannot hold, a slot outside the pool) are
 *    checked on the device: the access is skipped or clamped and a sticky bit
 *    is set in the pool's status word, read back by pa_pool_check.
 *
 * Layouts (row-major, element = one 16-bit fp16 or bf16 value):
 *   K pool, V pool   [num_blocks, num_kv_heads, block_size, head_dim]
 *   new k, v         [num_tokens, num_kv_heads, head_dim]
 *   q, out           [num_seqs, q_len, num_q_heads, head_dim]
 *   block_tables     int32 [num_seqs, block_table_stride]
 *   context_lens     int32 [num_seqs], counting the q_len newest tokens
 *   slot_mapping     int64 [num_tokens], slot = block * block_size + offset
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or geometry; nothing launched */
    PA_ERR_UNSUPPORTED = 2,    /* valid but not built (e.g. head_dim not in {64, 128}) */
    PA_ERR_CUDA = 3,           /* a CUDA runtime or driver call failed */
    PA_ERR_OOM = 4,            /* pa_pool_create could not allocate */
    PA_ERR_DEVICE_BOUNDS = 5,  /* pa_pool_check: a kernel saw an out-of-range block id, slot or length */
    PA_ERR_TIMEOUT = 6         /* pa_pool_check: a kernel gave up waiting on a copy (bounded wait) */
} pa_status;

typedef enum pa_dtype { PA_FP16 = 0, PA_BF16 = 1 } pa_dtype;

/*
 * How K and V are stored in the pool.
 *  PA_KV_16BIT     in the model dtype: each cache is [num_blocks, Hkv, bs, head_dim] 16-bit values.
 *  PA_KV_FP8_E4M3  FP8 E4M3 codes with one float32 scale per (slot, head): each cache is one buffer
 *                  of num_blocks*Hkv*bs*head_dim code bytes followed by num_blocks*Hkv*bs float32
 *                  scales ([num_blocks, Hkv, bs]). pa_cache_write quantises: scale = amax|row| / 448
 *                  (1 for an all-zero row), code = e4m3(x / scale), nearest even, saturated; decode
 *                  uses code * scale. head_dim 128 only. (yangyu.win blog #54 section 4 and the
 *                  quantisation section of learn.tanhdev.com part 8: FP8 E4M3 halves the KV cache.)
 */
typedef enum pa_kv_format { PA_KV_16BIT = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_format;

typedef struct pa_pool pa_pool;

/*
 * Geometry of one KV pool and the limits the pool's workspace is sized for.
 * A pool describes one attention layer's cache. Layers with the same geometry
 * may share one pool object and pass their own caches to pa_cache_write and
 * pa_decode.
 */
typedef struct pa_pool_config {
    int32_t num_blocks;        /* physical blocks in the pool (> 0) */
    int32_t block_size;        /* tokens per block: 16 or 32 */
    int32_t num_kv_heads;      /* KV heads (> 0) */
    int32_t head_dim;          /* 64 or 128 */
    int32_t dtype;             /* pa_dtype of K, V, q and out */
    int32_t device;            /* CUDA device ordinal */
    int32_t partition_tokens;  /* context partition length for the split pass; 0 = 512.
                                  Must be a positive multiple of block_size. */
    int32_t max_seqs;          /* largest num_seqs passed to pa_decode */
    int32_t max_q_heads;       /* largest num_q_heads */
    int32_t max_q_len;         /* largest q_len (1..8) */
    int32_t max_context_len;   /* largest context length (sizes the split workspace) */
    void *k_cache;             /* device pointer to a caller-owned K pool, or NULL to allocate */
    void *v_cache;             /* same for V */
    int32_t kv_format;         /* pa_kv_format (0 = 16-bit in the model dtype) */
} pa_pool_config;

/*
 * Create a pool: validates the geometry, allocates the caches when the config
 * passes NULL (left uninitialised), the split workspace and the status word on
 * `device`. On success *out owns them until pa_destroy.
 * Errors: PA_ERR_INVALID_ARG (geometry), PA_ERR_UNSUPPORTED, PA_ERR_OOM, PA_ERR_CUDA.
 */
pa_status pa_pool_create(const pa_pool_config *config, pa_pool **out);

/* Release everything the pool allocated (not caller-owned caches). NULL is a no-op. */
void pa_destroy(pa_pool *pool);

/* The pool's own K and V caches (device pointers; the ones passed in or allocated) and their bytes each
   (for FP8 pools: codes plus scales). */
pa_status pa_pool_caches(const pa_pool *pool, void **k_cache, void **v_cache, uint64_t *bytes_each);

/*
 * Cache write (scatter): for each token i with slot s = slot_mapping[i] >= 0
 * and each KV head h, copy k[i][h][:] to K[s / block_size][h][s % block_size][:]
 * and v likewise. Raw 16-bit words are copied without conversion (FP8 pools:
 * each row is quantised with its own scale, see pa_kv_format); negative
 * slots are skipped (padding). Slots beyond the pool are skipped and flagged
 * (PA_ERR_DEVICE_BOUNDS). Two tokens with one slot: which one lands is unspecified.
 * (A sequence growing past a block boundary receives a new physical block:
 * yangyu.win blog #54, section 5 question 2.)
 *   k, v            device, [num_tokens, num_kv_heads, head_dim]
 *   slot_mapping    device, int64 [num_tokens]
 *   k_cache/v_cache device pools to write, or NULL for the pool's own
 */
pa_status pa_cache_write(pa_pool *pool, const void *k, const void *v, const int64_t *slot_mapping,
                         int32_t num_tokens, void *k_cache, void *v_cache, void *stream);

/*
 * Paged attention decode. For sequence b, query row qi (0 <= qi < q_len) and
 * query head h (KV head g = h / (num_q_heads / num_kv_heads)):
 *   the row sits at position p = context_lens[b] - q_len + qi and attends to
 *   tokens t = 0..p, token t read from physical block block_tables[b][t / bs]
 *   at offset t % bs;
 *   out[b][qi][h] = sum_t softmax_t(scale * q[b][qi][h] . K_t) * V_t
 * (learn.tanhdev.com part 8: A_i = softmax(q_i K^T / sqrt(d_k)) computed block
 * by block with an online softmax, o_i = sum_j sum_t a_{i,j,t} v_{(j,t)}).
 * q_len > 1 verifies q_len speculative draft tokens in one pass with a causal
 * mask (itimpress.au section 1; yangyu.win section 2.4). Several tables may
 * name the same physical blocks (a shared copy-on-write prefix); no special
 * case is needed. Contexts longer than the pool's partition_tokens are cut into
 * partitions whose (max, sum, weighted V) are combined by a log-sum-exp merge
 * (maths.nthquan ch. 17 "Scaling and deployment", section on sequence
 * parallelism: local attention per segment, then a reduction); the merge uses
 * the pool's workspace and a second kernel on the same stream.
 * Accumulation is fp32; out is rounded to nearest even. Results are
 * deterministic run to run. Concurrent pa_decode calls on one pool must be
 * ordered (they share the workspace).
 *   q                     device [num_seqs, q_len, num_q_heads, head_dim]
 *   k_cache, v_cache      device pools, or NULL for the pool's own
 *   block_tables          device int32 [num_seqs, block_table_stride]; entries at or
 *                         beyond ceil(context_lens[b] / bs) are never read
 *   context_lens          device int32 [num_seqs]; q_len <= context_lens[b] <= stride * bs
 *   num_q_heads           a multiple of num_kv_heads; (num_q_heads / num_kv_heads) * q_len <= 32
 *   scale                 softmax scale (1/sqrt(head_dim) in the pages' formula)
 *   out                   device [num_seqs, q_len, num_q_heads, head_dim]
 */
pa_status pa_decode(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                    int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale, void *out,
                    void *stream);

/*
 * Paged decode for a batch whose sequences share a prefix (copy-on-write
 * blocks named by every table: yangyu.win blog #54, section 5 question 2;
 * itimpress.au section 1). Computes exactly pa_decode's result; the shared
 * part is evaluated once for the whole batch: every query row of every
 * sequence attends to each prefix partition on the 5th-generation tensor
 * cores (one pass over the prefix's K/V instead of one per sequence), the
 * decode kernel covers each sequence's own tokens, and the log-sum-exp merge
 * combines the partitions (maths.nthquan ch. 17 "Sequence parallelism").
 * Preconditions, checked on the device (violations are flagged,
 * PA_ERR_DEVICE_BOUNDS at pa_pool_check, outputs then unspecified):
 *   block_tables[b][i] == block_tables[0][i] for i < prefix_tokens / block_size;
 *   context_lens[b] - q_len >= prefix_tokens (every query row follows the prefix).
 * Host-checked: 16-bit pool, head_dim 128, the pool's partition_tokens a
 * multiple of 128, prefix_tokens a positive multiple of partition_tokens and
 * below the launch's longest context, scale > 0; all other arguments as
 * pa_decode (which this call replaces; it uses the pool's workspace).
 */
pa_status pa_decode_shared_prefix(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, int32_t block_table_stride,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t q_len, float scale, int32_t prefix_tokens, void *out,
                                  void *stream);

/*
 * Chunked prefill: attention for a chunk of q_len new tokens per sequence, the
 * chunk's K and V already written to the pool (pa_cache_write). A long prompt
 * is processed in chunks (yangyu.win blog #54, section 4 "Chunked Prefill":
 * an 8,000-token prompt as 512-token chunks); chunk row qi sits at position
 * context_lens[b] - q_len + qi and attends causally to tokens 0..that position,
 * which is exactly pa_decode's definition with a large q_len (learn.tanhdev.com
 * part 8: A_i = softmax(q_i K^T / sqrt(d_k)), o_i = sum a v). The products run
 * on the 5th-generation tensor cores (tcgen05.mma, fp32 accumulators in tensor
 * memory); the softmax is fp32; out is rounded to nearest even.
 * Requires a 16-bit pool with head_dim 128 (PA_ERR_UNSUPPORTED otherwise).
 * Uses no workspace: concurrent calls on one pool are allowed.
 *   q              device [num_seqs, q_len, num_q_heads, 128]
 *   k_cache, v_cache  device pools, or NULL for the pool's own
 *   block_tables   device int32 [num_seqs, block_table_stride]
 *   context_lens   device int32 [num_seqs]; q_len <= context_lens[b] <= stride * bs
 *                  (violations are flagged, PA_ERR_DEVICE_BOUNDS at pa_pool_check)
 *   q_len          1 .. PA_PREFILL_MAX_Q_LEN; num_q_heads a multiple of num_kv_heads
 *   scale          softmax scale, finite and > 0 (1/sqrt(head_dim) in the pages' formula)
 *   out            device [num_seqs, q_len, num_q_heads, 128]
 */
#define PA_PREFILL_MAX_Q_LEN 8192
pa_status pa_prefill(pa_pool *pool, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                     int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale, void *out,
                     void *stream);

/*
 * Synchronise the device, read and clear the pool's status word.
 * Returns PA_OK, PA_ERR_DEVICE_BOUNDS, PA_ERR_TIMEOUT or PA_ERR_CUDA.
 */
pa_status pa_pool_check(pa_pool *pool, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Block manager (host side) and copy-on-write.
 *
 * The pool's physical blocks are handed out from one shared free pool; a
 * block named by several block tables (a shared prompt, parallel samples)
 * carries a reference count; before a sequence writes into a block it shares,
 * the block is copied to a private one (copy-on-write). (yangyu.win blog #54,
 * section 5 question 2; itimpress.au section 1.) The allocator is plain host
 * memory and host code, thread-safe, and never touches the GPU; the copy is
 * pa_copy_blocks. A failed call changes nothing.
 */
typedef struct pa_block_allocator pa_block_allocator;

/* An allocator of num_blocks blocks of block_size tokens, all free. */
pa_status pa_allocator_create(int32_t num_blocks, int32_t block_size, pa_block_allocator **out);
void pa_allocator_destroy(pa_block_allocator *allocator);

/* Free blocks left; the reference count of one block (0 = free). -1 on a bad argument. */
int32_t pa_allocator_num_free(pa_block_allocator *allocator);
int32_t pa_allocator_ref_count(pa_block_allocator *allocator, int32_t block_id);

/* Take n free blocks (reference count 1 each) into ids[n]; PA_ERR_OOM if fewer are free. */
pa_status pa_allocator_alloc(pa_block_allocator *allocator, int32_t n, int32_t *ids);

/* One more reference to each listed live block (a new table shares them). */
pa_status pa_allocator_fork(pa_block_allocator *allocator, const int32_t *ids, int32_t n);

/* Drop one reference per listed id (an id may repeat); blocks reaching 0 return to the free pool. */
pa_status pa_allocator_free(pa_block_allocator *allocator, const int32_t *ids, int32_t n);

/*
 * Copy-on-write before writing into block_id: if it is shared (count > 1), one
 * reference is dropped, a free block is taken into *out_id and *copy = 1 (the
 * caller copies block_id -> *out_id with pa_copy_blocks before writing);
 * otherwise *out_id = block_id and *copy = 0.
 */
pa_status pa_allocator_cow(pa_block_allocator *allocator, int32_t block_id, int32_t *out_id, int32_t *copy);

/*
 * Append n_new tokens to a sequence of *len tokens whose block-table row
 * (host int32 [stride]) holds ceil(*len / block_size) live blocks: takes a new
 * block each time a token crosses a block boundary, copy-on-writes the partly
 * filled last block if it is shared (then copy_pair = {old, new} and
 * *n_copies = 1, else 0), writes each new token's slot
 * (block * block_size + offset) to slots[n_new] (host int64), and advances *len.
 */
pa_status pa_allocator_append(pa_block_allocator *allocator, int32_t *table_row, int32_t stride, int32_t *len,
                              int32_t n_new, int64_t *slots, int32_t *copy_pair, int32_t *n_copies);

/*
 * Copy whole blocks on the device: for i < n, block pairs[2i] -> block
 * pairs[2i+1] of both caches (every KV head), raw words. pairs is a device
 * int32 [n][2]; destinations must be distinct and not sources of another pair.
 * Ids outside the pool are skipped and flagged (PA_ERR_DEVICE_BOUNDS).
 * k_cache/v_cache NULL = the pool's own.
 */
pa_status pa_copy_blocks(pa_pool *pool, const int32_t *pairs, int32_t n, void *k_cache, void *v_cache, void *stream);

/*
 * Speculative rejection sampling after the target model verified num_draft
 * draft tokens in one pass (yangyu.win blog #54, section 5 question 3;
 * maths.nthquan ch. 17 "Speculative decoding"). For each sequence b, draft
 * x_i is kept while u_i * q_i(x_i) < p_i(x_i) (fp32; i.e. with probability
 * min(1, p/q)); the first rejected position is resampled from
 * max(0, p_i - q_i) renormalised (from p_i if that has no mass) and later
 * drafts are dropped; if all are kept, one more token is drawn from
 * p_num_draft. Draws use the inverse CDF at v_b, summed as float pairs
 * (about 44 significant bits); a drawn token always has positive weight.
 *   p      device fp32 [num_seqs, num_draft + 1, vocab]  target distributions
 *   q      device fp32 [num_seqs, num_draft, vocab]      draft distributions
 *   draft  device int32 [num_seqs, num_draft]            a token outside the vocabulary counts as rejected
 *   u      device fp32 [num_seqs, num_draft]  uniforms in [0, 1) for the accept tests
 *   v      device fp32 [num_seqs]              uniforms in [0, 1) for the final draw
 *   out    device int32 [num_seqs, num_draft + 1]  kept drafts, then the drawn token, then -1
 *   n_out  device int32 [num_seqs]             tokens emitted (kept drafts + 1); 0 if the rows
 *          could not be read (a bounded wait on a copy ran out), out[b] then holds no drawn token
 * num_draft <= 64. No pool is needed.
 */
pa_status pa_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                         int32_t num_seqs, int32_t num_draft, int64_t vocab, int32_t *out, int32_t *n_out,
                         void *stream);

/*
 * Self-test of failure detection. Every wait of the kernels' copy pipelines is
 * bounded: after a time limit the kernel records PA_ERR_TIMEOUT in the pool's
 * status word and returns instead of spinning. This launches one warp that
 * waits, through the same bounded wait, on a barrier that nothing completes;
 * after limit_ns (at most 10 s) it records the timeout and returns, leaving
 * the context usable. pa_pool_check then returns PA_ERR_TIMEOUT.
 */
pa_status pa_pool_selftest_wait(pa_pool *pool, uint64_t limit_ns, void *stream);

/* Number of kernels pa_decode launches for these arguments (1, or 2 with the merge); -1 on bad args. */
int32_t pa_decode_launches(const pa_pool *pool, int32_t block_table_stride, int32_t num_seqs,
                           int32_t num_q_heads, int32_t q_len);

/*
 * Allocation-free decode.
 *
 * Some callers cannot allocate device memory: a plugin inside a host runtime
 * that owns every device allocation through its own allocator and memory
 * budget, or a latency-critical loop that must not make cudaMalloc's
 * synchronising call. Such a caller cannot create a pool, because
 * pa_pool_create allocates the split workspace. This entry point takes the
 * pool geometry directly and keeps its scratch (a status word, two work
 * counters and the split workspace) in one static device array of PA_NOALLOC_SCRATCH_BYTES, which
 * every GPU that runs it holds from its first call until the process exits.
 * The pages have no counterpart to this entry point; it computes what
 * pa_decode computes, with the same decode and merge kernels.
 *
 *  - Inputs and outputs are the caller's, with pa_decode's layouts and meaning;
 *    num_blocks .. dtype and partition_tokens (0 = 512) are as in pa_pool_config.
 *  - Scratch needed: 256 bytes (the status word and the counters with which
 *    the tensor-core kernel's CTAs share out their items; each launch leaves
 *    them at zero), plus, when P =
 *    ceil(block_table_stride * block_size / partition_tokens) > 1,
 *    num_seqs * q_len * num_q_heads * P * head_dim * 4 bytes (rounded up to
 *    256) and num_seqs * q_len * num_q_heads * P * 8. A larger request returns
 *    PA_ERR_INVALID_ARG before anything is launched.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call in a device's context, made with that device current,
 *    looks up the array's device address (again after the context is reset);
 *    make that first call before any stream capture.
 *  - Every call shares the one array and leaves its contents behind. Each call
 *    clears the status word (cudaMemsetAsync) and writes every partition slot
 *    before reading it; calls that overlap on the GPU (e.g. on two streams)
 *    race on the array and must be ordered by the caller.
 *  - There is no status word to read back. Instead, when the kernels flag
 *    anything -- a copy wait that ran out (its outputs would be left unwritten)
 *    or an out-of-range block id or context length (clamped, so the kernel
 *    does not fault) -- the call's last kernel fills the whole of `out` with
 *    NaN, so a failed call never returns stale or partial results as numbers.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

pa_status pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, int32_t num_blocks,
                            int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                            const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_q_heads, int32_t q_len, float scale,
                            int32_t partition_tokens, void *out, void *stream);

/* A static, human-readable name of a status code. */
const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
