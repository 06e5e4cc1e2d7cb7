// decode.cu -- paged-attention decode / causal verify over a block-table-mapped KV pool,
// plus the log-sum-exp merge of context partitions.
//
// What is computed (learn.tanhdev.com "Part 8: Inference optimization with vLLM",
// section on executing the kernel math in CUDA): for query row i,
//   A_{i,j} = q_i K_(j)^T / sqrt(d_k) block by block, an online softmax across blocks,
//   o_i = sum_j sum_t a_{i,j,t} v_(j,t).
// K_(j) is the j-th logical block of the sequence, found at physical block
// block_table[b][j] (itimpress.au section 1; yangyu.win blog #54 section 2.2).
//
// Work decomposition. One CTA handles one (sequence b, KV head g, context
// partition p). All q_len * G query rows that read KV head g (GQA groups;
// q_len > 1 for verifying draft tokens) are handled together, so every K/V byte
// of the partition is read from HBM once. The partition's tokens are cut into
// 16-token tiles, dealt round-robin to the CTA's W warps (4; 2 for the short
// suffix partitions of the shared-prefix decode). Each warp runs its own
// STAGES-deep pipeline: its lane 0 issues TMA tile loads (128-byte swizzle, so
// the ldmatrix reads below are bank-conflict free) completing on a per-stage
// mbarrier, and the warp consumes tiles in order.
//
// Per tile the contraction is a small dense one, done on the tensor cores with
// the keys as the M dimension (swap-AB): S^T[16 keys x 8*NT rows] = K_tile . Q^T,
// then the fp32 online softmax per query row (column), then
// O^T[D x 8*NT] += V_tile^T . P^T, where P^T comes out of the S^T accumulator
// with one movmatrix per 8x8 block. The query rows fill the N dimension (8 per
// MMA), so G = 8 heads use every column.
//
// Partitions (maths.nthquan ch. 17 "Scaling and deployment", section on sequence
// parallelism: local attention per segment, then a reduction): a CTA whose
// sequence has one partition writes the normalised output; otherwise it writes
// (unnormalised O, running max, sum) and merge_kernel combines the partitions.
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

// Pipeline stages per warp and CTAs per SM (the launch bounds; the same warps per SM whatever the warps
// per CTA, w). 16-bit stages hold 8 KB of K+V at head_dim 128, FP8 stages 4 KB of codes.
// - 16-bit pools with one 8-column tile of query rows: 2 stages and 3 CTAs per SM (12 warps, 64 KB of
//   tiles per CTA). 3 stages at 2 CTAs per SM keep more bytes in flight per warp but fewer warps and
//   CTAs to cover each CTA's start and end. Same box, six rounds against that shape: Llama-3-8B-shaped
//   0-4% faster, 70B-shaped layer and long context 0-2% faster, none slower.
// - More 16-bit rows: 3 stages at 2 CTAs per SM (the registers of 16-32 rows allow no more).
// - FP8 pools: 3 stages, 4 single-column-tile CTAs per SM (16 warps).
constexpr int PA_FP8_STAGES = 3;
__host__ __device__ constexpr int stages_for(bool kv8, int nt) { return kv8 ? PA_FP8_STAGES : (nt == 1 ? 2 : 3); }
__host__ __device__ constexpr int min_ctas_for(bool kv8, int nt, int w) {
    return (kv8 && nt == 1 ? 4 : (!kv8 && nt == 1 ? 3 : 2)) * (4 / w);
}

// Shared memory of the tile pipelines (w warps per CTA, one pipeline each). 16-bit pools: each stage
// holds the K tile then the V tile (16 rows x D 16-bit values each). FP8 pools (D = 128): each stage
// holds the K codes tile and the V codes tile (16 rows x 128 bytes each, 1024-byte aligned for the
// 128-byte swizzle); the stages' K and V scales (16 floats each) sit in a small region after all code
// tiles. The codes are converted to fp16 in registers, on their way from ldmatrix to the MMAs.
__host__ __device__ constexpr int stage_bytes(int D, bool kv8) { return kv8 ? 2 * TILE_TOKENS * 128 : 2 * TILE_TOKENS * D * 2; }
__host__ __device__ constexpr int scale_region(bool kv8, int nt, int w) {
    return kv8 ? w * stages_for(kv8, nt) * 2 * TILE_TOKENS * 4 : 0;
}
__host__ __device__ constexpr int ring_bytes(int D, bool kv8, int nt, int w) {
    return w * stages_for(kv8, nt) * stage_bytes(D, kv8) + (kv8 ? ((scale_region(kv8, nt, w) + 1023) & ~1023) : 0);
}
__host__ __device__ constexpr int merge_bytes(int D, int nt, int w) {
    return w * nt * 8 * (D + 4) * 4 + w * nt * 8 * 2 * 4 + nt * 8 * (w + 2) * 4;
}
__host__ __device__ constexpr int body_bytes(int D, int nt, bool kv8, int w) {
    return ring_bytes(D, kv8, nt, w) > merge_bytes(D, nt, w) ? ring_bytes(D, kv8, nt, w) : merge_bytes(D, nt, w);
}

static size_t smem_bytes(int D, int nt, bool kv8, int table_entries, int w = DECODE_WARPS) {
    return 1024 /* alignment slack */ + (size_t)body_bytes(D, nt, kv8, w) + w * stages_for(kv8, nt) * 8 +
           (size_t)table_entries * 4;
}

size_t decode_smem_bytes(int head_dim, int nt) { return smem_bytes(head_dim, nt, false, 0); }

constexpr float DEC_RESCALE_LOG2 = 8.f;   // stale-maximum headroom of the decode softmax (P <= 2^8)

template <typename T, int D, int NT, bool KV8, int W>
__global__ void __launch_bounds__(W * 32, min_ctas_for(KV8, NT, W))
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
    static_assert(!KV8 || D == 128, "FP8 pools are built for head_dim 128");
    // FP8 pools compute in fp16 whatever the model dtype: E4M3 codes are exact in fp16 (one cvt per
    // pair), bf16 queries are exact in fp16 within its normal range, and P times the V scale keeps
    // fp16's 11 bits. Outputs are rounded to T.
    using M = typename std::conditional<KV8, __half, T>::type;
    constexpr int HALVES = D / 64;                     // 128-byte swizzle spans per key row
    constexpr int HALF_BYTES = TILE_TOKENS * 128;      // one span of a 16-row tile
    constexpr int TILE_BYTES = TILE_TOKENS * D * 2;    // K (or V) of one 16-bit tile
    constexpr int STAGE_BYTES = stage_bytes(D, KV8);
    constexpr int CODE_BYTES = TILE_TOKENS * 128;      // FP8: K (or V) codes of one tile
    constexpr int KSTEPS = D / 16;
    constexpr int MT = D / 16;                         // m16 tiles of the head dimension (P.V)
    constexpr int STAGES = stages_for(KV8, NT);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    const uint32_t bars_u32 = base_u32 + body_bytes(D, NT, KV8, W);
    int *tbl = reinterpret_cast<int *>(smem + body_bytes(D, NT, KV8, W) + W * STAGES * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nlaunch = p.max_parts - p.part0;         // partitions launched per (sequence, KV head)
    // CTA order over (unit = (sequence, KV head), partition): 16-bit pools take a unit's partitions one
    // after another; FP8 pools take every unit's last partition first, then the one before, and so on.
    // Measured on one box, three rounds: for FP8 the Llama-3-8B-shaped and long-context decodes were ~2%
    // faster that way and the 70B-shaped one unchanged; for 16-bit pools it was no faster (0-1% slower),
    // and partition-major in ascending order was 2-4% slower.
    const int units = (int)(gridDim.x / nlaunch);
    const int part = KV8 ? p.part0 + (nlaunch - 1 - (int)(blockIdx.x / units)) : p.part0 + (int)(blockIdx.x % nlaunch);
    const int bg = KV8 ? (int)(blockIdx.x % units) : (int)(blockIdx.x / nlaunch);
    // launched with programmatic serialization: the merge behind this kernel may be launched now (its CTAs
    // take only what this grid leaves free and wait for its end); this kernel waits for the work ahead of it
    pdl_trigger();
    pdl_wait();
    const int g = bg % p.Hkv;
    const int b = bg / p.Hkv;

    // ---- query fragments: B operand (col-major 16 x 8) of S^T = K . Q^T (loaded first: their latency
    // overlaps the context length and block table loads below)
    const int gq = lane >> 2;   // MMA group id: key row within an 8-row half; query column for B
    const int tq = lane & 3;    // thread in group
    uint32_t qf[NT][KSTEPS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 8 + gq;
        if (r < p.rows) {
            const int qi = r / p.G, hh = r - (r / p.G) * p.G;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const T *>(p.q) + (((int64_t)b * p.q_len + qi) * p.Hq + g * p.G + hh) * D);
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                // FP8 pools: the K codes reach the MMA with each lane holding 4 consecutive dims
                // (16 ks + 4 tq ..), so the contraction index is permuted the same way for Q
                qf[nt][ks][0] = __ldg(qrow + ks * 8 + (KV8 ? 2 * tq : tq));
                qf[nt][ks][1] = __ldg(qrow + ks * 8 + (KV8 ? 2 * tq + 1 : 4 + tq));
                if constexpr (KV8 && std::is_same<T, __nv_bfloat16>::value) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const __nv_bfloat162 bq = *reinterpret_cast<const __nv_bfloat162 *>(&qf[nt][ks][e]);
                        const float2 f = __bfloat1622float2(bq);
                        qf[nt][ks][e] = pack2<__half>(f.x, f.y);
                    }
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) qf[nt][ks][0] = qf[nt][ks][1] = 0u;
        }
    }
    // ---- context of this sequence, clamped to what the table / launch can hold
    int L = __ldg(p.context_lens + b);
    if (L < p.q_len || L > p.max_ctx) {
        if (threadIdx.x == 0 && part == 0) set_status(p.status, STATUS_BOUNDS);
        L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
    }
    if (p.part0 > 0 && part == p.part0 && g == 0) {
        // shared-prefix decode: the prefix kernel read sequence 0's blocks for every sequence and
        // assumed that every query row follows the whole prefix; check both for this sequence
        const int pre_blocks = p.part0 * p.part_tokens / p.bs;
        if (L - p.q_len < p.part0 * p.part_tokens) {
            if (threadIdx.x == 0) set_status(p.status, STATUS_BOUNDS);
        }
        for (int i = threadIdx.x; i < pre_blocks; i += blockDim.x)
            if (__ldg(p.block_tables + (int64_t)b * p.stride + i) != __ldg(p.block_tables + i))
                set_status(p.status, STATUS_BOUNDS);
    }
    const int nparts = (L + p.part_tokens - 1) / p.part_tokens;
    if (part >= nparts) return;
    const int t_begin = part * p.part_tokens;
    const int ntok = min(p.part_tokens, L - t_begin);
    const int ntiles = (ntok + TILE_TOKENS - 1) / TILE_TOKENS;
    const int blk0 = t_begin / p.bs;
    const int nblk = (ntok + p.bs - 1) / p.bs;

    // ---- this partition's block ids (block-table gather), validated
    const int32_t *trow = p.block_tables + (int64_t)b * p.stride + blk0;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
        int id = __ldg(trow + i);
        if (id < 0 || id >= p.num_blocks) {
            set_status(p.status, STATUS_BOUNDS);
            id = 0;
        }
        tbl[i] = id;
    }
    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(bars_u32 + (warp * STAGES + s) * 8, 1);
        fence_barrier_init();
    }
    __syncthreads();

    const int my_tiles = ntiles > warp ? (ntiles - warp + W - 1) / W : 0;
    const uint32_t ring_u32 = base_u32 + warp * STAGES * STAGE_BYTES;
    const uint32_t scales_u32 = base_u32 + W * STAGES * STAGE_BYTES;                 // FP8 only
    const uint64_t policy = l2_policy_evict_first();

    auto issue = [&](int it) {
        const int i = warp + it * W;          // tile index within the partition
        const int s = it % STAGES;
        const int tok = i * TILE_TOKENS;                 // token offset within the partition
        const int row0 = (tbl[tok / p.bs] * p.Hkv + g) * p.bs + (tok % p.bs);
        const uint32_t bar = bars_u32 + (warp * STAGES + s) * 8;
        const uint32_t kdst = ring_u32 + s * STAGE_BYTES;
        fence_proxy_async_smem();
        if constexpr (KV8) {
            const uint32_t sdst = scales_u32 + (warp * STAGES + s) * 2 * TILE_TOKENS * 4;
            mbar_arrive_expect_tx(bar, 2 * CODE_BYTES + 2 * TILE_TOKENS * 4);
            tma_load_2d(kdst, &tmk, 0, row0, bar, policy);
            tma_load_2d(kdst + CODE_BYTES, &tmv, 0, row0, bar, policy);
            bulk_load(sdst, p.k_scales + row0, TILE_TOKENS * 4, bar, policy);
            bulk_load(sdst + TILE_TOKENS * 4, p.v_scales + row0, TILE_TOKENS * 4, bar, policy);
        } else {
            mbar_arrive_expect_tx(bar, STAGE_BYTES);
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
                tma_load_2d(kdst + h * HALF_BYTES, &tmk, h * 64, row0, bar, policy);
                tma_load_2d(kdst + TILE_BYTES + h * HALF_BYTES, &tmv, h * 64, row0, bar, policy);
            }
        }
    };

    int issued = 0;
    if (lane == 0) {
        const int n0 = my_tiles < STAGES ? my_tiles : STAGES;
        for (int it = 0; it < n0; ++it) issue(it);
    }
    issued = my_tiles < STAGES ? my_tiles : STAGES;

    // causal limit (inclusive) of the query columns this thread accumulates
    int lim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            int r = nt * 8 + 2 * tq + j;
            int qi = r / p.G;
            if (qi > p.q_len - 1) qi = p.q_len - 1;
            lim[nt][j] = L - p.q_len + qi;
        }

    float m[NT][2], l[NT][2], o[MT][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int md = 0; md < MT; ++md) o[md][nt][0] = o[md][nt][1] = o[md][nt][2] = o[md][nt][3] = 0.f;
    }

    bool ok = true;
    int it = 0;
    for (; it < my_tiles; ++it) {
        const int s = it % STAGES;
        if (!mbar_wait_bounded(bars_u32 + (warp * STAGES + s) * 8, (uint32_t)(it / STAGES) & 1u, p.wait_ns)) {
            ok = false;
            break;
        }
        const int i = warp + it * W;
        const int tile_t0 = t_begin + i * TILE_TOKENS;   // absolute token index of the tile's first row
        const int gq_ = lane >> 2;
        uint32_t kb = ring_u32 + s * STAGE_BYTES;
        uint32_t vb = kb + TILE_BYTES;
        float ks_lo = 1.f, ks_hi = 1.f, vs_lo = 1.f, vs_hi = 1.f;   // FP8: scales of this thread's key rows
        if constexpr (KV8) {
            // K and V codes enter the MMAs straight from the stage (exact in fp16). The K scale
            // multiplies the scores and the V scale multiplies P.
            const float *sk = reinterpret_cast<const float *>(smem + (scales_u32 - base_u32)) +
                              (warp * STAGES + s) * 2 * TILE_TOKENS;
            const float *sv = sk + TILE_TOKENS;
            ks_lo = sk[gq_] * p.scale_log2;
            ks_hi = sk[gq_ + 8] * p.scale_log2;
            vs_lo = sv[gq_];
            vs_hi = sv[gq_ + 8];
            vb = kb + CODE_BYTES;
        }

        // Rows past the context hold other data (possibly NaN): zero them in V so that
        // 0-weight x row stays 0 in the P.V product. Scores of those rows are masked below.
        const int nvalid = L - tile_t0;
        if (!KV8 && nvalid < TILE_TOKENS) {
            const int nz = (TILE_TOKENS - nvalid) * 8;   // 16-byte chunks per span
            uint8_t *vgen = smem + (vb - base_u32);
            for (int c = lane; c < nz * HALVES; c += 32) {
                const int h = c / nz, rc = c - (c / nz) * nz;
                *reinterpret_cast<uint4 *>(vgen + h * HALF_BYTES + (nvalid + rc / 8) * 128 + (rc % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // S^T = K . Q^T (16 keys x 8*NT query columns)
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        if constexpr (KV8) {
            // ldmatrix.x4 on the codes viewed as 16-bit pairs: matrices (keys 0-7 | 8-15) x (chunk
            // 2kp | 2kp+1), each lane receiving 4 consecutive codes (dims 16c + 4tq ..) of key gq or
            // gq + 8. Codes 0-1 / 2-3 are the A fragment's k pairs (2tq) / (2tq + 8) of the permuted
            // contraction index.
            const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kp = 0; kp < KSTEPS / 2; ++kp) {
                const int chunk = kp * 2 + (lane >> 4);
                const uint32_t addr = kb + krow * 128 + ((chunk ^ (krow & 7)) << 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(addr, r0, r1, r2, r3);
                const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)r0), a2 = e4m3x2_to_f16x2((uint16_t)(r0 >> 16));
                const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)r1), a3 = e4m3x2_to_f16x2((uint16_t)(r1 >> 16));
                const uint32_t c0 = e4m3x2_to_f16x2((uint16_t)r2), c2 = e4m3x2_to_f16x2((uint16_t)(r2 >> 16));
                const uint32_t c1 = e4m3x2_to_f16x2((uint16_t)r3), c3 = e4m3x2_to_f16x2((uint16_t)(r3 >> 16));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816<M>(sacc[nt], a0, a1, a2, a3, qf[nt][2 * kp][0], qf[nt][2 * kp][1]);
                    mma_16816<M>(sacc[nt], c0, c1, c2, c3, qf[nt][2 * kp + 1][0], qf[nt][2 * kp + 1][1]);
                }
            }
        } else {
            const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const int chunk = ks * 2 + (lane >> 4);
                const uint32_t addr = kb + (chunk >> 3) * HALF_BYTES + krow * 128 + (((chunk & 7) ^ (krow & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816<M>(sacc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
            }
        }

        // online softmax per query column (log2 domain). Each column keeps a reference maximum that
        // moves only when the tile's maximum passes it by more than 2^DEC_RESCALE_LOG2, so P <= 2^8 and
        // O is rescaled on few tiles (O and l are relative to the reference, exactly as to a true max).
        const int t_lo = tile_t0 + gq, t_hi = t_lo + 8;
        float alpha[NT][2];
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float s0 = t_lo <= lim[nt][j] ? sacc[nt][j] * (KV8 ? ks_lo : p.scale_log2) : -INFINITY;
                const float s1 = t_hi <= lim[nt][j] ? sacc[nt][2 + j] * (KV8 ? ks_hi : p.scale_log2) : -INFINITY;
                float mx = fmaxf(s0, s1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                alpha[nt][j] = 1.f;
                if (mx > m[nt][j] + DEC_RESCALE_LOG2) {   // also the first finite maximum (m = -inf)
                    alpha[nt][j] = ex2_approx(m[nt][j] - mx);
                    m[nt][j] = mx;
                    rescale = true;
                }
                const float muse = m[nt][j] == -INFINITY ? 0.f : m[nt][j];
                const float p0 = ex2_approx(s0 - muse), p1 = ex2_approx(s1 - muse);
                l[nt][j] = l[nt][j] * alpha[nt][j] + p0 + p1;
                if constexpr (KV8) {
                    // V scale of each key row; rows past the context have no scale (select, not multiply)
                    sacc[nt][j] = t_lo < L ? p0 * vs_lo : 0.f;
                    sacc[nt][2 + j] = t_hi < L ? p1 * vs_hi : 0.f;
                } else {
                    sacc[nt][j] = p0;
                    sacc[nt][2 + j] = p1;
                }
            }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int md = 0; md < MT; ++md) {
                        o[md][nt][j] *= alpha[nt][j];
                        o[md][nt][2 + j] *= alpha[nt][j];
                    }
        }

        // P^T as the B operand (16 keys x 8 columns): transpose the two 8x8 halves of S^T.
        // The MMA takes P in V's 16-bit type. bf16 keeps 8 mantissa bits, too few for short
        // contexts whose weighted values cancel, so for bf16 P is carried as hi + lo bf16 parts
        // (hi = bf16(P), lo = bf16(P - hi)) and P.V is two MMAs; fp16's 11 bits suffice alone.
        constexpr bool SPLIT_P = std::is_same<M, __nv_bfloat16>::value;
        uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if constexpr (SPLIT_P) {
                // a bf16 is the top half of an fp32: the high parts are unpacked from their packed pair
                const uint32_t h01 = pack2<M>(sacc[nt][0], sacc[nt][1]);
                const uint32_t h23 = pack2<M>(sacc[nt][2], sacc[nt][3]);
                const uint32_t l01 = pack2<M>(sacc[nt][0] - __uint_as_float(h01 << 16),
                                              sacc[nt][1] - __uint_as_float(h01 & 0xFFFF0000u));
                const uint32_t l23 = pack2<M>(sacc[nt][2] - __uint_as_float(h23 << 16),
                                              sacc[nt][3] - __uint_as_float(h23 & 0xFFFF0000u));
                pb[nt][0] = movmatrix_trans(h01);
                pb[nt][1] = movmatrix_trans(h23);
                pl[nt][0] = movmatrix_trans(l01);
                pl[nt][1] = movmatrix_trans(l23);
            } else {
                pb[nt][0] = movmatrix_trans(pack2<M>(sacc[nt][0], sacc[nt][1]));
                pb[nt][1] = movmatrix_trans(pack2<M>(sacc[nt][2], sacc[nt][3]));
                pl[nt][0] = pl[nt][1] = 0u;
            }
        }

        if constexpr (KV8) {
            if (nvalid < TILE_TOKENS) {                   // V code rows past the context: zero (may be NaN)
                uint8_t *vgen = smem + (vb - base_u32);
                for (int c = lane; c < (TILE_TOKENS - nvalid) * 8; c += 32)
                    *reinterpret_cast<uint4 *>(vgen + (nvalid + c / 8) * 128 + (c % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                __syncwarp();
            }
        }

        // O^T += V^T . P^T
        if constexpr (KV8) {
            // ldmatrix.x4.trans on the codes viewed as 16-bit pairs: matrices (keys 0-7 | 8-15) x
            // (chunk 2mp | 2mp+1); each lane receives keys 2tq, 2tq+1 x dims 2gq, 2gq+1 of the chunk.
            // Bytes (0, 2) / (1, 3) give the A fragment of V^T whose rows are the chunk's even / odd
            // dims (row m <-> dim 16 md + 2 (m % 8) + m / 8, undone when O is written).
            const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mp = 0; mp < MT / 2; ++mp) {
                const int chunk = mp * 2 + (lane >> 4);
                const uint32_t addr = vb + vrow * 128 + ((chunk ^ (vrow & 7)) << 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_trans(addr, r0, r1, r2, r3);
                const uint32_t rr[4] = {r0, r1, r2, r3};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t lo = rr[2 * h], hi = rr[2 * h + 1];   // keys 0-7 / 8-15 of chunk 2mp + h
                    const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)__byte_perm(lo, 0u, 0x4420));
                    const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)__byte_perm(lo, 0u, 0x4431));
                    const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)__byte_perm(hi, 0u, 0x4420));
                    const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)__byte_perm(hi, 0u, 0x4431));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_16816<M>(o[2 * mp + h][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
        } else {
            const int vrow = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
            for (int md = 0; md < MT; ++md) {
                const int chunk = md * 2 + ((lane >> 3) & 1);
                const uint32_t addr = vb + (chunk >> 3) * HALF_BYTES + vrow * 128 + (((chunk & 7) ^ (vrow & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816<M>(o[md][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    if constexpr (SPLIT_P) mma_16816<M>(o[md][nt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
                }
            }
        }
        __syncwarp();
        if (it + STAGES < my_tiles) {
            if (lane == 0) issue(it + STAGES);
            ++issued;
        }
    }

    // full row sums of this warp (the 8 lanes sharing a column hold disjoint keys)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float v = l[nt][j];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            l[nt][j] = v;
        }

    if (__syncthreads_or(!ok)) {
        // A copy did not arrive in time: record it, wait (bounded) for this warp's copies still in
        // flight so none lands after the CTA exits, and leave without writing results.
        if (threadIdx.x == 0) set_status(p.status, STATUS_TIMEOUT);
        if (lane == 0)
            for (int k = it; k < issued; ++k)
                mbar_wait_bounded(bars_u32 + (warp * STAGES + (k % STAGES)) * 8, (uint32_t)(k / STAGES) & 1u,
                                  p.wait_ns);
        return;
    }

    // ---- combine the W warps (smem; the tile ring is free now)
    constexpr int RP = NT * 8;
    constexpr int OSTR = D + 4;   // padded row: the fragment stores below hit 32 distinct banks
    float *ow = reinterpret_cast<float *>(smem);
    float *mlw = ow + W * RP * OSTR;
#pragma unroll
    for (int md = 0; md < MT; ++md)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                // FP8 pools: O's rows are the chunk's even dims, then its odd dims
                const int dim = KV8 ? md * 16 + 2 * gq + (e >> 1) : md * 16 + gq + (e >> 1) * 8;
                const int col = nt * 8 + 2 * tq + (e & 1);
                ow[(warp * RP + col) * OSTR + dim] = o[md][nt][e];
            }
    if (gq == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = nt * 8 + 2 * tq + j;
                mlw[(warp * RP + col) * 2] = m[nt][j];
                mlw[(warp * RP + col) * 2 + 1] = l[nt][j];
            }
    }
    __syncthreads();
    // per row: the running max over the warps, each warp's factor 2^(m_w - M) and the row sum, once
    float *wsc = mlw + W * RP * 2;           // [RP][W] factors, then [RP][2] (M, sum)
    float *rml = wsc + RP * W;
    for (int r = threadIdx.x; r < p.rows; r += blockDim.x) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, mlw[(w * RP + r) * 2]);
        const float Muse = M == -INFINITY ? 0.f : M;
        float ls = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float sc = exp2f(mlw[(w * RP + r) * 2] - Muse);
            wsc[r * W + w] = sc;
            ls += sc * mlw[(w * RP + r) * 2 + 1];
        }
        rml[r * 2] = M;
        rml[r * 2 + 1] = ls;
    }
    __syncthreads();

    // 8 dims of one row per thread and step (out is 16-byte aligned: every entry point checks it)
    const bool direct = nparts == 1 && p.part0 == 0;
    constexpr int D8 = D / 8;
    for (int idx = threadIdx.x; idx < p.rows * D8; idx += blockDim.x) {
        const int r = idx / D8;
        const int d0 = (idx - r * D8) * 8;
        const float M = rml[r * 2], ls = rml[r * 2 + 1];
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float sc = wsc[r * W + w];
            const float4 a = *reinterpret_cast<const float4 *>(ow + (w * RP + r) * OSTR + d0);
            const float4 c = *reinterpret_cast<const float4 *>(ow + (w * RP + r) * OSTR + d0 + 4);
            acc[0] += sc * a.x;
            acc[1] += sc * a.y;
            acc[2] += sc * a.z;
            acc[3] += sc * a.w;
            acc[4] += sc * c.x;
            acc[5] += sc * c.y;
            acc[6] += sc * c.z;
            acc[7] += sc * c.w;
        }
        const int qi = r / p.G;
        const int h = g * p.G + (r - qi * p.G);
        const int64_t orow = ((int64_t)b * p.q_len + qi) * p.Hq + h;
        if (direct) {
            *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) + orow * D + d0) =
                make_uint4(pack2<T>(acc[0] / ls, acc[1] / ls), pack2<T>(acc[2] / ls, acc[3] / ls),
                           pack2<T>(acc[4] / ls, acc[5] / ls), pack2<T>(acc[6] / ls, acc[7] / ls));
        } else {
            const int64_t prow = orow * p.max_parts + part;
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * D + d0);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (d0 == 0) p.part_ml[prow] = make_float2(M, ls);
        }
    }
}

// Log-sum-exp merge of the partitions of one sequence's query position qi and KV head g
// (its G output rows):
//   M = max_p m_p,  w_p = 2^(m_p - M) (0 for an empty partition),
//   out = sum_p w_p O_p / sum_p w_p l_p
// Phase 1: warp r of the CTA reads all (m_p, l_p) of row r at once and leaves the weights in
// shared memory. Phase 2: MERGE_THREADS threads are split into groups; each thread owns one
// (row, 4 dims) pair and sums a fixed subset of partitions with independent loads; the group
// sums are added in group order. The result does not depend on timing.
constexpr int MERGE_THREADS = 512;

// Shared-memory layout of merge_kernel, in floats: weights [G][max_parts], den [G], then the
// float4 group sums. Each region starts on a 16-byte boundary.
__host__ __device__ inline int merge_wt_floats(int G, int max_parts) { return (G * max_parts + 3) & ~3; }
__host__ __device__ inline int merge_den_floats(int G) { return (G + 3) & ~3; }
// Thread groups per (row, 4 dims) pair: about 8 partitions per thread, at most MERGE_THREADS threads.
__host__ __device__ inline int merge_groups(int pairs, int max_parts) {
    int g = (max_parts + 7) / 8;
    const int cap = MERGE_THREADS / pairs > 0 ? MERGE_THREADS / pairs : 1;
    return g < 1 ? 1 : (g > cap ? cap : g);
}
__host__ __device__ inline int merge_threads(int pairs, int max_parts) {
    int t = pairs * merge_groups(pairs, max_parts);
    t = t > MERGE_THREADS ? MERGE_THREADS : t;
    return (t + 31) & ~31;
}

template <typename T, int D>
__global__ void __launch_bounds__(MERGE_THREADS) merge_kernel(const DecodeParams p) {
    pdl_wait();   // the partitions' states are written by the kernel ahead of this one
    extern __shared__ float msm[];                 // weights [G][max_parts], den [G], sums [groups][pairs]
    const int unit = blockIdx.x / p.merge_splits;  // (b, qi, g)
    const int split = blockIdx.x - unit * p.merge_splits;
    const int g = unit % p.Hkv;
    const int bq = unit / p.Hkv;                   // b * q_len + qi
    const int b = bq / p.q_len;
    int L = __ldg(p.context_lens + b);
    L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
    const int nparts = (L + p.part_tokens - 1) / p.part_tokens;
    if (nparts <= 1) return;
    const int G = p.G;
    float *wt = msm;                               // [G][max_parts]
    float *den = wt + merge_wt_floats(G, p.max_parts);   // [G]
    float4 *sums = reinterpret_cast<float4 *>(den + merge_den_floats(G));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)bq * p.Hq + g * G;   // first output row of the unit

    const int nthreads = blockDim.x;
    for (int r = warp; r < G; r += nthreads / 32) {
        const float2 *ml = p.part_ml + (row0 + r) * p.max_parts;
        float M = -INFINITY;
        for (int pp = lane; pp < nparts; pp += 32) {
            const float2 v = __ldcg(ml + pp);
            if (v.y > 0.f) M = fmaxf(M, v.x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float ds = 0.f;
        for (int pp = lane; pp < nparts; pp += 32) {
            const float2 v = __ldcg(ml + pp);
            const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
            wt[r * p.max_parts + pp] = w;
            ds += w * v.y;
        }
        // fixed-order sum over lanes
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
        if (lane == 0) den[r] = ds;
    }
    __syncthreads();

    // this CTA's share of the unit's (row, 4 dims) pairs
    const int all_pairs = G * (D / 4);
    const int pps = (all_pairs + p.merge_splits - 1) / p.merge_splits;
    const int pair0 = split * pps;
    const int pairs = min(pps, all_pairs - pair0);
    if (pairs <= 0) return;
    const int groups = merge_groups(pps, p.max_parts);
    for (int t = threadIdx.x; t < pairs * groups; t += nthreads) {
        const int pair = pair0 + t % pairs;
        const int grp = t / pairs;
        const int r = pair / (D / 4);
        const int d4 = pair - r * (D / 4);
        const float4 *po = reinterpret_cast<const float4 *>(p.part_o + (row0 + r) * p.max_parts * D) + d4;
        const float *w = wt + r * p.max_parts;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int pp = grp; pp < nparts; pp += groups) {
            const float c = w[pp];
            if (c == 0.f) continue;                    // an empty partition: its O is not read (it may be unwritten)
            const float4 x = __ldcg(po + (int64_t)pp * (D / 4));
            acc.x += c * x.x;
            acc.y += c * x.y;
            acc.z += c * x.z;
            acc.w += c * x.w;
        }
        sums[grp * pairs + (pair - pair0)] = acc;
    }
    __syncthreads();
    for (int q0 = threadIdx.x; q0 < pairs; q0 += nthreads) {
        const int q = pair0 + q0;
        float4 t = sums[q0];
        for (int k = 1; k < groups; ++k) {
            const float4 u = sums[k * pairs + q0];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        const int r = q / (D / 4);
        const int d4 = q - r * (D / 4);
        const float inv = 1.f / den[r];
        T *out = reinterpret_cast<T *>(p.out) + (row0 + r) * D + d4 * 4;
        const uint32_t lo = pack2<T>(t.x * inv, t.y * inv), hi = pack2<T>(t.z * inv, t.w * inv);
        *reinterpret_cast<uint2 *>(out) = make_uint2(lo, hi);
    }
}

// The same merge with one warp per output row, for at most 32 partitions: lane pp holds partition
// pp's (max, sum), the weights and their sum come from warp shuffles, and each lane accumulates
// D / 32 dims over the partitions in order. No block barrier. The context length, every launched
// partition's (max, sum) and the O of the first MERGE_SPEC partitions are loaded in one round,
// before it is known which of them hold data: values of partitions past the context or of zero
// weight (possibly never written) are selected away, never multiplied.
constexpr int MERGE_ROW_WARPS = 8;
constexpr int MERGE_SPEC = 8;

template <typename T, int D>
__global__ void __launch_bounds__(MERGE_ROW_WARPS * 32) merge_rows_kernel(const DecodeParams p) {
    static_assert(D % 32 == 0 && D / 32 <= 4, "dims per lane");
    constexpr int DL = D / 32;                     // dims per lane
    pdl_wait();   // the partitions' states are written by the kernel ahead of this one
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * MERGE_ROW_WARPS + warp;   // (b * q_len + qi) * Hq + h
    if (row >= (int64_t)p.num_seqs * p.q_len * p.Hq) return;
    const int b = (int)(row / p.Hq) / p.q_len;
    const float *po = p.part_o + row * p.max_parts * D + lane * DL;
    int L = __ldg(p.context_lens + b);
    const float2 v0 = lane < p.max_parts ? __ldcg(p.part_ml + row * p.max_parts + lane) : make_float2(0.f, 0.f);
    float x[MERGE_SPEC][DL];
#pragma unroll
    for (int pp = 0; pp < MERGE_SPEC; ++pp) {
        if (pp < p.max_parts) {
            if constexpr (DL == 4) {
                const float4 t = __ldcg(reinterpret_cast<const float4 *>(po + (int64_t)pp * D));
                x[pp][0] = t.x, x[pp][1] = t.y, x[pp][2] = t.z, x[pp][3] = t.w;
            } else {
#pragma unroll
                for (int i = 0; i < DL; ++i) x[pp][i] = __ldcg(po + (int64_t)pp * D + i);
            }
        } else {
#pragma unroll
            for (int i = 0; i < DL; ++i) x[pp][i] = 0.f;
        }
    }
    L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
    const int nparts = (L + p.part_tokens - 1) / p.part_tokens;
    if (nparts <= 1) return;
    const float2 v = lane < nparts ? v0 : make_float2(0.f, 0.f);
    float M = v.y > 0.f ? v.x : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
    float ds = w * v.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
    float acc[DL];
#pragma unroll
    for (int i = 0; i < DL; ++i) acc[i] = 0.f;
#pragma unroll
    for (int pp = 0; pp < MERGE_SPEC; ++pp) {
        const float c = __shfl_sync(0xffffffffu, w, pp);   // 0 for partitions past the context
        if (c != 0.f) {
#pragma unroll
            for (int i = 0; i < DL; ++i) acc[i] += c * x[pp][i];
        }
    }
#pragma unroll 4
    for (int pp = MERGE_SPEC; pp < nparts; ++pp) {
        const float c = __shfl_sync(0xffffffffu, w, pp);
        if (c == 0.f) continue;                    // an empty partition: its O is not read (it may be unwritten)
        if constexpr (DL == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(po + (int64_t)pp * D));
            acc[0] += c * t.x;
            acc[1] += c * t.y;
            acc[2] += c * t.z;
            acc[3] += c * t.w;
        } else {
#pragma unroll
            for (int i = 0; i < DL; ++i) acc[i] += c * __ldcg(po + (int64_t)pp * D + i);
        }
    }
    const float inv = 1.f / ds;
    T *out = reinterpret_cast<T *>(p.out) + row * D + lane * DL;
    if constexpr (DL == 4) {
        *reinterpret_cast<uint2 *>(out) = make_uint2(pack2<T>(acc[0] * inv, acc[1] * inv), pack2<T>(acc[2] * inv, acc[3] * inv));
    } else {
#pragma unroll
        for (int i = 0; i < DL; i += 2) *reinterpret_cast<uint32_t *>(out + i) = pack2<T>(acc[i] * inv, acc[i + 1] * inv);
    }
}

// ------------------------------------------------------------------ launchers

template <typename T, int D, int NT, bool KV8, int W>
static cudaError_t launch_decode_t(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   cudaStream_t stream) {
    const size_t smem = smem_bytes(D, NT, KV8, (p.part_tokens + p.bs - 1) / p.bs, W);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, NT, KV8, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)p.num_seqs * p.Hkv * (p.max_parts - p.part0);
    e = launch_pdl(decode_kernel<T, D, NT, KV8, W>, dim3((unsigned)grid), dim3(W * 32), smem, stream, tmk, tmv, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Warps per CTA: 4, except for the suffix pass of the shared-prefix decode, whose (sequence, KV head)
// units hold a few hundred tokens each. There each CTA's fixed costs (query, context length and
// block-table loads, the pipeline fill, the combine of the warps' states) weigh on few tiles per warp;
// two-warp CTAs (twice the CTAs per SM) give each warp twice the tiles: 0.068 -> 0.065 ms on the
// shared-prefix verify workload. One warp per CTA, or two elsewhere, measured slower or no faster.
template <typename T, int D, int NT, bool KV8>
static cudaError_t launch_decode_w(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   cudaStream_t stream) {
    if constexpr (!KV8 && D == 128)
        if (p.part0 > 0) return launch_decode_t<T, D, NT, KV8, 2>(p, tmk, tmv, stream);
    return launch_decode_t<T, D, NT, KV8, DECODE_WARPS>(p, tmk, tmv, stream);
}

template <typename T, int D, bool KV8>
static cudaError_t launch_decode_d(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   cudaStream_t stream) {
    switch ((p.rows + 7) / 8) {
        case 1: return launch_decode_w<T, D, 1, KV8>(p, tmk, tmv, stream);
        case 2: return launch_decode_w<T, D, 2, KV8>(p, tmk, tmv, stream);
        case 3: return launch_decode_w<T, D, 3, KV8>(p, tmk, tmv, stream);
        case 4: return launch_decode_w<T, D, 4, KV8>(p, tmk, tmv, stream);
        default: return cudaErrorInvalidValue;
    }
}

// The tensor-core kernel of verify.cu takes 16-bit pools with head_dim 128 when a KV head has more than one
// 8-column MMA tile of query rows here (9..32 rows). Measured against this kernel: 1.45x for the 70B-shaped
// 4-draft verify (32 rows, 8192 tokens), 1.48x for 32 fp16 rows at 4096 tokens, 1.37x for a 32-head group at
// 32768 tokens, 1.16x for 20 rows (q_len 5, G 4) at 8192 tokens, 1.13x on the shared-prefix verify workload,
// 1.04x for 128 sequences of 1088..1536 tokens, 0.98x for 12 rows at 2000 tokens.
bool decode_uses_verify(int head_dim, int rows, bool kv8) { return !kv8 && head_dim == 128 && rows > 8; }

cudaError_t launch_decode(const DecodeParams &p, int dtype, int head_dim, const CUtensorMap &tmk,
                          const CUtensorMap &tmv, cudaStream_t stream, bool kv8) {
    if (p.allow_verify && decode_uses_verify(head_dim, p.rows, kv8)) {
        int ctas = p.vf_ctas;
        if (ctas <= 0) {
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return cudaErrorInvalidValue;
        }
        return launch_verify(p, dtype, tmk, tmv, ctas, stream);
    }
    if (kv8) {
        if (head_dim != 128) return cudaErrorInvalidValue;
        if (dtype == PA_FP16) return launch_decode_d<__half, 128, true>(p, tmk, tmv, stream);
        return launch_decode_d<__nv_bfloat16, 128, true>(p, tmk, tmv, stream);
    }
    if (dtype == PA_FP16) {
        if (head_dim == 128) return launch_decode_d<__half, 128, false>(p, tmk, tmv, stream);
        if (head_dim == 64) return launch_decode_d<__half, 64, false>(p, tmk, tmv, stream);
    } else {
        if (head_dim == 128) return launch_decode_d<__nv_bfloat16, 128, false>(p, tmk, tmv, stream);
        if (head_dim == 64) return launch_decode_d<__nv_bfloat16, 64, false>(p, tmk, tmv, stream);
    }
    return cudaErrorInvalidValue;
}

size_t merge_smem_bytes(int G, int max_parts, int head_dim, int splits) {
    const int pps = (G * (head_dim / 4) + splits - 1) / splits;
    return (size_t)(merge_wt_floats(G, max_parts) + merge_den_floats(G)) * sizeof(float) +
           (size_t)merge_groups(pps, max_parts) * pps * sizeof(float4);
}

// Merge CTAs per unit: enough for about two CTAs per SM, each keeping at least 8 (row, 4-dim) pairs.
int merge_splits_for(int64_t units, int G, int head_dim, int sm_count) {
    const int pairs = G * (head_dim / 4);
    if (units <= 0 || sm_count <= 0) return 1;
    int64_t want = (2LL * sm_count + units - 1) / units;
    const int cap = pairs / 8 > 0 ? pairs / 8 : 1;
    if (want > cap) want = cap;
    return want < 1 ? 1 : (int)want;
}

cudaError_t launch_merge(const DecodeParams &p, int dtype, int head_dim, cudaStream_t stream, bool pdl) {
    cudaError_t e = cudaSuccess;
    if (p.max_parts <= 32) {
        const int64_t rows = (int64_t)p.num_seqs * p.q_len * p.Hq;
        const unsigned grid = (unsigned)((rows + MERGE_ROW_WARPS - 1) / MERGE_ROW_WARPS);
        if (dtype == PA_FP16) {
            if (head_dim == 128) e = launch_maybe_pdl(pdl, merge_rows_kernel<__half, 128>, dim3(grid), dim3(MERGE_ROW_WARPS * 32), 0, stream, p);
            else e = launch_maybe_pdl(pdl, merge_rows_kernel<__half, 64>, dim3(grid), dim3(MERGE_ROW_WARPS * 32), 0, stream, p);
        } else {
            if (head_dim == 128) e = launch_maybe_pdl(pdl, merge_rows_kernel<__nv_bfloat16, 128>, dim3(grid), dim3(MERGE_ROW_WARPS * 32), 0, stream, p);
            else e = launch_maybe_pdl(pdl, merge_rows_kernel<__nv_bfloat16, 64>, dim3(grid), dim3(MERGE_ROW_WARPS * 32), 0, stream, p);
        }
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t units = (int64_t)p.num_seqs * p.q_len * p.Hkv * p.merge_splits;
    const size_t smem = merge_smem_bytes(p.G, p.max_parts, head_dim, p.merge_splits);
    const int pps = (p.G * (head_dim / 4) + p.merge_splits - 1) / p.merge_splits;
    const int threads = merge_threads(pps, p.max_parts);
#define PA_MERGE(TT, DD)                                                                                       \
    e = cudaFuncSetAttribute(merge_kernel<TT, DD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
    if (e != cudaSuccess) return e;                                                                            \
    e = launch_maybe_pdl(pdl, merge_kernel<TT, DD>, dim3((unsigned)units), dim3(threads), smem, stream, p);             \
    if (e != cudaSuccess) return e;
    if (dtype == PA_FP16) {
        if (head_dim == 128) { PA_MERGE(__half, 128) } else { PA_MERGE(__half, 64) }
    } else {
        if (head_dim == 128) { PA_MERGE(__nv_bfloat16, 128) } else { PA_MERGE(__nv_bfloat16, 64) }
    }
#undef PA_MERGE
    return cudaGetLastError();
}

}  // namespace pa
