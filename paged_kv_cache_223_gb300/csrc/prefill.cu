// prefill.cu -- paged attention for a chunk of many new tokens per sequence (chunked prefill),
// on the 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// A long prompt is cut into chunks that are processed one at a time, each chunk's K/V written to
// the pool first (yangyu.win blog #54, section 4 "Chunked Prefill": split an 8,000-token prompt
// into 512-token chunks). Each chunk query row qi sits at position L - C + qi of its sequence and
// attends causally to tokens 0..L - C + qi through the block table, exactly as pa_decode with
// q_len = C (learn.tanhdev.com part 8: A_i = softmax(q_i K^T / sqrt(d_k)), o_i = sum a v).
//
// One CTA handles 128 query rows of one (sequence, KV head): the G query heads of the group times
// 128 / G chunk positions, one row per thread and per tensor-memory lane. For every 64-token K/V
// tile (two-stage TMA pipeline, 128-byte swizzle):
//   S = Q K^T    tcgen05.mma M=128, N=64, K=128 from shared memory (both operands K-major) -> TMEM
//   softmax      each thread loads its row of S from TMEM, masks (causal), keeps a running max
//                (the O rescale is skipped while the max grows by less than 2^8) and the row sum
//   P            written to shared memory in the operand layout (bf16: hi and lo parts)
//   O += P V     tcgen05.mma M=128, N=128, K=64, V as an MN-major operand -> TMEM
// Thread 0 issues the copies and the MMAs; completion is tracked by tcgen05.commit on mbarriers.
#include "pa_device.cuh"

namespace pa {

constexpr int PF_BM = 128;            // query rows per CTA
constexpr int PF_BN = 64;             // keys per K/V tile
constexpr int PF_D = 128;             // head dimension
constexpr int PF_THREADS = 128;
constexpr int PF_Q_BYTES = PF_BM * PF_D * 2;                  // 32 KB: 2 halves of [128 rows x 128 B]
constexpr int PF_KV_BYTES = PF_BN * PF_D * 2;                 // 16 KB: 2 halves of [64 rows x 128 B]
constexpr int PF_STAGE_BYTES = 2 * PF_KV_BYTES;               // K tile + V tile
constexpr int PF_P_BYTES = PF_BM * PF_BN * 2;                 // 16 KB: [128 rows x 128 B]
constexpr int PF_OFF_STAGE = PF_Q_BYTES;
constexpr int PF_OFF_P = PF_OFF_STAGE + 2 * PF_STAGE_BYTES;   // P hi, then P lo
constexpr int PF_OFF_BAR = PF_OFF_P + 2 * PF_P_BYTES;
constexpr int PF_SMEM = 1024 + PF_OFF_BAR + 64;
constexpr uint32_t PF_TMEM_COLS = 256;                        // S: columns 0..63, O: 64..191
constexpr float PF_RESCALE_LOG2 = 8.f;                        // stale-max headroom (P <= 2^8)

size_t prefill_smem_bytes() { return PF_SMEM; }

template <typename T>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const DecodeParams p) {
    constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_u32);
    const uint32_t bar_full = base + PF_OFF_BAR;               // [2]
    const uint32_t bar_s = bar_full + 16, bar_o = bar_full + 24;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PF_OFF_BAR + 32);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int mtiles = (p.rows + PF_BM - 1) / PF_BM;
    const int mt = blockIdx.x % mtiles;
    const int bg = blockIdx.x / mtiles;
    const int g = bg % p.Hkv, b = bg / p.Hkv;

    int L = __ldg(p.context_lens + b);
    if (L < p.q_len || L > p.max_ctx) {
        if (tid == 0 && mt == 0) set_status(p.status, STATUS_BOUNDS);
        L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
    }
    const int r = mt * PF_BM + tid;                            // this thread's query row in the unit
    const bool row_ok = r < p.rows;
    const int qi = row_ok ? r / p.G : p.q_len - 1;
    const int hh = row_ok ? r - (r / p.G) * p.G : 0;
    const int lim = L - p.q_len + qi;                          // last key this row may see
    int last_q = (mt * PF_BM + PF_BM - 1) / p.G;
    if (last_q > p.q_len - 1) last_q = p.q_len - 1;
    const int kv_end = L - p.q_len + last_q + 1;               // keys any row of the CTA sees
    const int ntiles = kv_end > 0 ? (kv_end + PF_BN - 1) / PF_BN : 0;

    // ---- prologue: tensor memory, barriers, Q tile
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), PF_TMEM_COLS);
    if (tid == 0) {
        mbar_init(bar_full, 1);
        mbar_init(bar_full + 8, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_barrier_init();
    }
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const T *>(p.q) + (((int64_t)b * p.q_len + qi) * p.Hq + g * p.G + hh) * PF_D);
#pragma unroll
        for (int c = 0; c < 16; ++c) {                         // 16 chunks of 8 values
            const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            const int half = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4 *>(smem + half * (PF_BM * 128) + tid * 128 + ((cc ^ (tid & 7)) << 4)) = v;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_s = tmem, tmem_o = tmem + PF_BN;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint64_t policy = l2_policy_evict_last();    // re-read by the other row tiles of the unit

    // K/V tile j -> stage j & 1: 16-token sub-tiles that start inside the context
    auto issue = [&](int j) {
        const int st = j & 1;
        const uint32_t kdst = base + PF_OFF_STAGE + st * PF_STAGE_BYTES, vdst = kdst + PF_KV_BYTES;
        const uint32_t bar = bar_full + st * 8;
        int nsub = 0;
        for (int sb = 0; sb < PF_BN / TILE_TOKENS; ++sb)
            if (j * PF_BN + sb * TILE_TOKENS < L) ++nsub;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, nsub * 4 * TILE_TOKENS * 128);
        for (int sb = 0; sb < nsub; ++sb) {
            const int tok = j * PF_BN + sb * TILE_TOKENS;
            int id = __ldg(p.block_tables + (int64_t)b * p.stride + tok / p.bs);
            if (id < 0 || id >= p.num_blocks) {
                set_status(p.status, STATUS_BOUNDS);
                id = 0;
            }
            const int row0 = (id * p.Hkv + g) * p.bs + tok % p.bs;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t off = h * (PF_BN * 128) + sb * TILE_TOKENS * 128;
                tma_load_2d(kdst + off, &tmk, h * 64, row0, bar, policy);
                tma_load_2d(vdst + off, &tmv, h * 64, row0, bar, policy);
            }
        }
    };
    int issued = 0, full_seen = 0, s_commits = 0, s_seen = 0, o_commits = 0, o_seen = 0;  // thread 0
    if (tid == 0)
        for (; issued < 2 && issued < ntiles; ++issued) issue(issued);

    const uint32_t idesc_s = umma_idesc<T>(PF_BM, PF_BN, false);
    const uint32_t idesc_o = umma_idesc<T>(PF_BM, PF_D, true);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
        const int st = j & 1;
        const uint32_t kst = base + PF_OFF_STAGE + st * PF_STAGE_BYTES, vst = kst + PF_KV_BYTES;
        // a failed wait is acted on at the next block barrier, by every thread alike
        bool bad = !mbar_wait_bounded(bar_full + st * 8, (uint32_t)(j >> 1) & 1u, p.wait_ns);
        // S = Q K^T (shared-memory reads only, issued even after a failed wait)
        if (tid == 0) {
            if (!bad) full_seen = j + 1;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < PF_D / 16; ++ks) {
                const uint32_t qa = base + (ks >> 2) * (PF_BM * 128) + (ks & 3) * 32;
                const uint32_t ka = kst + (ks >> 2) * (PF_BN * 128) + (ks & 3) * 32;
                umma_f16(tmem_s, umma_desc_sw128(qa, 16, 1024), umma_desc_sw128(ka, 16, 1024), idesc_s, ks > 0);
            }
            umma_commit(bar_s);
            ++s_commits;
        }
        if (mbar_wait_bounded(bar_s, (uint32_t)j & 1u, p.wait_ns)) {
            if (tid == 0) s_seen = j + 1;
        } else {
            bad = true;
        }
        tc_fence_after();
        float sv[PF_BN];
        {
            float a[32];
            tmem_ld32(tmem_s + lane_base, a);
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[c] = a[c];
            tmem_ld32(tmem_s + lane_base + 32, a);
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[32 + c] = a[c];
        }
        // mask, running max (kept stale while it grows by less than 2^8), weights, row sum
        const int t0 = j * PF_BN;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < PF_BN; ++c) {
            sv[c] = t0 + c <= lim ? sv[c] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sv[c]);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_ref + PF_RESCALE_LOG2 || (m_ref == -INFINITY && mx > -INFINITY)) {
            alpha = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mx);
            m_ref = mx;
            rescale = true;
        }
        const float muse = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < PF_BN; ++c) {
            sv[c] = exp2f(sv[c] - muse);
            rs += sv[c];
        }
        l = l * alpha + rs;
        // rescale this warp's O rows when a row's reference max moved (the previous P.V completed
        // before the last block barrier)
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c0 = 0; c0 < PF_D; c0 += 32) {
                float a[32];
                tmem_ld32(tmem_o + lane_base + c0, a);
#pragma unroll
                for (int c = 0; c < 32; ++c) a[c] *= alpha;
                tmem_st32(tmem_o + lane_base + c0, a);
            }
        }
        // P -> shared memory, K-major operand layout: row = this thread, 64 keys = one 128-byte row
        {
            uint8_t *ph = smem + PF_OFF_P + tid * 128;
            uint8_t *pl = ph + PF_P_BYTES;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4], wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = sv[c * 8 + 2 * e], x1 = sv[c * 8 + 2 * e + 1];
                    if constexpr (SPLIT_P) {
                        const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
                        const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
                        w[e] = pack2<T>(h0, h1);
                        wl[e] = pack2<T>(x0 - h0, x1 - h1);
                    } else {
                        w[e] = pack2<T>(x0, x1);
                    }
                }
                const int pos = (c ^ (tid & 7)) << 4;
                *reinterpret_cast<uint4 *>(ph + pos) = make_uint4(w[0], w[1], w[2], w[3]);
                if constexpr (SPLIT_P) *reinterpret_cast<uint4 *>(pl + pos) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }
        // V rows past the context (last tile) hold other tokens' data or stale words: zero them
        if (t0 + PF_BN > L) {
            const int nvalid = L - t0 > 0 ? L - t0 : 0;
            const int nz = (PF_BN - nvalid) * 8;               // 16-byte chunks per half
            uint8_t *vg = smem + (vst - base);
            for (int c = tid; c < 2 * nz; c += PF_THREADS) {
                const int h = c / nz, rc = c - h * nz;
                *reinterpret_cast<uint4 *>(vg + h * (PF_BN * 128) + (nvalid + rc / 8) * 128 + (rc % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) {
            ok = false;
            break;
        }
        // O += P V
        bool got_o = true;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < (SPLIT_P ? 2 : 1); ++part) {
#pragma unroll
                for (int ks = 0; ks < PF_BN / 16; ++ks) {
                    const uint32_t pa = base + PF_OFF_P + part * PF_P_BYTES + ks * 32;
                    const uint32_t va = vst + ks * 16 * 128;
                    umma_f16(tmem_o, umma_desc_sw128(pa, 16, 1024), umma_desc_sw128(va, PF_BN * 128, 1024), idesc_o,
                             (j > 0 || ks > 0 || part > 0) ? 1u : 0u);
                }
            }
            umma_commit(bar_o);
            ++o_commits;
            // the stage and P are free once this P.V is done: refill the stage with tile j + 2
            got_o = mbar_wait_bounded(bar_o, (uint32_t)j & 1u, p.wait_ns);
            if (got_o) {
                o_seen = j + 1;
                if (issued < ntiles) issue(issued++);
            }
        }
        if (__syncthreads_or(!got_o)) {
            ok = false;
            break;
        }
    }

    if (!ok) {
        // record the timeout and wait (bounded) for every copy and MMA still in flight, so that
        // none lands in shared or tensor memory after the CTA has released it
        if (tid == 0) {
            set_status(p.status, STATUS_TIMEOUT);
            for (int t = full_seen; t < issued; ++t)
                mbar_wait_bounded(bar_full + (t & 1) * 8, (uint32_t)(t >> 1) & 1u, p.wait_ns);
            for (int t = s_seen; t < s_commits; ++t) mbar_wait_bounded(bar_s, (uint32_t)t & 1u, p.wait_ns);
            for (int t = o_seen; t < o_commits; ++t) mbar_wait_bounded(bar_o, (uint32_t)t & 1u, p.wait_ns);
        }
    } else if (ntiles > 0) {
        // epilogue: the last P.V has completed (thread 0 waited on it before the final barrier)
        tc_fence_after();
        const float inv = 1.f / l;
        T *dst = reinterpret_cast<T *>(p.out) + (((int64_t)b * p.q_len + qi) * p.Hq + g * p.G + hh) * PF_D;
#pragma unroll
        for (int c0 = 0; c0 < PF_D; c0 += 32) {
            float a[32];
            tmem_ld32(tmem_o + lane_base + c0, a);
            if (row_ok) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    const uint4 v = make_uint4(pack2<T>(a[c] * inv, a[c + 1] * inv), pack2<T>(a[c + 2] * inv, a[c + 3] * inv),
                                               pack2<T>(a[c + 4] * inv, a[c + 5] * inv), pack2<T>(a[c + 6] * inv, a[c + 7] * inv));
                    *reinterpret_cast<uint4 *>(dst + c0 + c) = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, PF_TMEM_COLS);
}

cudaError_t launch_prefill(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           cudaStream_t stream) {
    const int64_t grid = (int64_t)p.num_seqs * p.Hkv * ((p.rows + PF_BM - 1) / PF_BM);
    cudaError_t e;
    if (dtype == PA_FP16) {
        e = cudaFuncSetAttribute(prefill_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
        if (e != cudaSuccess) return e;
        prefill_kernel<__half><<<(unsigned)grid, PF_THREADS, PF_SMEM, stream>>>(tmk, tmv, p);
    } else {
        e = cudaFuncSetAttribute(prefill_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
        if (e != cudaSuccess) return e;
        prefill_kernel<__nv_bfloat16><<<(unsigned)grid, PF_THREADS, PF_SMEM, stream>>>(tmk, tmv, p);
    }
    return cudaGetLastError();
}

}  // namespace pa
