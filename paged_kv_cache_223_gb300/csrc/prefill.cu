// prefill.cu -- paged attention for a chunk of many new tokens per sequence (chunked prefill),
// on the 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// A long prompt is cut into chunks that are processed one at a time, each chunk's K/V written to
// the pool first (yangyu.win blog #54, section 4 "Chunked Prefill": split an 8,000-token prompt
// into 512-token chunks). Each chunk query row qi sits at position L - C + qi of its sequence and
// attends causally to tokens 0..L - C + qi through the block table, exactly as pa_decode with
// q_len = C (learn.tanhdev.com part 8: A_i = softmax(q_i K^T / sqrt(d_k)), o_i = sum a v).
//
// A query "row" is one (chunk position, query head of the KV group) pair: r = qi * G + h. One CTA
// takes two tiles of 128 rows of one (sequence, KV head) and walks the keys in 64-token tiles:
//   warp 8 (producer)  block-table lookups and TMA copies of K/V tiles into a ring of stages
//   warp 9 (MMA)       S_t = Q_t K^T  (tcgen05.mma M=128 N=64 K=128 from shared memory) -> TMEM
//                      O_t += P_t V   (M=128 N=128 K=64: P read from TMEM, V an MN-major smem operand)
//                      one elected thread issues; completion is signalled by tcgen05.commit
//   warps 0-3, 4-7     softmax of row tile 0 and 1, one row per thread = one tensor-memory lane:
//                      S from TMEM, causal mask, running max (the O rescale is skipped while the
//                      max grows by less than 2^8), row sum, P (bf16: hi + lo parts) written back to
//                      TMEM over the S it came from
// Tensor memory per row tile: two S buffers of 64 columns (S of key tile j in buffer j & 1) and O
// (128 columns). S of key tile j is issued before P.V of tile j-1, so the softmax of tile j runs
// while the tensor cores finish tile j-1; MMAs of one thread execute in issue order, so S(j+2)
// overwrites P(j) only after P(j).V has read it.
#include "pa_device.cuh"

namespace pa {

constexpr int PF_BM = 128;            // query rows per row tile
constexpr int PF_BN = 64;             // keys per K/V tile
constexpr int PF_D = 128;             // head dimension
constexpr int PF_QT = 2;              // row tiles per CTA
constexpr int PF_SM_THREADS = PF_QT * PF_BM;
constexpr int PF_PRODUCER_WARP = PF_SM_THREADS / 32;
constexpr int PF_MMA_WARP = PF_PRODUCER_WARP + 1;
constexpr int PF_THREADS = PF_SM_THREADS + 64;
constexpr int PF_Q_BYTES = PF_BM * PF_D * 2;                  // 32 KB: 2 halves of [128 rows x 128 B]
constexpr int PF_KV_BYTES = PF_BN * PF_D * 2;                 // 16 KB: 2 halves of [64 rows x 128 B]
constexpr int PF_STAGE_BYTES = 2 * PF_KV_BYTES;               // K tile + V tile
constexpr uint32_t PF_TMEM_COLS = 512;                        // row tile t: S at 256 t (+64), O at 256 t + 128
constexpr float PF_RESCALE_LOG2 = 8.f;                        // stale-max headroom (P <= 2^8)

template <typename T>
struct PrefillLayout {
    static constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int STAGES = 4;
    static constexpr int OFF_STAGE = PF_QT * PF_Q_BYTES;
    static constexpr int OFF_BAR = OFF_STAGE + STAGES * PF_STAGE_BYTES;
    // barriers: kv_full[STAGES], kv_empty[STAGES], then per row tile s_full[2], p_full[2], o_bar[2],
    // then o_done[2], drain
    static constexpr int NBAR = 2 * STAGES + 6 * PF_QT + PF_QT + 1;
    static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
};
static_assert(PrefillLayout<__half>::SMEM <= 227 * 1024, "prefill shared memory");
static_assert(PrefillLayout<__nv_bfloat16>::SMEM <= 227 * 1024, "prefill shared memory");

size_t prefill_smem_bytes() { return PrefillLayout<__nv_bfloat16>::SMEM; }

template <typename T>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const DecodeParams p) {
    using LY = PrefillLayout<T>;
    constexpr bool SPLIT_P = LY::SPLIT_P;
    constexpr int STAGES = LY::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_u32);
    const uint32_t bar_kv_full = base + LY::OFF_BAR;
    const uint32_t bar_kv_empty = bar_kv_full + STAGES * 8;
    const uint32_t bar_s_full = bar_kv_empty + STAGES * 8;        // [t][buffer]
    const uint32_t bar_p_full = bar_s_full + PF_QT * 16;          // [t][buffer]
    const uint32_t bar_o_bar = bar_p_full + PF_QT * 16;           // [t][buffer]: P.V of that buffer done
    const uint32_t bar_o_done = bar_o_bar + PF_QT * 16;
    const uint32_t bar_drain = bar_o_done + PF_QT * 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + LY::OFF_BAR + LY::NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *issued_tiles = reinterpret_cast<volatile int *>(tmem_slot + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mtiles = (p.rows + PF_BM - 1) / PF_BM;
    const int ctiles = (mtiles + PF_QT - 1) / PF_QT;
    const int ct = ctiles - 1 - (int)(blockIdx.x % ctiles);  // the unit's longest row tiles start first
    const int bg = blockIdx.x / ctiles;
    const int g = bg % p.Hkv, b = bg / p.Hkv;

    int L = __ldg(p.context_lens + b);
    if (L < p.q_len || L > p.max_ctx) {
        if (tid == 0 && ct == 0) set_status(p.status, STATUS_BOUNDS);
        L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
    }
    // key tiles each row tile needs: up to the last key its last row sees
    int nt_of[PF_QT];
#pragma unroll
    for (int t = 0; t < PF_QT; ++t) {
        const int mt = ct * PF_QT + t;
        int last_q = (mt * PF_BM + PF_BM - 1) / p.G;
        if (last_q > p.q_len - 1) last_q = p.q_len - 1;
        const int kv_end = L - p.q_len + last_q + 1;
        nt_of[t] = (mt < mtiles && kv_end > 0) ? (kv_end + PF_BN - 1) / PF_BN : 0;
    }
    const int ntiles = nt_of[0] > nt_of[1] ? nt_of[0] : nt_of[1];

    // ---- prologue: tensor memory, barriers, Q tiles
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), PF_TMEM_COLS);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_kv_full + s * 8, 1);
            mbar_init(bar_kv_empty + s * 8, 1);
        }
        for (int i = 0; i < 2 * PF_QT; ++i) {
            mbar_init(bar_s_full + i * 8, 1);
            mbar_init(bar_p_full + i * 8, PF_BM);
            mbar_init(bar_o_bar + i * 8, 1);
        }
        for (int t = 0; t < PF_QT; ++t) mbar_init(bar_o_done + t * 8, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        *issued_tiles = 0;
        fence_barrier_init();
    }
    // softmax threads: row tile t = tid / 128, row rt = tid % 128
    const int t_of = tid >> 7, rt = tid & (PF_BM - 1);
    const int r = (ct * PF_QT + t_of) * PF_BM + rt;
    const bool row_ok = tid < PF_SM_THREADS && r < p.rows;
    const int qi = row_ok ? r / p.G : p.q_len - 1;
    const int hh = row_ok ? r - (r / p.G) * p.G : 0;
    if (tid < PF_SM_THREADS) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const T *>(p.q) + (((int64_t)b * p.q_len + qi) * p.Hq + g * p.G + hh) * PF_D);
        uint8_t *qdst = smem + t_of * PF_Q_BYTES + rt * 128;
#pragma unroll
        for (int c = 0; c < 16; ++c) {                         // 16 chunks of 8 values, 128-byte swizzle
            const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(qdst + (c >> 3) * (PF_BM * 128) + (((c & 7) ^ (rt & 7)) << 4)) = v;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int consumed = 0;                                          // MMA warp: key tiles whose copies landed

    if (warp == PF_PRODUCER_WARP) {
        // ---------------------------------------------------------------- producer
        // A tile is 16 copies of 16 rows x 128 bytes (4 sub-tiles x 2 halves x K/V), one per lane:
        // a single thread issuing them all could not keep the tensor cores fed. Each lane looks up
        // its sub-tile's block one tile ahead.
        const uint64_t policy = l2_policy_evict_last();       // re-read by the unit's other row tiles
        const int sb = lane >> 2, h = (lane >> 1) & 1, is_v = lane & 1;
        const bool copier = lane < 4 * (PF_BN / TILE_TOKENS);
        auto lookup = [&](int j) -> int {
            const int tok = j * PF_BN + sb * TILE_TOKENS;
            return (copier && tok < L) ? __ldg(p.block_tables + (int64_t)b * p.stride + tok / p.bs) : 0;
        };
        int id_next = ntiles > 0 ? lookup(0) : 0;
        int j = 0;
        for (; j < ntiles; ++j) {
            const int st = j % STAGES;
            if (j >= STAGES) {
                const bool got =
                    mbar_wait_bounded(bar_kv_empty + st * 8, (uint32_t)((j - STAGES) / STAGES) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            int id = id_next;
            if (j + 1 < ntiles) id_next = lookup(j + 1);
            const int rem = L - j * PF_BN;                     // > 0 for every tile issued
            const int nsub = rem >= PF_BN ? PF_BN / TILE_TOKENS : (rem + TILE_TOKENS - 1) / TILE_TOKENS;
            const uint32_t bar = bar_kv_full + st * 8;
            if (lane == 0) mbar_arrive_expect_tx(bar, nsub * 4 * TILE_TOKENS * 128);
            __syncwarp();
            if (copier && sb < nsub) {
                if (id < 0 || id >= p.num_blocks) {
                    set_status(p.status, STATUS_BOUNDS);
                    id = 0;
                }
                const int tok = j * PF_BN + sb * TILE_TOKENS;
                const int row0 = (id * p.Hkv + g) * p.bs + tok % p.bs;
                const uint32_t dst = base + LY::OFF_STAGE + st * PF_STAGE_BYTES + is_v * PF_KV_BYTES +
                                     h * (PF_BN * 128) + sb * TILE_TOKENS * 128;
                tma_load_2d(dst, is_v ? &tmv : &tmk, h * 64, row0, bar, policy);
            }
        }
        if (lane == 0) *issued_tiles = j;
    } else if (warp == PF_MMA_WARP) {
        // ---------------------------------------------------------------- MMA issue
        const uint32_t idesc_s = umma_idesc<T>(PF_BM, PF_BN, false);
        const uint32_t idesc_o = umma_idesc<T>(PF_BM, PF_D, true);
        // Shared-memory descriptors are built once; per MMA only a constant (address >> 4) is added
        // (every operand lies below 256 KB, so the 14-bit address field never carries).
        const uint64_t dq0 = umma_desc_sw128(base, 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(base + LY::OFF_STAGE, 16, 1024);
        const uint64_t dv0 = umma_desc_sw128(base + LY::OFF_STAGE + PF_KV_BYTES, PF_BN * 128, 1024);
        auto issue_pv = [&](int t, int j) {                   // O_t += P_t(j) V(j), P in TMEM buffer j & 1
            const uint64_t dv = dv0 + (uint64_t)((j % STAGES) * (PF_STAGE_BYTES >> 4));
            const uint32_t pt = tmem + t * 256 + (j & 1) * PF_BN, ot = tmem + t * 256 + 128;
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int part = 0; part < (SPLIT_P ? 2 : 1); ++part) {
#pragma unroll
                for (int ks = 0; ks < PF_BN / 16; ++ks)
                    umma_f16_tmem_a(ot, pt + part * 32 + ks * 8, dv + (uint64_t)((ks * 16 * 128) >> 4), idesc_o,
                                    (ks > 0 || part > 0) ? 1u : acc0);
            }
            umma_commit(bar_o_bar + (t * 2 + (j & 1)) * 8);
        };
        auto wait_p = [&](int t, int j) -> bool {            // softmax of row tile t wrote P(j)
            const bool got =
                mbar_wait_bounded(bar_p_full + (t * 2 + (j & 1)) * 8, (uint32_t)(j >> 1) & 1u, p.wait_ns);
            return __all_sync(0xffffffffu, got);
        };
        bool ok = true;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int st = j % STAGES;
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(bar_kv_full + st * 8, (uint32_t)(j / STAGES) & 1u, p.wait_ns));
            if (!ok) break;
            consumed = j + 1;
            const int t0 = j * PF_BN;
            if (t0 + PF_BN > L) {
                // V rows past the context hold other tokens' data or stale words: zero them
                const int nvalid = L - t0 > 0 ? L - t0 : 0;
                const int nz = (PF_BN - nvalid) * 8;           // 16-byte chunks per half
                uint8_t *vg = smem + LY::OFF_STAGE + st * PF_STAGE_BYTES + PF_KV_BYTES;
                for (int c = lane; c < 2 * nz; c += 32) {
                    const int h = c / nz, rc = c - h * nz;
                    *reinterpret_cast<uint4 *>(vg + h * (PF_BN * 128) + (nvalid + rc / 8) * 128 + (rc % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // S(t, j) into buffer j & 1 (its last reader, P(j-2).V, was issued one tile earlier)
            if (lane == 0) {
                const uint64_t dk = dk0 + (uint64_t)(st * (PF_STAGE_BYTES >> 4));
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < PF_QT; ++t) {
                    if (j < nt_of[t]) {
                        const uint64_t dq = dq0 + (uint64_t)(t * (PF_Q_BYTES >> 4));
                        const uint32_t sd = tmem + t * 256 + (j & 1) * PF_BN;
#pragma unroll
                        for (int ks = 0; ks < PF_D / 16; ++ks)
                            umma_f16(sd, dq + (uint64_t)(((ks >> 2) * (PF_BM * 128) + (ks & 3) * 32) >> 4),
                                     dk + (uint64_t)(((ks >> 2) * (PF_BN * 128) + (ks & 3) * 32) >> 4), idesc_s,
                                     ks > 0 ? 1u : 0u);
                        umma_commit(bar_s_full + (t * 2 + (j & 1)) * 8);
                    }
                }
            }
            // P(t, j-1) V(j-1) once the softmax of row tile t has written P(j-1)
            if (j > 0) {
#pragma unroll
                for (int t = 0; t < PF_QT; ++t) {
                    if (j - 1 < nt_of[t]) {
                        if (!(ok = wait_p(t, j - 1))) break;
                        if (lane == 0) {
                            tc_fence_after();
                            issue_pv(t, j - 1);
                        }
                    }
                }
                if (!ok) break;
                if (lane == 0) umma_commit(bar_kv_empty + ((j - 1) % STAGES) * 8);
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) ok = false;
        }
        if (ok && ntiles > 0) {
#pragma unroll
            for (int t = 0; t < PF_QT; ++t) {
                if (ntiles - 1 < nt_of[t]) {
                    if (!(ok = wait_p(t, ntiles - 1))) break;
                    if (lane == 0) {
                        tc_fence_after();
                        issue_pv(t, ntiles - 1);
                    }
                }
            }
            if (ok && lane == 0)
                for (int t = 0; t < PF_QT; ++t) umma_commit(bar_o_done + t * 8);
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else {
        // ---------------------------------------------------------------- softmax (row tile t_of)
        const int t = t_of;
        const int nt = t ? nt_of[1] : nt_of[0];
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tmem_t = tmem + t * 256 + lane_base, tmem_o = tmem_t + 128;
        const int lim = L - p.q_len + qi;                      // last key this row may see
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int buf = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_s_full + (t * 2 + buf) * 8, (uint32_t)(j >> 1) & 1u,
                                                           p.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float sv[PF_BN];
            tmem_ld64(tmem_t + buf * PF_BN, sv);
            // raw-score max (the scale is positive, so it commutes with the max); eight independent
            // partial maxima and sums keep the dependent chains short
            const int t0 = j * PF_BN;
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
            if (t0 + PF_BN - 1 <= lim) {
#pragma unroll
                for (int c = 0; c < PF_BN; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
            } else {
#pragma unroll
                for (int c = 0; c < PF_BN; ++c) {
                    sv[c] = t0 + c <= lim ? sv[c] : -INFINITY;
                    m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * p.scale_log2;
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_ref + PF_RESCALE_LOG2 || (m_ref == -INFINITY && mx > -INFINITY)) {
                alpha = m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mx);
                m_ref = mx;
                rescale = true;
            }
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // O holds the sums through key tile j-1: wait for P(j-1).V, then scale this warp's rows
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_o_bar + (t * 2 + (buf ^ 1)) * 8,
                                                               (uint32_t)((j - 1) >> 1) & 1u, p.wait_ns));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < PF_D; c0 += 32) {
                    float a[32];
                    tmem_ld32(tmem_o + c0, a);
#pragma unroll
                    for (int c = 0; c < 32; ++c) a[c] *= alpha;
                    tmem_st32(tmem_o + c0, a);
                }
            }
            const float nmuse = m_ref == -INFINITY ? 0.f : -m_ref;
            float r8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) r8[i] = 0.f;
#pragma unroll
            for (int c = 0; c < PF_BN; ++c) {
                sv[c] = ex2_approx(fmaf(sv[c], p.scale_log2, nmuse));
                r8[c & 7] += sv[c];
            }
            l = l * alpha + ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
            // P over this buffer's S: 64 keys as 32 packed columns (bf16: hi, then lo = x - hi)
            {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) w[c] = pack2<T>(sv[2 * c], sv[2 * c + 1]);
                tmem_st32_raw(tmem_t + buf * PF_BN, w);
                if constexpr (SPLIT_P) {
                    uint32_t wl[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        // a bf16 is the top half of an fp32
                        const float h0 = __uint_as_float(w[c] << 16), h1 = __uint_as_float(w[c] & 0xFFFF0000u);
                        wl[c] = pack2<T>(sv[2 * c] - h0, sv[2 * c + 1] - h1);
                    }
                    tmem_st32_raw(tmem_t + buf * PF_BN + 32, wl);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar_p_full + (t * 2 + buf) * 8);
            if (__any_sync(0xffffffffu, *abort_flag != 0)) {
                ok = false;
                break;
            }
        }
        if (ok && nt > 0)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_o_done + t * 8, 0u, p.wait_ns));
        if (!ok) {
            if (lane == 0) *abort_flag = 1;
        } else if (nt > 0) {
            tc_fence_after();
            const float inv = 1.f / l;
            T *dst = reinterpret_cast<T *>(p.out) + (((int64_t)b * p.q_len + qi) * p.Hq + g * p.G + hh) * PF_D;
#pragma unroll
            for (int c0 = 0; c0 < PF_D; c0 += 32) {
                float a[32];
                tmem_ld32(tmem_o + c0, a);
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        const uint4 v =
                            make_uint4(pack2<T>(a[c] * inv, a[c + 1] * inv), pack2<T>(a[c + 2] * inv, a[c + 3] * inv),
                                       pack2<T>(a[c + 4] * inv, a[c + 5] * inv), pack2<T>(a[c + 6] * inv, a[c + 7] * inv));
                        *reinterpret_cast<uint4 *>(dst + c0 + c) = v;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait ran out: record it, then wait (bounded) for every copy and MMA still in flight so
        // that none lands in shared or tensor memory after the CTA has released them
        if (tid == 0) set_status(p.status, STATUS_TIMEOUT);
        if (warp == PF_MMA_WARP && lane == 0) {
            for (int j = consumed; j < *issued_tiles; ++j)
                mbar_wait_bounded(bar_kv_full + (j % STAGES) * 8, (uint32_t)(j / STAGES) & 1u, p.wait_ns);
            umma_commit(bar_drain);
            mbar_wait_bounded(bar_drain, 0u, p.wait_ns);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, PF_TMEM_COLS);
    }
}

template <typename T>
static cudaError_t launch_prefill_t(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                    cudaStream_t stream) {
    const int mtiles = (p.rows + PF_BM - 1) / PF_BM;
    const int64_t grid = (int64_t)p.num_seqs * p.Hkv * ((mtiles + PF_QT - 1) / PF_QT);
    constexpr int smem = PrefillLayout<T>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<T><<<(unsigned)grid, PF_THREADS, smem, stream>>>(tmk, tmv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           cudaStream_t stream) {
    return dtype == PA_FP16 ? launch_prefill_t<__half>(p, tmk, tmv, stream)
                            : launch_prefill_t<__nv_bfloat16>(p, tmk, tmv, stream);
}

}  // namespace pa
