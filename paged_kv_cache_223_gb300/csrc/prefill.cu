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
// takes two tiles of 128 rows of one (sequence, KV head) and walks the keys in 128-token tiles,
// the two row tiles in ping-pong so that one tile's softmax overlaps the other's products:
//   warps 8, 10        K and V producers: each lane looks up one 16-token sub-tile's block (one
//                      tile ahead) and issues one TMA copy (8 sub-tiles x 2 halves per tile) into
//                      a ring of K stages (freed once S is computed) or V stages (freed after P.V)
//   warp 9 (MMA)       one thread issues, per row tile t and key tile j:
//                        O_t += P_t(j-1) V(j-1)   M=128 N=128 K=128, P read from TMEM, V MN-major
//                        S_t  = Q_t K(j)^T        M=128 N=128 K=128, both operands in shared memory
//                      and signals completion with tcgen05.commit
//   warps 0-3, 4-7     softmax of row tile 0 and 1, one row per thread = one tensor-memory lane:
//                      S from TMEM, causal mask, running max (the O rescale is skipped while the
//                      max grows by less than 2^8), row sum, P (bf16: hi + lo parts) written back to
//                      TMEM over the S it came from
// The same kernel (CASCADE) computes a shared prefix once for a whole batch: its rows are every
// sequence's query rows, its keys one partition of the prefix (blocks from sequence 0's table, no
// mask: every query row follows the prefix), and it writes the unnormalised partition state
// (O, running max, sum) that the log-sum-exp merge combines with the decode of each suffix
// (a cascade over the pages' copy-on-write prefix blocks: yangyu.win blog #54 section 5
// question 2, itimpress.au section 1).
// Tensor memory per row tile: S/P (128 columns) and O (128 columns). MMAs of one thread execute in
// issue order, so S(j) overwrites P(j-1) only after P(j-1).V has read it, and the commit of S(j)
// also covers P(j-1).V: the softmax of tile j may rescale O without another wait.
#include "pa_device.cuh"

namespace pa {

constexpr int PF_BM = 128;            // query rows per row tile
constexpr int PF_BN = 128;            // keys per K/V tile
constexpr int PF_D = 128;             // head dimension
constexpr int PF_QT = 2;              // row tiles per CTA
constexpr int PF_SUB = PF_BN / TILE_TOKENS;                   // 16-token sub-tiles per key tile
constexpr int PF_SM_THREADS = PF_QT * PF_BM;
constexpr int PF_PRODUCER_WARP = PF_SM_THREADS / 32;          // K producer
constexpr int PF_MMA_WARP = PF_PRODUCER_WARP + 1;
constexpr int PF_VPRODUCER_WARP = PF_PRODUCER_WARP + 2;
constexpr int PF_THREADS = PF_SM_THREADS + 128;                // + one warpgroup: producers, MMA, 1 idle
// Register split: launched at 168 per thread (65536 / 384, rounded down to 8); the producer/MMA
// warpgroup gives up registers to the two softmax warpgroups: 2 x 128 x 216 + 128 x 72 = 384 x 168.
constexpr uint32_t PF_REGS_LAUNCH = 168, PF_REGS_SOFTMAX = 216, PF_REGS_OTHER = 72;
static_assert(2 * 128 * PF_REGS_SOFTMAX + 128 * PF_REGS_OTHER <= 384 * PF_REGS_LAUNCH, "register split");
constexpr int PF_Q_BYTES = PF_BM * PF_D * 2;                  // 32 KB: 2 halves of [128 rows x 128 B]
constexpr int PF_HALF_BYTES = PF_BN * 128;                    // 16 KB: [128 key rows x 128 B]
constexpr int PF_KV_BYTES = 2 * PF_HALF_BYTES;                // 32 KB: a K or V tile
constexpr int PF_KSTAGES = 3, PF_VSTAGES = 2;
constexpr int PF_OFF_K = PF_QT * PF_Q_BYTES;
constexpr int PF_OFF_V = PF_OFF_K + PF_KSTAGES * PF_KV_BYTES;
constexpr int PF_OFF_BAR = PF_OFF_V + PF_VSTAGES * PF_KV_BYTES;
// barriers: k_full[K], k_empty[K], v_full[V], v_empty[V], s_full[QT], p_full[QT], o_done[QT], drain
constexpr int PF_NBAR = 2 * PF_KSTAGES + 2 * PF_VSTAGES + 3 * PF_QT + 1;
constexpr int PF_SMEM = 1024 + PF_OFF_BAR + PF_NBAR * 8 + 16;
constexpr uint32_t PF_TMEM_COLS = 512;                        // row tile t: S/P at 256 t, O at 256 t + 128
constexpr float PF_RESCALE_LOG2 = 8.f;                        // stale-max headroom (P <= 2^8)
// epilogue staging of a warp's 32 output rows (fp32) in the copy rings; the padded row stride keeps
// both the per-thread row writes and the per-row warp reads free of bank conflicts
constexpr int PF_STAGE_STRIDE = PF_D + 4;
static_assert(8 * 32 * PF_STAGE_STRIDE * 4 <= PF_KSTAGES * PF_KV_BYTES + PF_VSTAGES * PF_KV_BYTES, "epilogue staging");
static_assert(PF_SUB * 2 <= 32, "one copy per producer lane");
static_assert(PF_SMEM <= 227 * 1024, "prefill shared memory");

size_t prefill_smem_bytes() { return PF_SMEM; }

template <typename T, bool CASCADE>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const DecodeParams p) {
    constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_u32);
    const uint32_t bar_k_full = base + PF_OFF_BAR;
    const uint32_t bar_k_empty = bar_k_full + PF_KSTAGES * 8;
    const uint32_t bar_v_full = bar_k_empty + PF_KSTAGES * 8;
    const uint32_t bar_v_empty = bar_v_full + PF_VSTAGES * 8;
    const uint32_t bar_s_full = bar_v_empty + PF_VSTAGES * 8;
    const uint32_t bar_p_full = bar_s_full + PF_QT * 8;
    const uint32_t bar_o_done = bar_p_full + PF_QT * 8;
    const uint32_t bar_drain = bar_o_done + PF_QT * 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PF_OFF_BAR + PF_NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *issued_tiles = reinterpret_cast<volatile int *>(tmem_slot + 2);   // [K, V]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total_rows = CASCADE ? p.num_seqs * p.rows : p.rows;   // query rows of one CTA's unit
    const int mtiles = (total_rows + PF_BM - 1) / PF_BM;
    const int ctiles = (mtiles + PF_QT - 1) / PF_QT;
    const int ct = ctiles - 1 - (int)(blockIdx.x % ctiles);  // the unit's longest row tiles start first
    const int unit = blockIdx.x / ctiles;
    const int g = unit % p.Hkv;
    // b: the sequence whose table names the keys; the keys are tokens [key0, L)
    int b, key0, L;
    if constexpr (CASCADE) {
        // prefix partitions [c * pchunk, min((c + 1) * pchunk, part0)) of chunk c
        b = 0;
        const int c = unit / p.Hkv;
        key0 = c * p.pchunk * p.part_tokens;
        L = min((c + 1) * p.pchunk, p.part0) * p.part_tokens;
    } else {
        b = unit / p.Hkv;
        key0 = 0;
        L = __ldg(p.context_lens + b);
        if (L < p.q_len || L > p.max_ctx) {
            if (tid == 0 && ct == 0) set_status(p.status, STATUS_BOUNDS);
            L = L < 0 ? 0 : (L > p.max_ctx ? p.max_ctx : L);
        }
    }
    // key tiles each row tile needs: up to the last key its last row sees
    int nt0, nt1;
    {
        int nt[PF_QT];
#pragma unroll
        for (int t = 0; t < PF_QT; ++t) {
            const int mt = ct * PF_QT + t;
            if constexpr (CASCADE) {
                nt[t] = mt < mtiles ? (L - key0) / PF_BN : 0;
            } else {
                int last_q = (mt * PF_BM + PF_BM - 1) / p.G;
                if (last_q > p.q_len - 1) last_q = p.q_len - 1;
                const int kv_end = L - p.q_len + last_q + 1;
                nt[t] = (mt < mtiles && kv_end > 0) ? (kv_end + PF_BN - 1) / PF_BN : 0;
            }
        }
        nt0 = nt[0];
        nt1 = nt[1];
    }
    const int ntiles = nt0 > nt1 ? nt0 : nt1;

    // ---- prologue: tensor memory, barriers, Q tiles
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), PF_TMEM_COLS);
    if (tid == 0) {
        for (int s = 0; s < PF_KSTAGES; ++s) {
            mbar_init(bar_k_full + s * 8, 1);
            mbar_init(bar_k_empty + s * 8, 1);
        }
        for (int s = 0; s < PF_VSTAGES; ++s) {
            mbar_init(bar_v_full + s * 8, 1);
            mbar_init(bar_v_empty + s * 8, 1);
        }
        for (int t = 0; t < PF_QT; ++t) {
            mbar_init(bar_s_full + t * 8, 1);
            mbar_init(bar_p_full + t * 8, PF_BM);
            mbar_init(bar_o_done + t * 8, 1);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        issued_tiles[0] = 0;
        issued_tiles[1] = 0;
        fence_barrier_init();
    }
    // barriers and the tensor-memory address are published; the copy warps start at once while the
    // softmax threads load Q (published to the MMA warp by named barrier 1)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int consumed_k = 0, consumed_v = 0;                        // MMA thread: tiles whose copies landed
    // softmax threads: row tile t = tid / 128, row rt = tid % 128
    const int t_of = tid >> 7, rt = tid & (PF_BM - 1);
    const int r = (ct * PF_QT + t_of) * PF_BM + rt;
    const bool row_ok = tid < PF_SM_THREADS && r < total_rows;
    const int rb = CASCADE ? (row_ok ? r / p.rows : 0) : b;   // this row's sequence
    const int rr = row_ok ? r - (CASCADE ? rb * p.rows : 0) : p.rows - 1;
    const int qi = rr / p.G;
    const int hh = rr - qi * p.G;
    const int64_t orow = ((int64_t)rb * p.q_len + qi) * p.Hq + g * p.G + hh;   // q / out row
    constexpr uint32_t Q_BARRIER = 1, Q_BARRIER_THREADS = PF_SM_THREADS + 32;   // softmax + MMA warps

    if (warp >= PF_PRODUCER_WARP) {
      setmaxnreg_dec<PF_REGS_OTHER>();
      if (warp == PF_PRODUCER_WARP || warp == PF_VPRODUCER_WARP) {
        // ---------------------------------------------------------------- K or V producer
        const bool is_v = warp == PF_VPRODUCER_WARP;
        const int nst = is_v ? PF_VSTAGES : PF_KSTAGES;
        const uint32_t full0 = is_v ? bar_v_full : bar_k_full;
        const uint32_t ring = base + (is_v ? PF_OFF_V : PF_OFF_K);
        const CUtensorMap *map = is_v ? &tmv : &tmk;
        const uint64_t policy = l2_policy_evict_last();       // re-read by the unit's other row tiles
        const int sb = lane >> 1, h = lane & 1;
        const bool copier = lane < 2 * PF_SUB;
        auto lookup = [&](int j) -> int {
            const int tok = key0 + j * PF_BN + sb * TILE_TOKENS;
            return (copier && tok < L) ? __ldg(p.block_tables + (int64_t)b * p.stride + tok / p.bs) : 0;
        };
        int id_next = ntiles > 0 ? lookup(0) : 0;
        int j = 0;
        for (; j < ntiles; ++j) {
            const int st = j % nst;
            // K(j) reuses the stage of K(j - 3), freed by the commit after S(j - 3). V(j) reuses the
            // stage of V(j - 2), read by P(j - 2).V, which was issued before S(j - 1): the commit
            // after S(j - 1) covers it
            const int rel = is_v ? j - 1 : j - PF_KSTAGES;     // key tile whose release frees the stage
            if (j >= nst) {
                const bool got = mbar_wait_bounded(bar_k_empty + (rel % PF_KSTAGES) * 8,
                                                   (uint32_t)(rel / PF_KSTAGES) & 1u, p.wait_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            int id = id_next;
            if (j + 1 < ntiles) id_next = lookup(j + 1);
            const int rem = L - key0 - j * PF_BN;              // > 0 for every tile issued
            const int nsub = rem >= PF_BN ? PF_SUB : (rem + TILE_TOKENS - 1) / TILE_TOKENS;
            const uint32_t bar = full0 + st * 8;
            if (lane == 0) mbar_arrive_expect_tx(bar, nsub * 2 * TILE_TOKENS * 128);
            __syncwarp();
            if (copier && sb < nsub) {
                if (id < 0 || id >= p.num_blocks) {
                    set_status(p.status, STATUS_BOUNDS);
                    id = 0;
                }
                const int tok = key0 + j * PF_BN + sb * TILE_TOKENS;
                const int row0 = (id * p.Hkv + g) * p.bs + tok % p.bs;
                tma_load_2d(ring + st * PF_KV_BYTES + h * PF_HALF_BYTES + sb * TILE_TOKENS * 128, map, h * 64, row0,
                            bar, policy);
            }
        }
        if (lane == 0) issued_tiles[is_v ? 1 : 0] = j;
      } else if (warp == PF_MMA_WARP) {
        // ---------------------------------------------------------------- MMA issue (lane 0)
        // Shared-memory descriptors are built once; per MMA only a constant (address >> 4) is added
        // (every operand lies below 256 KB, so the 14-bit address field never carries).
        const uint32_t idesc_s = umma_idesc<T>(PF_BM, PF_BN, false);
        const uint32_t idesc_o = umma_idesc<T>(PF_BM, PF_D, true);
        const uint64_t dq0 = umma_desc_sw128(base, 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(base + PF_OFF_K, 16, 1024);
        const uint64_t dv0 = umma_desc_sw128(base + PF_OFF_V, PF_HALF_BYTES, 1024);
        bool ok = true;
        named_barrier_sync(Q_BARRIER, Q_BARRIER_THREADS);      // Q is in shared memory
        auto wait_lane0 = [&](uint32_t bar, uint32_t parity) -> bool {
            return mbar_wait_bounded(bar, parity, p.wait_ns);
        };
        auto issue_pv = [&](int t, int j) {                   // O_t += P_t(j) V(j)
            const uint64_t dv = dv0 + (uint64_t)((j % PF_VSTAGES) * (PF_KV_BYTES >> 4));
            const uint32_t pt = tmem + t * 256, ot = pt + 128;
            const uint32_t acc0 = j > 0 ? 1u : 0u;
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < (SPLIT_P ? 2 : 1); ++part) {
#pragma unroll
                for (int ks = 0; ks < PF_BN / 16; ++ks)
                    umma_f16_tmem_a(ot, pt + part * (PF_BN / 2) + ks * 8, dv + (uint64_t)((ks * 16 * 128) >> 4),
                                    idesc_o, (ks > 0 || part > 0) ? 1u : acc0);
            }
        };
        auto issue_s = [&](int t, int j) {                    // S_t = Q_t K(j)^T
            const uint64_t dk = dk0 + (uint64_t)((j % PF_KSTAGES) * (PF_KV_BYTES >> 4));
            const uint64_t dq = dq0 + (uint64_t)(t * (PF_Q_BYTES >> 4));
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < PF_D / 16; ++ks)
                umma_f16(tmem + t * 256, dq + (uint64_t)(((ks >> 2) * (PF_BM * 128) + (ks & 3) * 32) >> 4),
                         dk + (uint64_t)(((ks >> 2) * PF_HALF_BYTES + (ks & 3) * 32) >> 4), idesc_s,
                         ks > 0 ? 1u : 0u);
            umma_commit(bar_s_full + t * 8);
        };
        // V(j) has arrived: zero its rows past the context (other tokens' data or stale words)
        auto v_ready = [&](int j) -> bool {
            const int st = j % PF_VSTAGES;
            if (!wait_lane0(bar_v_full + st * 8, (uint32_t)(j / PF_VSTAGES) & 1u)) return false;
            consumed_v = j + 1;
            const int t0 = key0 + j * PF_BN;
            if (t0 + PF_BN > L) {
                const int nvalid = L - t0 > 0 ? L - t0 : 0;
                const int nz = (PF_BN - nvalid) * 8;           // 16-byte chunks per half
                uint8_t *vg = smem + PF_OFF_V + st * PF_KV_BYTES;
                for (int c = 0; c < 2 * nz; ++c) {
                    const int hf = c / nz, rc = c - hf * nz;
                    *reinterpret_cast<uint4 *>(vg + hf * PF_HALF_BYTES + (nvalid + rc / 8) * 128 + (rc % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            return true;
        };
        if (lane == 0) {                                       // one thread issues; the warp's other lanes idle
        for (int j = 0; j < ntiles && ok; ++j) {
            if (!(ok = wait_lane0(bar_k_full + (j % PF_KSTAGES) * 8, (uint32_t)(j / PF_KSTAGES) & 1u))) break;
            consumed_k = j + 1;
            if (j > 0 && !(ok = v_ready(j - 1))) break;
            if (j > 0 && j - 1 < nt0) {
                if (!(ok = wait_lane0(bar_p_full, (uint32_t)(j - 1) & 1u))) break;
                if (lane == 0) issue_pv(0, j - 1);
            }
            if (j < nt0 && lane == 0) issue_s(0, j);
            if (j > 0 && j - 1 < nt1) {
                if (!(ok = wait_lane0(bar_p_full + 8, (uint32_t)(j - 1) & 1u))) break;
                if (lane == 0) issue_pv(1, j - 1);
            }
            if (j < nt1 && lane == 0) issue_s(1, j);
            umma_commit(bar_k_empty + (j % PF_KSTAGES) * 8);   // frees K(j), and V(j - 1) after P(j-1).V
        }
        if (ok && ntiles > 0) {
            ok = v_ready(ntiles - 1);
            if (ok && ntiles - 1 < nt0) {
                ok = wait_lane0(bar_p_full, (uint32_t)(ntiles - 1) & 1u);
                if (ok && lane == 0) issue_pv(0, ntiles - 1);
            }
            if (ok && ntiles - 1 < nt1) {
                ok = wait_lane0(bar_p_full + 8, (uint32_t)(ntiles - 1) & 1u);
                if (ok && lane == 0) issue_pv(1, ntiles - 1);
            }
            if (ok)
                for (int t = 0; t < PF_QT; ++t) umma_commit(bar_o_done + t * 8);
        }
        }
        __syncwarp();
        if (!ok) *abort_flag = 1;
      }
    } else {
        setmaxnreg_inc<PF_REGS_SOFTMAX>();
        {
            // the warp's 32 Q rows, two per load (16 lanes x 16 bytes = one 256-byte row, coalesced), into
            // 16 chunks of 8 values per row with the 128-byte swizzle
            uint8_t *qtile = smem + t_of * PF_Q_BYTES;
            const int c = lane & 15;
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {
                uint4 v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int src = 2 * (k0 + k) + (lane >> 4);
                    const int64_t orow_k = __shfl_sync(0xffffffffu, orow, src);
                    const bool ok_k = __shfl_sync(0xffffffffu, row_ok, src);
                    v[k] = ok_k ? __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) + orow_k * PF_D) + c)
                                : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rt_k = (warp & 3) * 32 + 2 * (k0 + k) + (lane >> 4);
                    *reinterpret_cast<uint4 *>(qtile + rt_k * 128 + (c >> 3) * (PF_BM * 128) +
                                               (((c & 7) ^ (rt_k & 7)) << 4)) = v[k];
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(Q_BARRIER, Q_BARRIER_THREADS);
        }
        // ---------------------------------------------------------------- softmax (row tile t_of)
        const int t = t_of;
        const int nt = t ? nt1 : nt0;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tmem_s = tmem + t * 256 + lane_base, tmem_o = tmem_s + 128;
        // last key this row may see (a cascade row follows the whole prefix)
        const int lim = CASCADE ? 0x7fffffff : L - p.q_len + qi;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_s_full + t * 8, (uint32_t)j & 1u, p.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float sv[PF_BN];
            tmem_ld_cols(tmem_s, sv);
            // raw-score max (the scale is positive, so it commutes with the max); eight independent
            // partial maxima and sums keep the dependent chains short
            const int t0 = key0 + j * PF_BN;
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
            // P(j-1).V completed before S(j) (one commit covers both): rescale this warp's O rows
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
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
            // P over S: 128 keys as 64 packed columns (bf16: hi in columns 0..63, lo = x - hi in 64..127)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) w[c] = pack2<T>(sv[64 * q + 2 * c], sv[64 * q + 2 * c + 1]);
                tmem_st32_raw(tmem_s + 32 * q, w);
                if constexpr (SPLIT_P) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        // a bf16 is the top half of an fp32
                        const float h0 = __uint_as_float(w[c] << 16), h1 = __uint_as_float(w[c] & 0xFFFF0000u);
                        w[c] = pack2<T>(sv[64 * q + 2 * c] - h0, sv[64 * q + 2 * c + 1] - h1);
                    }
                    tmem_st32_raw(tmem_s + PF_BN / 2 + 32 * q, w);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_p_full + t * 8);
        }
        if (ok && nt > 0)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_o_done + t * 8, 0u, p.wait_ns));
        if (!ok) {
            if (lane == 0) *abort_flag = 1;
        } else if (nt > 0) {
            // the warp's 32 output rows go through the free copy rings (all MMAs have completed and every
            // copy was consumed): each thread stages its row, then the warp stores row by row, coalesced.
            // A cascade writes the unnormalised state of the chunk's keys in its first partition slot; the
            // chunk's other slots get sum 0, which the merge reads as empty
            tc_fence_after();
            float *stage = reinterpret_cast<float *>(smem + PF_OFF_K) + warp * 32 * PF_STAGE_STRIDE;
            float *mine = stage + lane * PF_STAGE_STRIDE;
            const float sc = CASCADE ? 1.f : 1.f / l;
#pragma unroll
            for (int c0 = 0; c0 < PF_D; c0 += 32) {
                float a[32];
                tmem_ld32(tmem_o + c0, a);
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(mine + c0 + c) = make_float4(a[c] * sc, a[c + 1] * sc, a[c + 2] * sc,
                                                                             a[c + 3] * sc);
            }
            __syncwarp();
            const int slot0 = CASCADE ? key0 / p.part_tokens : 0;
#pragma unroll 4
            for (int k = 0; k < 32; ++k) {
                const int64_t orow_k = __shfl_sync(0xffffffffu, orow, k);
                const bool ok_k = __shfl_sync(0xffffffffu, row_ok, k);
                const float4 x = *reinterpret_cast<const float4 *>(stage + k * PF_STAGE_STRIDE + lane * 4);
                if (ok_k) {
                    if constexpr (CASCADE) {
                        *reinterpret_cast<float4 *>(p.part_o + (orow_k * p.max_parts + slot0) * PF_D + lane * 4) = x;
                    } else {
                        T *dst = reinterpret_cast<T *>(p.out) + orow_k * PF_D + lane * 4;
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack2<T>(x.x, x.y), pack2<T>(x.z, x.w));
                    }
                }
            }
            if (CASCADE && row_ok) {
                const int slot1 = L / p.part_tokens;
                p.part_ml[orow * p.max_parts + slot0] = make_float2(m_ref, l);
                for (int sl = slot0 + 1; sl < slot1; ++sl) p.part_ml[orow * p.max_parts + sl] = make_float2(0.f, 0.f);
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
            for (int j = consumed_k; j < issued_tiles[0]; ++j)
                mbar_wait_bounded(bar_k_full + (j % PF_KSTAGES) * 8, (uint32_t)(j / PF_KSTAGES) & 1u, p.wait_ns);
            for (int j = consumed_v; j < issued_tiles[1]; ++j)
                mbar_wait_bounded(bar_v_full + (j % PF_VSTAGES) * 8, (uint32_t)(j / PF_VSTAGES) & 1u, p.wait_ns);
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

template <typename T, bool CASCADE>
static cudaError_t launch_prefill_t(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                    cudaStream_t stream) {
    const int64_t rows = CASCADE ? (int64_t)p.num_seqs * p.rows : p.rows;
    const int64_t ctiles = ((rows + PF_BM - 1) / PF_BM + PF_QT - 1) / PF_QT;
    const int64_t units = CASCADE ? (int64_t)(p.part0 + p.pchunk - 1) / p.pchunk : (int64_t)p.num_seqs;
    const int64_t grid = units * p.Hkv * ctiles;
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<T, CASCADE>, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
    if (e != cudaSuccess) return e;
    prefill_kernel<T, CASCADE><<<(unsigned)grid, PF_THREADS, PF_SMEM, stream>>>(tmk, tmv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           cudaStream_t stream) {
    return dtype == PA_FP16 ? launch_prefill_t<__half, false>(p, tmk, tmv, stream)
                            : launch_prefill_t<__nv_bfloat16, false>(p, tmk, tmv, stream);
}

cudaError_t launch_prefix(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          cudaStream_t stream) {
    return dtype == PA_FP16 ? launch_prefill_t<__half, true>(p, tmk, tmv, stream)
                            : launch_prefill_t<__nv_bfloat16, true>(p, tmk, tmv, stream);
}

}  // namespace pa
