// verify.cu -- paged attention for 9..32 query rows per KV head (a head group's speculative draft
// rows, or a wide GQA group) on the 5th-generation tensor cores.
//
// What is computed is pa_decode's definition (learn.tanhdev.com "Part 8: Inference optimization
// with vLLM", section on executing the kernel math in CUDA: A_{i,j} = q_i K_(j)^T / sqrt(d_k),
// softmax across the blocks, o_i = sum_j sum_t a_{i,j,t} v_(j,t)), with the draft rows of a verify
// pass (itimpress.au section 1: the target checks the K = 5 drafted tokens in one parallel pass;
// yangyu.win blog #54 section 2.4) each seeing the context up to its own position. Work items are
// the decode's (sequence, KV head, context partition) triples, so partial states and the
// log-sum-exp merge are shared with decode.cu.
//
// Per 128-key tile:
//   S   [128 x 128 keys] = Q4 [128 x 128 d] . K_tile^T     (M128 N128 K16 x 8; Q4 in tensor memory)
//   O^T [128 d x NP]    += V_tile^T [128 d x 128 keys] . P^T [128 keys x NP]   (M128 N{64,32} K16 x 8)
// Q4 holds four copies of the head group's (up to 32) query rows, one per 32-lane quarter of tensor
// memory, so that each of the four softmax warps (a warp reaches only its own quarter) reads every
// row's scores for its own slice of 32 keys of the tile. The four slices share one running maximum
// per row (exchanged through shared memory each tile), so their weights are on one scale: each warp
// writes its slice of P^T (query rows on the N side) into shared memory and one product per tile
// accumulates every slice into O^T (head dimension on the lanes, one column per query row). bf16
// weights are carried as high parts bf16(p) in columns 0..31 and low parts bf16(p - hi) in columns
// 32..63 (8 significant bits alone fail the tolerance where weighted values cancel; the two halves
// cost one N = 64 product); fp16 needs only the 32 columns. The epilogue of an item is a read of
// O^T (each thread one dimension of every row) and coalesced row stores: no merge between warps.
// K and V tiles are read from shared memory by the tensor cores once per tile each.
//
// One persistent CTA per SM takes items from a counter shared by the launch (its first item is its own
// index; it holds at most two ahead of its copies, so CTAs that start late, beside another kernel, or run
// short items take more); every role follows the same sequence of tiles, so the copies of the next item
// start while the current one finishes.
//   warps 0-3   softmax of key slice w (rows of quarter w), then the item's epilogue: warp w stores
//               dimensions 32w..32w+31 of every row. Every sub-partition also hosts an issuing warp,
//               and a warp scheduler that keeps picking a busy softmax warp starves it (an MMA issued
//               from a sub-partition shared with one busy FP32 warp took 235 instead of 65 cycles),
//               so the softmax yields its issue slot (nanosleep 0) every 16 exponentials.
//   warp 4      MMA issue (one thread) and tensor-memory allocation.
//   warp 5      item fetch (one thread): the next item and its sequence's context length into a ring
//               that every role reads.
//   warp 6      V rows past an item: follows every V copy as it lands; in an item's last, partial tile it
//               zeroes the rows past the item (they may hold other data, NaN included, and a zero weight
//               times NaN is NaN); then it releases the tile's P.V. Done by the softmax before, it made the
//               softmax of every item's last tile wait for that tile's V copy, which lands about a tile after
//               K: ~4,000 cycles on the MMA chain per item.
//   warps 8-11  K producers, warps 12-15 V producers: each warp copies two 16-key sub-tiles of every
//               tile, one TMA box per 64-dimension half; block ids looked up one tile ahead (one warp's
//               copies are issued one after another, and TMA throughput scales with issuing warps).
//               The K producer of quarter q also writes the item's query rows into Q4's quarter q.
// Every wait is bounded and abortable; a timeout sets the status word, the CTA drains its copies
// and MMAs, frees tensor memory and returns without writing results.
#include "pa_device.cuh"

namespace pa {

constexpr int VF_KT = 128;                             // keys per tile
constexpr int VF_D = 128;                              // head dimension
constexpr int VF_ROWS = 32;                            // query rows per KV head, at most
constexpr int VF_KSTAGES = 2, VF_VSTAGES = 2;
constexpr int VF_TILE_BYTES = VF_KT * VF_D * 2;        // 32 KB: K or V tile, [2 halves][128 keys][128 B]
constexpr int VF_HALF_BYTES = VF_KT * 128;             // 16 KB
constexpr int VF_SW = 32;                              // keys per slice: one slice per softmax warp
constexpr int VF_P_BYTES = 16 * 1024;                  // one P^T buffer: [2 blocks of 64 keys][<= 64 rows][128 B]
constexpr int VF_OFF_K = 0;
constexpr int VF_OFF_V = VF_OFF_K + VF_KSTAGES * VF_TILE_BYTES;
constexpr int VF_OFF_P = VF_OFF_V + VF_VSTAGES * VF_TILE_BYTES;    // P^T [2 buffers]
constexpr int VF_OFF_O = VF_OFF_P + 2 * VF_P_BYTES;    // output rows of an item [32 rows][128 d] (fp32 or T)
constexpr int VF_OFF_X = VF_OFF_O + VF_ROWS * VF_D * 4;   // slice maxima [2 tiles][32 rows][4], slice sums [32][4]
constexpr int VF_QSLOTS = 8;                           // ring entries: items between the copies and the softmax
constexpr int VF_LOOKAHEAD = 2;                        // items a CTA holds ahead of its copies (its current one included)
constexpr int VF_OFF_RING = VF_OFF_X + 3 * VF_ROWS * 4 * 4;   // item ring: (item index or -1, context length)
constexpr int VF_OFF_BAR = VF_OFF_RING + VF_QSLOTS * 8;
// barriers: k_full[2] k_empty[2] v_full[2] v_empty[2] q_full[2] q_free[2] s_full[2] p_full[2] pv_done[2]
//           o_full o_free mx lx ost drain v_fixed[2] item_full[8] item_empty[8]
constexpr int VF_NBAR = 2 * VF_KSTAGES + 2 * VF_VSTAGES + 5 * 2 + 6 + 2 + 2 * VF_QSLOTS;
// roles that read every item of the ring: 4 K producer warps, 4 V producer warps, the MMA thread, 4 softmax warps,
// the V-row warp
constexpr int VF_ITEM_READERS = 14;
constexpr int VF_OFF_MISC = VF_OFF_BAR + VF_NBAR * 8;  // tmem slot, abort flag, issued counters [2][4], items taken
constexpr int VF_SMEM = 1024 + VF_OFF_MISC + 64;
static_assert(VF_OFF_BAR % 8 == 0, "barrier alignment");
static_assert(VF_SMEM <= 227 * 1024, "verify shared memory");

// 16 warps; warp 5 fetches the CTA's items, warp 6 zeroes V rows past the items, warp 7 only takes part in the
// prologue and teardown. Launched at 128 registers per thread;
// the softmax warpgroup raises its share and the other three lower theirs (setmaxnreg):
// 128 x 232 + 384 x 88 <= 512 x 128.
constexpr int VF_THREADS = 512;
constexpr int VF_MMA_WARP = 4, VF_SCHED_WARP = 5, VF_VFIX_WARP = 6, VF_KPROD_WARP = 8, VF_VPROD_WARP = 12;
constexpr uint32_t VF_REGS_HIGH = 232, VF_REGS_LOW = 88;
static_assert(128 * VF_REGS_HIGH + 384 * VF_REGS_LOW <= VF_THREADS * 128, "register split");
// tensor memory: Q4[2] at columns 0 / 64 (128 d as 64 packed columns), S[2] at 128 / 256, O^T at 384 (64 columns)
constexpr uint32_t VF_TMEM_COLS = 512;
constexpr uint32_t VF_COL_Q = 0, VF_COL_S = 128, VF_COL_O = 384;
constexpr float VF_RESCALE_LOG2 = 8.f;                 // stale-max headroom (P <= 2^8)

size_t verify_smem_bytes() { return VF_SMEM; }

template <typename T>
__device__ __forceinline__ T vf_round(float x);
template <>
__device__ __forceinline__ __half vf_round<__half>(float x) {
    return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 vf_round<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Copies keep the normal L2 priority: blocks shared by several tables (a copy-on-write prefix) are read
// again by other CTAs, other blocks once.
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One poll of a barrier phase that suspends the thread (up to `hint_ns`) until the phase completes
// instead of returning at once: waiting threads give their sub-partition's issue slots to the others.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Bounded wait that also gives up when another role has aborted the CTA. Each poll suspends for up
// to 1 us (the phase's completion ends it early); roles that run ahead of the others (copies, Q loads)
// pass a back-off and also sleep between polls.
__device__ __forceinline__ bool vf_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort_flag,
                                        uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try_wait_suspend(bar, parity, 1000u)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait until a counter another warp advances reaches `target` (or another role aborted).
__device__ __forceinline__ bool vf_wait_count(volatile int *cnt, int target, uint64_t limit_ns, volatile int *abort_flag) {
    if (*cnt >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(128);
        if (*cnt >= target) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}

struct VfItem {
    int idx;              // item index: (sequence, KV head, partition)
    int b, g, part, L;
    int t_begin, t_end;   // the item's tokens [t_begin, t_end): its partition, cut at the context end
    int ntiles;
};

// The CTA's items, in the order one thread of the CTA took them from the launch's shared counter (so
// that CTAs which start late, or whose items are short, take more): every role reads the same ring of
// (item, context length) entries and releases each entry once read. next() returns 1 for an item,
// 0 at the end, -1 when the wait gave up (timeout or abort).
struct VfItems {
    const DecodeParams &p;
    const int2 *ring;
    uint32_t full0, empty0;
    volatile int *abort_flag;
    int nlaunch, k;
    bool whole_warp;   // all 32 lanes call next() (lane 0 releases the entry), else one thread

    __device__ __forceinline__ VfItems(const DecodeParams &p_, const int2 *ring_, uint32_t full0_, uint32_t empty0_,
                                       volatile int *abort_, int nlaunch_, bool whole_warp_)
        : p(p_), ring(ring_), full0(full0_), empty0(empty0_), abort_flag(abort_), nlaunch(nlaunch_), k(0),
          whole_warp(whole_warp_) {}

    __device__ __forceinline__ int next(VfItem &it) {
        const int slot = k % VF_QSLOTS;
        bool got = vf_wait(full0 + slot * 8, (uint32_t)(k / VF_QSLOTS) & 1u, p.wait_ns, abort_flag);
        if (whole_warp) got = __all_sync(0xffffffffu, got);
        if (!got) return -1;
        const volatile int *e = reinterpret_cast<const volatile int *>(ring + slot);
        const int idx = e[0], Lraw = e[1];
        if (whole_warp) __syncwarp();
        if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(empty0 + slot * 8);
        ++k;
        if (idx < 0) return 0;
        it.idx = idx;
        it.part = p.part0 + idx % nlaunch;
        const int bg = idx / nlaunch;
        it.g = bg % p.Hkv;
        it.b = bg / p.Hkv;
        const int L = Lraw < 0 ? 0 : (Lraw > p.max_ctx ? p.max_ctx : Lraw);
        it.L = L;
        const int nparts = (L + p.part_tokens - 1) / p.part_tokens;
        it.t_begin = it.part * p.part_tokens;
        if (it.part >= nparts) {
            it.t_end = it.t_begin;
            it.ntiles = 0;
        } else {
            it.t_end = min(it.t_begin + p.part_tokens, L);
            it.ntiles = (it.t_end - it.t_begin + VF_KT - 1) / VF_KT;
        }
        return 1;
    }
};

template <typename T>
__global__ void __launch_bounds__(VF_THREADS, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
    constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
    constexpr int NP = SPLIT_P ? 64 : 32;                // P^T rows = O^T columns (bf16: high parts, then low parts)
    constexpr int PBLK = NP * 128;                        // bytes of one 64-key block of P^T
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_u32);
    const uint32_t bar_k_full = base + VF_OFF_BAR;
    const uint32_t bar_k_empty = bar_k_full + VF_KSTAGES * 8;
    const uint32_t bar_v_full = bar_k_empty + VF_KSTAGES * 8;
    const uint32_t bar_v_empty = bar_v_full + VF_VSTAGES * 8;
    const uint32_t bar_q_full = bar_v_empty + VF_VSTAGES * 8;
    const uint32_t bar_q_free = bar_q_full + 16;
    const uint32_t bar_s_full = bar_q_free + 16;
    const uint32_t bar_p_full = bar_s_full + 16;
    const uint32_t bar_pv_done = bar_p_full + 16;
    const uint32_t bar_o_full = bar_pv_done + 16;
    const uint32_t bar_o_free = bar_o_full + 8;
    const uint32_t bar_mx = bar_o_free + 8;
    const uint32_t bar_lx = bar_mx + 8;
    const uint32_t bar_ost = bar_lx + 8;
    const uint32_t bar_drain = bar_ost + 8;
    const uint32_t bar_v_fixed = bar_drain + 8;   // [2 stages]: the V tile is ready for its P.V (rows past the item zeroed)
    const uint32_t bar_item_full = bar_v_fixed + 16;
    const uint32_t bar_item_empty = bar_item_full + VF_QSLOTS * 8;
    int2 *item_ring = reinterpret_cast<int2 *>(smem + VF_OFF_RING);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + VF_OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *issued = reinterpret_cast<volatile int *>(tmem_slot + 2);   // [K warps 0..3, V warps 0..3]
    volatile int *taken = reinterpret_cast<volatile int *>(tmem_slot + 10);   // ring entries the copies have started
    float *mxs = reinterpret_cast<float *>(smem + VF_OFF_X);                   // [2 tiles][32 rows][4 slices]
    float *lsx = mxs + 2 * VF_ROWS * 4;                                        // [32 rows][4 slices]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // launched with programmatic serialization: the merge behind this kernel may be launched now (its CTAs wait
    // for this grid's end); this kernel waits for the work ahead of it before reading anything
    pdl_trigger();
    pdl_wait();
    const int nlaunch = p.max_parts - p.part0;
    const int n_items = p.num_seqs * p.Hkv * nlaunch;

    // ---- prologue: barriers, tensor memory
    if (warp == VF_MMA_WARP) tmem_alloc(smem_u32(tmem_slot), VF_TMEM_COLS);
    if (tid == 0) {
        for (int s = 0; s < VF_KSTAGES; ++s) {
            mbar_init(bar_k_full + s * 8, 4);
            mbar_init(bar_k_empty + s * 8, 1);
        }
        for (int s = 0; s < VF_VSTAGES; ++s) {
            mbar_init(bar_v_full + s * 8, 4);
            mbar_init(bar_v_empty + s * 8, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_q_full + s * 8, 128);
            mbar_init(bar_q_free + s * 8, 1);
            mbar_init(bar_s_full + s * 8, 1);
            mbar_init(bar_p_full + s * 8, 128);
            mbar_init(bar_pv_done + s * 8, 1);
        }
        mbar_init(bar_o_full, 1);
        mbar_init(bar_o_free, 128);
        mbar_init(bar_mx, 128);
        mbar_init(bar_lx, 128);
        mbar_init(bar_ost, 128);
        mbar_init(bar_drain, 1);
        mbar_init(bar_v_fixed, 32);
        mbar_init(bar_v_fixed + 8, 32);
        for (int s = 0; s < VF_QSLOTS; ++s) {
            mbar_init(bar_item_full + s * 8, 1);
            mbar_init(bar_item_empty + s * 8, VF_ITEM_READERS);
        }
        *abort_flag = 0;
        for (int i = 0; i < 8; ++i) issued[i] = 0;
        *taken = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int consumed_k = 0, consumed_v = 0;   // MMA thread: tiles whose copies were seen to land

    if (warp >= 4) {
        setmaxnreg_dec<VF_REGS_LOW>();
        if (warp >= VF_KPROD_WARP) {
            // ------------------------------------------------------------------ K / V producers
            const bool is_v = warp >= VF_VPROD_WARP;
            const int pw = warp - (is_v ? VF_VPROD_WARP : VF_KPROD_WARP);   // also the tensor-memory quarter
            const int NS = is_v ? VF_VSTAGES : VF_KSTAGES;
            const uint32_t full0 = is_v ? bar_v_full : bar_k_full;
            const uint32_t empty0 = is_v ? bar_v_empty : bar_k_empty;
            const uint32_t ring = base + (is_v ? VF_OFF_V : VF_OFF_K);
            const CUtensorMap *map = is_v ? &tmv : &tmk;
            const int sub = 2 * pw + ((lane >> 1) & 1);   // lanes 0..3: two sub-tiles x two halves
            const int h = lane & 1;
            const uint64_t policy = l2_policy_evict_normal();
            const uint32_t q_lane_base = (uint32_t)(pw * 32) << 16;
            const int qn = lane, qqi = qn < p.rows ? qn / p.G : 0, qhh = qn - qqi * p.G;
            int jj = 0, ii = 0;
            bool ok = true;
            VfItems items(p, item_ring, bar_item_full, bar_item_empty, abort_flag, nlaunch, true);
            VfItem it;
            while (ok) {
                const int got = items.next(it);
                if (got <= 0) {
                    ok = got == 0;
                    break;
                }
                if (!is_v && pw == 0 && lane == 0) *taken = items.k;   // lets the fetch take the next item
                if (!is_v && pw == 0 && it.part == p.part0) {
                    const int Lraw = __ldg(p.context_lens + it.b);
                    if ((Lraw < p.q_len || Lraw > p.max_ctx) && lane == 0) set_status(p.status, STATUS_BOUNDS);
                    if (p.part0 > 0 && it.g == 0) {
                        // shared-prefix decode: the prefix kernel read sequence 0's blocks for every sequence and
                        // assumed that every query row follows the whole prefix; check both for this sequence
                        const int pre_blocks = p.part0 * p.part_tokens / p.bs;
                        if (it.L - p.q_len < p.part0 * p.part_tokens && lane == 0) set_status(p.status, STATUS_BOUNDS);
                        for (int i = lane; i < pre_blocks; i += 32)
                            if (__ldg(p.block_tables + (int64_t)it.b * p.stride + i) != __ldg(p.block_tables + i))
                                set_status(p.status, STATUS_BOUNDS);
                    }
                }
                if (it.ntiles == 0) continue;
                const int32_t *trow = p.block_tables + (int64_t)it.b * p.stride;
                const int tok0 = it.t_begin + sub * TILE_TOKENS;      // this lane's sub-tile in tile 0
                int id_next = (lane < 4 && tok0 < it.t_end) ? __ldg(trow + tok0 / p.bs) : 0;
                if (!is_v) {
                    // the item's query rows into quarter pw of Q4 (buffer ii & 1, free once the item two before
                    // has had its last S)
                    if (ii >= 2 &&
                        !__all_sync(0xffffffffu, vf_wait(bar_q_free + (ii & 1) * 8, (uint32_t)((ii >> 1) - 1) & 1u,
                                                         p.wait_ns, abort_flag, 256))) {
                        ok = false;
                        break;
                    }
                    const uint4 *qrow = reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const T *>(p.q) + (((int64_t)it.b * p.q_len + qqi) * p.Hq + it.g * p.G + qhh) * VF_D);
                    const uint32_t qcol = tmem + q_lane_base + VF_COL_Q + (ii & 1) * 64;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t w[32];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 v = qn < p.rows ? __ldg(qrow + 8 * half + c) : make_uint4(0u, 0u, 0u, 0u);
                            w[4 * c] = v.x;
                            w[4 * c + 1] = v.y;
                            w[4 * c + 2] = v.z;
                            w[4 * c + 3] = v.w;
                        }
                        tmem_st32_raw(qcol + 32 * half, w);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar_q_full + (ii & 1) * 8);
                }
                ++ii;
                for (int t = 0; t < it.ntiles; ++t, ++jj) {
                    const int tok = tok0 + t * VF_KT;
                    const bool valid = lane < 4 && tok < it.t_end;
                    int id = id_next;
                    // the block id of the next tile's sub-tile is loaded now, used one tile later
                    if (t + 1 < it.ntiles && lane < 4 && tok + VF_KT < it.t_end) id_next = __ldg(trow + (tok + VF_KT) / p.bs);
                    const int st = jj % NS;
                    if (jj >= NS) {
                        const bool got = vf_wait(empty0 + st * 8, (uint32_t)((jj / NS) - 1) & 1u, p.wait_ns, abort_flag, 256);
                        if (!__all_sync(0xffffffffu, got)) {
                            ok = false;
                            break;
                        }
                    }
                    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
                    if (lane == 0) mbar_arrive_expect_tx(full0 + st * 8, (uint32_t)__popc(vmask) * (TILE_TOKENS * 128));
                    __syncwarp();
                    if (valid) {
                        if (id < 0 || id >= p.num_blocks) {
                            set_status(p.status, STATUS_BOUNDS);
                            id = 0;
                        }
                        const int row0 = (id * p.Hkv + it.g) * p.bs + tok % p.bs;
                        tma_load_2d(ring + st * VF_TILE_BYTES + h * VF_HALF_BYTES + sub * TILE_TOKENS * 128, map,
                                    h * 64, row0, full0 + st * 8, policy);
                    }
                }
            }
            if (lane == 0) issued[(is_v ? 4 : 0) + pw] = jj;
        } else if (warp == VF_MMA_WARP) {
            // ------------------------------------------------------------------ MMA issue (lane 0)
            if (lane == 0) {
                const uint32_t idesc_s = umma_idesc<T>(128, VF_KT, false);
                // O^T = V^T P^T: A = the V tile read M(= d)-major (bit 15), B = P^T, K-major
                const uint32_t idesc_o = umma_idesc<T>(128, NP, false) | (1u << 15);
                const uint64_t dk0 = umma_desc_sw128(base + VF_OFF_K, 16, 1024);
                const uint64_t dv0 = umma_desc_sw128(base + VF_OFF_V, VF_HALF_BYTES, 1024);
                const uint64_t dp0 = umma_desc_sw128(base + VF_OFF_P, 16, 1024);
                bool ok = true;
                int jj = 0, ii = 0;
                int pv_jj = -1, pv_ii = 0;
                bool pv_first = false, pv_last = false;
                auto do_pv = [&]() -> bool {       // O^T += V(pv_jj)^T P(pv_jj)^T
                    if (!vf_wait(bar_p_full + (pv_jj & 1) * 8, (uint32_t)(pv_jj >> 1) & 1u, p.wait_ns, abort_flag))
                        return false;
                    if (!vf_wait(bar_v_full + (pv_jj % VF_VSTAGES) * 8, (uint32_t)(pv_jj / VF_VSTAGES) & 1u, p.wait_ns,
                                 abort_flag))
                        return false;
                    consumed_v = pv_jj + 1;
                    // the V-row warp has seen the tile land (and zeroed the rows past the item of a partial tile)
                    if (!vf_wait(bar_v_fixed + (pv_jj % VF_VSTAGES) * 8, (uint32_t)(pv_jj / VF_VSTAGES) & 1u, p.wait_ns,
                                 abort_flag))
                        return false;
                    // the item's first product overwrites O: the previous item's epilogue must have read it
                    if (pv_first && pv_ii >= 1 &&
                        !vf_wait(bar_o_free, (uint32_t)(pv_ii - 1) & 1u, p.wait_ns, abort_flag))
                        return false;
                    tc_fence_after();
                    const uint64_t dv = dv0 + (uint64_t)(((pv_jj % VF_VSTAGES) * VF_TILE_BYTES) >> 4);
                    const uint64_t dp = dp0 + (uint64_t)(((pv_jj & 1) * VF_P_BYTES) >> 4);
#pragma unroll
                    for (int ks = 0; ks < VF_KT / 16; ++ks)
                        umma_f16(tmem + VF_COL_O, dv + (uint64_t)((ks * 16 * 128) >> 4),
                                 dp + (uint64_t)(((ks >> 2) * PBLK + (ks & 3) * 32) >> 4), idesc_o,
                                 (ks > 0 || !pv_first) ? 1u : 0u);
                    umma_commit(bar_v_empty + (pv_jj % VF_VSTAGES) * 8);
                    umma_commit(bar_pv_done + (pv_jj & 1) * 8);
                    if (pv_last) umma_commit(bar_o_full);
                    return true;
                };
                VfItems items(p, item_ring, bar_item_full, bar_item_empty, abort_flag, nlaunch, false);
                VfItem it;
                while (ok) {
                    const int got = items.next(it);
                    if (got <= 0) {
                        ok = got == 0;
                        break;
                    }
                    if (it.ntiles == 0) continue;
                    if (!(ok = vf_wait(bar_q_full + (ii & 1) * 8, (uint32_t)(ii >> 1) & 1u, p.wait_ns, abort_flag)))
                        break;
                    const uint32_t qcol = tmem + VF_COL_Q + (ii & 1) * 64;
                    for (int t = 0; t < it.ntiles; ++t, ++jj) {
                        // the previous item's last P.V first: its epilogue waits on it, the first S of this item
                        // is not needed before that epilogue ends
                        if (t == 0 && pv_jj >= 0) {
                            if (!(ok = do_pv())) break;
                            pv_jj = -1;
                        }
                        if (!(ok = vf_wait(bar_k_full + (jj % VF_KSTAGES) * 8, (uint32_t)(jj / VF_KSTAGES) & 1u,
                                           p.wait_ns, abort_flag)))
                            break;
                        consumed_k = jj + 1;
                        tc_fence_after();
                        // S(jj) = Q4 K(jj)^T into S buffer jj & 1; it is issued after P(jj-2).V, whose weights came
                        // from that buffer and whose P^T buffer the softmax of tile jj rewrites (one thread's MMAs
                        // execute in order, and the commit of S(jj) covers P(jj-2).V)
                        const uint64_t dk = dk0 + (uint64_t)(((jj % VF_KSTAGES) * VF_TILE_BYTES) >> 4);
                        const uint32_t scol = tmem + VF_COL_S + (jj & 1) * 128;
#pragma unroll
                        for (int ks = 0; ks < VF_D / 16; ++ks)
                            umma_f16_tmem_a(scol, qcol + ks * 8,
                                            dk + (uint64_t)(((ks >> 2) * VF_HALF_BYTES + (ks & 3) * 32) >> 4), idesc_s,
                                            ks > 0 ? 1u : 0u);
                        umma_commit(bar_k_empty + (jj % VF_KSTAGES) * 8);
                        umma_commit(bar_s_full + (jj & 1) * 8);
                        if (t == it.ntiles - 1) umma_commit(bar_q_free + (ii & 1) * 8);
                        if (pv_jj >= 0 && !(ok = do_pv())) break;
                        pv_jj = jj;
                        pv_ii = ii;
                        pv_first = t == 0;
                        pv_last = t == it.ntiles - 1;
                    }
                    ++ii;
                }
                if (ok && pv_jj >= 0) ok = do_pv();
                if (!ok) *abort_flag = 1;
            }
            __syncwarp();
        } else if (warp == VF_SCHED_WARP) {
            // ------------------------------------------------------------------ item fetch (lane 0)
            // the CTA's first item is its own index; each later one comes from the launch's shared counter, taken
            // only once the copies have started the item before it (a CTA reserves at most VF_LOOKAHEAD items, so
            // CTAs that start late or run short items take more); with it goes its sequence's context length.
            // -1 marks the end.
            if (lane == 0) {
                for (int k = 0;; ++k) {
                    const int slot = k % VF_QSLOTS;
                    if (k >= VF_QSLOTS && !vf_wait(bar_item_empty + slot * 8, (uint32_t)((k / VF_QSLOTS) - 1) & 1u,
                                                   p.wait_ns, abort_flag, 256))
                        break;
                    if (k >= VF_LOOKAHEAD && !vf_wait_count(taken, k - VF_LOOKAHEAD + 1, p.wait_ns, abort_flag)) break;
                    int idx = k == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.vf_work, 1);
                    int L = 0;
                    if (idx >= n_items) idx = -1;
                    else L = __ldg(p.context_lens + idx / nlaunch / p.Hkv);
                    item_ring[slot] = make_int2(idx, L);
                    mbar_arrive(bar_item_full + slot * 8);
                    if (idx < 0) break;
                }
            }
            __syncwarp();
        } else if (warp == VF_VFIX_WARP) {
            // ------------------------------------------------------------------ V rows past an item
            // Every V tile, in order: wait for its copy, zero the rows past the item in a partial tile, release its
            // P.V (v_fixed has the stages and phases of v_full). Waiting on every tile keeps this warp from running
            // ahead of the copies (a parity wait two phases ahead would pass at once), and since the P.V of each
            // tile waits for this release, no copy into the stage can land before this warp has seen the one before.
            int jj = 0;
            bool ok = true;
            VfItems items(p, item_ring, bar_item_full, bar_item_empty, abort_flag, nlaunch, true);
            VfItem it;
            while (ok) {
                const int got = items.next(it);
                if (got <= 0) {
                    ok = got == 0;
                    break;
                }
                for (int t = 0; t < it.ntiles; ++t, ++jj) {
                    ok = __all_sync(0xffffffffu, vf_wait(bar_v_full + (jj % VF_VSTAGES) * 8,
                                                         (uint32_t)(jj / VF_VSTAGES) & 1u, p.wait_ns, abort_flag, 64));
                    if (!ok) break;
                    const int nvalid = it.t_end - (it.t_begin + t * VF_KT);
                    if (nvalid < VF_KT) {
                        uint8_t *vt = smem + VF_OFF_V + (jj % VF_VSTAGES) * VF_TILE_BYTES;
                        // two rows per step: a row is 2 x 128 bytes (both 64-dimension halves), 16 lanes x 16 bytes
                        for (int c = nvalid + (lane >> 4); c < VF_KT; c += 2)
                            *reinterpret_cast<uint4 *>(vt + ((lane >> 3) & 1) * VF_HALF_BYTES + c * 128 +
                                                       (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();   // the zeroed rows are read by the tensor cores
                    }
                    mbar_arrive(bar_v_fixed + (jj % VF_VSTAGES) * 8);
                }
            }
            if (!ok) *abort_flag = 1;
            __syncwarp();
        }
    } else {
        setmaxnreg_inc<VF_REGS_HIGH>();
        // ---------------------------------------------------------------------- softmax of slice `warp`, epilogue
        const int slice = warp;                              // keys [32 w, 32 w + 32) of every tile
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int n = lane;                                  // query row (of the head group)
        const int qi = n < p.rows ? n / p.G : p.q_len - 1;
        // this row's P^T rows (high parts: row n; low parts: row 32 + n) inside the slice's 64-key block, 128-byte
        // swizzled: the 16-byte chunk j of a row lands at chunk j ^ (row & 7)
        const uint32_t p_hi = base + VF_OFF_P + (slice >> 1) * PBLK + (n >> 3) * 1024 + (n & 7) * 128;
        const uint32_t p_lo = p_hi + 4 * 1024;
        const int chunk0 = (slice & 1) * 4;
        const int n_qi = n < p.rows ? n / p.G : 0;         // query position of row n (0 for padding rows)
        int jj = 0, ii = 0;
        bool ok = true;
        VfItems items(p, item_ring, bar_item_full, bar_item_empty, abort_flag, nlaunch, true);
        VfItem it;
        while (ok) {
            const int got = items.next(it);
            if (got <= 0) {
                ok = got == 0;
                break;
            }
            if (it.ntiles == 0) continue;
            const int lim = it.L - p.q_len + qi;              // last key this row sees
            float m_ref = -INFINITY, l = 0.f;                 // the row's reference max (all slices) and slice sum
            for (int t = 0; t < it.ntiles; ++t, ++jj) {
                ok = __all_sync(0xffffffffu, vf_wait(bar_s_full + (jj & 1) * 8, (uint32_t)(jj >> 1) & 1u, p.wait_ns,
                                                     abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint32_t scol = tmem + lane_base + VF_COL_S + (jj & 1) * 128;
                float sv[VF_SW];
                tmem_ld_cols<VF_SW>(scol + slice * VF_SW, sv);
                const int t0 = it.t_begin + t * VF_KT;
                const int k0 = t0 + slice * VF_SW;            // absolute index of the slice's first key
                // last visible key of this row in the slice (keys past the item or the row's limit are masked)
                const int cut = min(it.t_end - 1, lim) - k0;
                float m4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = -INFINITY;
                if (cut >= VF_SW - 1) {
#pragma unroll
                    for (int c = 0; c < VF_SW; ++c) m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < VF_SW; ++c) {
                        sv[c] = c <= cut ? sv[c] : -INFINITY;
                        m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
                    }
                }
                // the tile's maximum of the row over all four slices
                float *mrow = mxs + ((jj & 1) * VF_ROWS + n) * 4;
                mrow[slice] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
                mbar_arrive(bar_mx);
                __nanosleep(0);   // let the MMA warp of this sub-partition issue
                ok = __all_sync(0xffffffffu, vf_wait(bar_mx, (uint32_t)jj & 1u, p.wait_ns, abort_flag));
                if (!ok) break;
                const float4 mv = *reinterpret_cast<const float4 *>(mrow);
                const float mx = fmaxf(fmaxf(mv.x, mv.y), fmaxf(mv.z, mv.w));
                float alpha = 1.f;
                bool rescale = false;
                if (mx > m_ref + VF_RESCALE_LOG2 || (m_ref == -INFINITY && mx > -INFINITY)) {
                    alpha = m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - mx);
                    m_ref = mx;
                    rescale = true;
                }
                // every slice takes the same decision for a row, so the four warps agree on this vote
                if (t > 0 && __any_sync(0xffffffffu, rescale)) {
                    // O^T holds the item's P.V up to tile t-1: wait for that product, then rescale the columns of
                    // the rows whose reference max moved (this warp's 32 dimensions of each)
                    ok = __all_sync(0xffffffffu, vf_wait(bar_pv_done + ((jj - 1) & 1) * 8,
                                                         (uint32_t)((jj - 1) >> 1) & 1u, p.wait_ns, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < NP; c0 += 32) {
                        float a[32];
                        tmem_ld32(tmem + lane_base + VF_COL_O + c0, a);
#pragma unroll
                        for (int c = 0; c < 32; ++c) a[c] *= __shfl_sync(0xffffffffu, alpha, c);
                        tmem_st32(tmem + lane_base + VF_COL_O + c0, a);
                    }
                }
                const float nmuse = m_ref == -INFINITY ? 0.f : -m_ref;
                float r4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) r4[i] = 0.f;
#pragma unroll
                for (int c = 0; c < VF_SW; ++c) {
                    sv[c] = ex2_approx(fmaf(sv[c], p.scale_log2, nmuse));
                    r4[c & 3] += sv[c];
                    if ((c & 15) == 15) __nanosleep(0);
                }
                l = l * alpha + ((r4[0] + r4[1]) + (r4[2] + r4[3]));
                // the slice's weights into P^T buffer jj & 1 (its previous reader, P(jj-2).V, completed before S(jj))
                {
                    const uint32_t pb = (uint32_t)(jj & 1) * VF_P_BYTES;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = sv[8 * j + 2 * e], x1 = sv[8 * j + 2 * e + 1];
                            hw[e] = pack2<T>(x0, x1);
                            if (SPLIT_P) {
                                // a bf16 is the top half of an fp32
                                const float h0 = __uint_as_float(hw[e] << 16), h1 = __uint_as_float(hw[e] & 0xFFFF0000u);
                                lw[e] = pack2<T>(x0 - h0, x1 - h1);
                            }
                        }
                        const uint32_t off = pb + (uint32_t)(((chunk0 + j) ^ (n & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(p_hi + off), "r"(hw[0]),
                                     "r"(hw[1]), "r"(hw[2]), "r"(hw[3])
                                     : "memory");
                        if (SPLIT_P)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(p_lo + off), "r"(lw[0]),
                                         "r"(lw[1]), "r"(lw[2]), "r"(lw[3])
                                         : "memory");
                    }
                }
                fence_proxy_async_smem();   // the weights are read by the tensor cores
                tc_fence_before();
                mbar_arrive(bar_p_full + (jj & 1) * 8);
            }
            if (!ok) break;
            // ---- epilogue of the item: O^T column n is row n's unnormalised output (bf16: plus column 32 + n)
            ok = __all_sync(0xffffffffu, vf_wait(bar_o_full, (uint32_t)ii & 1u, p.wait_ns, abort_flag));
            if (!ok) break;
            tc_fence_after();
            float oh[32], ol[32];
            tmem_ld32(tmem + lane_base + VF_COL_O, oh);
            if (SPLIT_P) tmem_ld32(tmem + lane_base + VF_COL_O + 32, ol);
            tc_fence_before();
            mbar_arrive(bar_o_free);
            // the row's sum over the four slices
            lsx[n * 4 + slice] = l;
            mbar_arrive(bar_lx);
            ok = __all_sync(0xffffffffu, vf_wait(bar_lx, (uint32_t)ii & 1u, p.wait_ns, abort_flag));
            if (!ok) break;
            const float4 lv = *reinterpret_cast<const float4 *>(lsx + n * 4);
            const float lsum = (lv.x + lv.y) + (lv.z + lv.w);
            {
                const bool direct = p.part0 == 0 && it.L <= p.part_tokens;   // the merge skips such sequences
                if (!direct && warp == 0 && n < p.rows) {
                    const int64_t orow_n = ((int64_t)it.b * p.q_len + n_qi) * p.Hq + it.g * p.G + (n - n_qi * p.G);
                    p.part_ml[orow_n * p.max_parts + it.part] = make_float2(m_ref, lsum);
                }
                // the item's rows into shared memory (warp w: dimensions 32w..32w+31 of each row; the previous item's
                // readers of these rows have all passed this item's sum exchange), then out in 16-byte stores (storing
                // each warp's 64- or 128-byte piece of every row straight from registers took ~4,000 cycles an item
                // on the shared-prefix verify workload, these few wide stores ~700)
                float sc[VF_ROWS];
                const float sc_n = direct ? 1.f / lsum : 1.f;
#pragma unroll
                for (int r = 0; r < VF_ROWS; ++r) sc[r] = __shfl_sync(0xffffffffu, sc_n, r);
                if (direct) {
                    T *orows = reinterpret_cast<T *>(smem + VF_OFF_O);                 // [32][128] T
#pragma unroll
                    for (int r = 0; r < VF_ROWS; ++r)
                        if (r < p.rows) orows[r * VF_D + 32 * warp + lane] = vf_round<T>((SPLIT_P ? oh[r] + ol[r] : oh[r]) * sc[r]);
                } else {
                    float *orows = reinterpret_cast<float *>(smem + VF_OFF_O);         // [32][128] fp32
#pragma unroll
                    for (int r = 0; r < VF_ROWS; ++r)
                        if (r < p.rows) orows[r * VF_D + 32 * warp + lane] = SPLIT_P ? oh[r] + ol[r] : oh[r];
                }
                mbar_arrive(bar_ost);
                ok = __all_sync(0xffffffffu, vf_wait(bar_ost, (uint32_t)ii & 1u, p.wait_ns, abort_flag));
                if (!ok) break;
                // row r is query position r / G, head g * G + r % G
                const int64_t obase = ((int64_t)it.b * p.q_len) * p.Hq + it.g * p.G;
                if (direct) {
                    // 256-byte rows: half a warp per row, warp w takes rows 2w, 2w + 1, 2w + 8, 2w + 9, ...
                    const int half = lane >> 4, c16 = lane & 15;
#pragma unroll 1
                    for (int r = 2 * warp + half; r < p.rows; r += 8) {
                        const int rq = r / p.G;
                        const int64_t orow = obase + (int64_t)rq * p.Hq + (r - rq * p.G);
                        const uint4 v = *reinterpret_cast<const uint4 *>(smem + VF_OFF_O + (r * VF_D) * sizeof(T) + 16 * c16);
                        *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) + orow * VF_D + 8 * c16) = v;
                    }
                } else {
                    // 512-byte partition-state rows: one warp per row
#pragma unroll 1
                    for (int r = warp; r < p.rows; r += 4) {
                        const int rq = r / p.G;
                        const int64_t orow = obase + (int64_t)rq * p.Hq + (r - rq * p.G);
                        const float4 v = *reinterpret_cast<const float4 *>(smem + VF_OFF_O + (r * VF_D + 4 * lane) * 4);
                        *reinterpret_cast<float4 *>(p.part_o + (orow * p.max_parts + it.part) * VF_D + 4 * lane) = v;
                    }
                }
            }
            ++ii;
        }
        if (!ok) *abort_flag = 1;
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait ran out: record it, then wait (bounded) for every copy and MMA still in flight so that
        // none lands in shared or tensor memory after the CTA has released them
        if (tid == 0) set_status(p.status, STATUS_TIMEOUT);
        if (warp == VF_MMA_WARP && lane == 0) {
            int ik = 0, iv = 0;
            for (int i = 0; i < 4; ++i) {
                ik = max(ik, (int)issued[i]);
                iv = max(iv, (int)issued[4 + i]);
            }
            for (int j = consumed_k; j < ik; ++j)
                mbar_wait_bounded(bar_k_full + (j % VF_KSTAGES) * 8, (uint32_t)(j / VF_KSTAGES) & 1u, p.wait_ns);
            for (int j = consumed_v; j < iv; ++j)
                mbar_wait_bounded(bar_v_full + (j % VF_VSTAGES) * 8, (uint32_t)(j / VF_VSTAGES) & 1u, p.wait_ns);
            umma_commit(bar_drain);
            mbar_wait_bounded(bar_drain, 0u, p.wait_ns);
        }
        __syncthreads();
    }
    if (warp == VF_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, VF_TMEM_COLS);
    }
    if (tid == 0) {
        // the last CTA to finish (every CTA has taken its last item by then) resets the counters for the next launch
        __threadfence();
        if (atomicAdd(p.vf_work + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(p.vf_work, 0);
            atomicExch(p.vf_work + 1, 0);
        }
    }
}

template <typename T>
static cudaError_t launch_verify_t(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                                   cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, VF_SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(verify_kernel<T>, dim3((unsigned)grid), dim3(VF_THREADS), VF_SMEM, stream, tmk, tmv, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_verify(const DecodeParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          int max_ctas, cudaStream_t stream) {
    if (p.rows < 1 || p.rows > VF_ROWS || p.vf_work == nullptr) return cudaErrorInvalidValue;
    const int64_t items = (int64_t)p.num_seqs * p.Hkv * (p.max_parts - p.part0);
    const int grid = (int)(items < max_ctas ? items : max_ctas);
    if (grid < 1) return cudaSuccess;
    return dtype == PA_FP16 ? launch_verify_t<__half>(p, tmk, tmv, grid, stream)
                            : launch_verify_t<__nv_bfloat16>(p, tmk, tmv, grid, stream);
}

}  // namespace pa
