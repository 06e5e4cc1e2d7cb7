// spec_verify.cu -- speculative rejection sampling after the target's one-pass verify of K
// draft tokens (yangyu.win blog #54, section 5 question 3; maths.nthquan ch. 17 "Speculative
// decoding", algorithm steps 3-4): draft x_i is kept with probability min(1, p_i(x_i) / q_i(x_i));
// the first rejected position is resampled from max(0, p_i - q_i) renormalised and later drafts
// are dropped; when every draft is kept, one more token is drawn from p_K.
//
// One CTA of 16 warps per sequence. Warp 0 runs the K accept tests in parallel (fp32: u * q < p) and
// takes the first failure. The draw is an inverse CDF over the vocabulary in three levels:
//   1. the row is cut into 256 segments of whole 512-value chunks; each warp sums 16 consecutive
//      segments into shared memory, streaming them through its own ring of three stages filled by
//      1-D bulk copies (rows that are not 16-byte aligned: coalesced float4 loads, eight 128-value
//      chunks in flight per lane, segments of whole 128-value chunks);
//   2. warp 0 scans the 256 segment sums and finds the first segment whose running sum passes
//      v * total;
//   3. the whole CTA walks that segment 512 values at a time, one value per thread (a warp scan, a
//      scan of the 16 warp sums), and the first value whose running sum passes the target is the
//      token.
// Sums are double-single (a float pair hi + lo: Knuth's two-sum, Dekker's fast two-sum, and the
// compensated sum of Ogita, Rump and Oishi within a lane), about 44 significant bits: near the fp64
// sums of the definition at the fp32 rate, as fp64 arithmetic is scarce on this part; comparisons
// with the target are exact comparisons of normalised pairs. A weight max(0, p - q) is formed
// exactly (Dekker's fast two-sum, exact whenever p >= q >= 0). A token is only ever drawn where its
// weight is > 0.
#include "pa_device.cuh"

namespace pa {

constexpr int SPEC_WARPS = 16;
constexpr int SPEC_THREADS = SPEC_WARPS * 32;
constexpr int SPEC_SEGS = 256;                         // segments per row
constexpr int SPEC_SEGS_WARP = SPEC_SEGS / SPEC_WARPS; // 16 consecutive segments summed by one warp
constexpr int SPEC_SEGS_LANE = SPEC_SEGS / 32;         // 8 consecutive segments per lane when locating
constexpr int SPEC_SUM_UNROLL = 8;                     // chunks a lane has in flight while summing
constexpr int SPEC_CH = 512;                           // values per bulk copy chunk
constexpr int SPEC_NS = 3;                             // chunks in flight per warp (bulk variant)
constexpr uint32_t SPEC_STAGE_BYTES = 2 * SPEC_CH * 4; // p then q
constexpr uint32_t SPEC_RING_BYTES = SPEC_WARPS * SPEC_NS * SPEC_STAGE_BYTES;
constexpr size_t SPEC_SMEM = SPEC_RING_BYTES + SPEC_WARPS * SPEC_NS * 8;
constexpr uint64_t SPEC_WAIT_NS = 2000000000ull;       // limit of one wait on a copy

struct DSum {
    float hi, lo;
};

// Knuth's two-sum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ DSum ds_add(DSum a, DSum b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, e);                  // Dekker's fast two-sum (|s| >= |e|)
    return DSum{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

// a > b for normalised pairs (|lo| at most half an ulp of hi, as ds_add leaves them).
__device__ __forceinline__ bool ds_gt(DSum a, DSum b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

// v * t as a normalised pair: the fma gives the exact error of v * t.hi.
__device__ __forceinline__ DSum ds_scale(float v, DSum t) {
    const float p = __fmul_rn(v, t.hi);
    const float lo = __fmaf_rn(v, t.lo, __fmaf_rn(v, t.hi, -p));
    const float hi = __fadd_rn(p, lo);
    return DSum{hi, __fsub_rn(lo, __fsub_rn(hi, p))};
}

// Weight of one vocabulary entry: max(0, p - q) (residual) or max(0, p), exactly as a pair. For the
// residual, d = p - q rounded and e = (p - d) - q is Dekker's fast two-sum, exact whenever p >= q >= 0,
// which covers every entry whose weight is kept.
__device__ __forceinline__ DSum weight(float p, float q, bool residual) {
    if (!residual) return DSum{p > 0.f ? p : 0.f, 0.f};
    const float d = __fsub_rn(p, q);
    const float e = __fsub_rn(__fsub_rn(p, d), q);
    return d > 0.f ? DSum{d, e} : DSum{0.f, 0.f};
}

// acc += weight(p, q), the weight's pair folded into the compensated sum.
template <bool RES>
__device__ __forceinline__ void accumulate(DSum &acc, float p, float q) {
    float hi, lo = 0.f;
    if constexpr (RES) {
        const float d = __fsub_rn(p, q);
        const float e = __fsub_rn(__fsub_rn(p, d), q);
        const bool pos = d > 0.f;
        hi = pos ? d : 0.f;
        lo = pos ? e : 0.f;
    } else {
        hi = fmaxf(p, 0.f);
    }
    float s, t;
    two_sum(acc.hi, hi, s, t);
    acc.hi = s;
    acc.lo = __fadd_rn(acc.lo, RES ? __fadd_rn(t, lo) : t);
}

template <bool RES>
__device__ __forceinline__ void accumulate4(DSum &acc, const float4 &a, const float4 &c) {
    accumulate<RES>(acc, a.x, c.x);
    accumulate<RES>(acc, a.y, c.y);
    accumulate<RES>(acc, a.z, c.z);
    accumulate<RES>(acc, a.w, c.w);
}

__device__ __forceinline__ DSum shfl_ds(DSum a, int src) {
    return DSum{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
__device__ __forceinline__ DSum shfl_up_ds(DSum a, int d) {
    return DSum{__shfl_up_sync(0xffffffffu, a.hi, d), __shfl_up_sync(0xffffffffu, a.lo, d)};
}
__device__ __forceinline__ DSum shfl_xor_ds(DSum a, int m) {
    return DSum{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}

// Inclusive and exclusive ordered scans of one DSum per lane.
__device__ __forceinline__ void warp_scan(DSum x, int lane, DSum &incl, DSum &excl) {
    incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const DSum up = shfl_up_ds(incl, d);
        if (lane >= d) incl = ds_add(up, incl);
    }
    excl = shfl_up_ds(incl, 1);
    if (lane == 0) excl = DSum{0.f, 0.f};
}

struct SpecRow {
    const float *p, *q;                                // q is read only for the residual
    bool residual, vec;
};

// The four values of one lane at [i, i + 4), zero at or past `end`.
__device__ __forceinline__ void load4(const SpecRow &r, int64_t i, int64_t end, float4 &a, float4 &c) {
    if (r.vec && i + 4 <= end) {
        a = __ldg(reinterpret_cast<const float4 *>(r.p + i));
        c = r.residual ? __ldg(reinterpret_cast<const float4 *>(r.q + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        float pa[4], qa[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pa[e] = i + e < end ? __ldg(r.p + i + e) : 0.f;
            qa[e] = r.residual && i + e < end ? __ldg(r.q + i + e) : 0.f;
        }
        a = make_float4(pa[0], pa[1], pa[2], pa[3]);
        c = make_float4(qa[0], qa[1], qa[2], qa[3]);
    }
}

// Level 1 from shared memory: each warp streams its span through a private ring of SPEC_NS stages
// filled by 1-D bulk copies (512 values of p, and of q for the residual, per stage). Returns false
// when a copy never completed within the limit (after waiting, bounded, for the copies in flight).
template <bool RES>
__device__ __forceinline__ bool segment_sums_bulk(const SpecRow &row, int64_t V, int64_t seg_len, uint8_t *ring_base,
                                                  uint32_t bars, uint32_t &issued_before, DSum *s_seg, int warp,
                                                  int lane) {
    const int nseg = (int)(seg_len / SPEC_CH);
    const int wch = SPEC_SEGS_WARP * nseg;
    const int64_t w0 = (int64_t)warp * SPEC_SEGS_WARP * seg_len;
    const int nv = w0 >= V ? 0 : (int)min((int64_t)wch, (V - w0 + SPEC_CH - 1) / SPEC_CH);
    const uint32_t ring = smem_u32(ring_base);
    const uint32_t g0 = issued_before;
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int c) {
        const int64_t start = w0 + (int64_t)c * SPEC_CH;
        const uint32_t n = (uint32_t)min((int64_t)SPEC_CH, V - start) * 4u;
        const uint32_t g = g0 + (uint32_t)c, st = g % SPEC_NS;
        const uint32_t bar = bars + st * 8, dst = ring + st * SPEC_STAGE_BYTES;
        mbar_arrive_expect_tx(bar, RES ? 2 * n : n);
        bulk_load(dst, row.p + start, n, bar, policy);
        if (RES) bulk_load(dst + SPEC_CH * 4, row.q + start, n, bar, policy);
    };
    if (lane == 0)
        for (int c = 0; c < nv && c < SPEC_NS; ++c) issue(c);
    issued_before = g0 + (uint32_t)nv;

    bool ok = true;
    int sg = warp * SPEC_SEGS_WARP;
    DSum acc{0.f, 0.f};
    for (int c = 0; c < wch; ++c) {
        if (c < nv && ok) {
            const uint32_t g = g0 + (uint32_t)c, st = g % SPEC_NS;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + st * 8, (g / SPEC_NS) & 1u, SPEC_WAIT_NS));
            if (ok) {
                const int nval = (int)min((int64_t)SPEC_CH, V - (w0 + (int64_t)c * SPEC_CH));
                const float *sp = reinterpret_cast<const float *>(ring_base + st * SPEC_STAGE_BYTES) + lane * 4;
                const float *sq = sp + SPEC_CH;
                float4 a[4], cq[4];
                if (nval == SPEC_CH) {                 // a whole chunk (all but a row's last)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        a[j] = *reinterpret_cast<const float4 *>(sp + j * 128);
                        if (RES) cq[j] = *reinterpret_cast<const float4 *>(sq + j * 128);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const bool in = j * 128 + lane * 4 < nval;
                        a[j] = in ? *reinterpret_cast<const float4 *>(sp + j * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
                        if (RES)
                            cq[j] = in ? *reinterpret_cast<const float4 *>(sq + j * 128)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                __syncwarp();                          // the stage is free: refill it
                if (lane == 0 && c + SPEC_NS < nv) {
                    fence_proxy_async_smem();
                    issue(c + SPEC_NS);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) accumulate4<RES>(acc, a[j], RES ? cq[j] : a[j]);
            } else if (lane == 0) {
                // wait (bounded) for this warp's copies still in flight before the ring is given up
                for (int k = c; k < nv && k < c + SPEC_NS; ++k)
                    mbar_wait_bounded(bars + ((g0 + k) % SPEC_NS) * 8, ((g0 + k) / SPEC_NS) & 1u, SPEC_WAIT_NS);
            }
        }
        if ((c + 1) % nseg == 0) {                     // the segment's last chunk
            acc = ds_add(acc, DSum{0.f, 0.f});
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) acc = ds_add(acc, shfl_xor_ds(acc, m));
            if (lane == 0) s_seg[sg] = acc;
            ++sg;
            acc = DSum{0.f, 0.f};
        }
    }
    return ok;
}

// Level 1 from registers (rows that are not 16-byte aligned): coalesced loads, eight chunks of 128
// values in flight per lane.
template <bool RES>
__device__ __forceinline__ void segment_sums_direct(const SpecRow &row, int64_t V, int64_t seg_len, DSum *s_seg,
                                                    int warp, int lane) {
    const int nch = (int)(seg_len / 128);
    const int wch = SPEC_SEGS_WARP * nch;
    const int64_t w0 = (int64_t)warp * SPEC_SEGS_WARP * seg_len;
    int sg = warp * SPEC_SEGS_WARP, left = nch;
    DSum acc{0.f, 0.f};
    for (int k = 0; k < wch; k += SPEC_SUM_UNROLL) {
        float4 a[SPEC_SUM_UNROLL], c[SPEC_SUM_UNROLL];
#pragma unroll
        for (int j = 0; j < SPEC_SUM_UNROLL; ++j)
            load4(row, w0 + (int64_t)(k + j) * 128 + lane * 4, k + j < wch ? V : 0, a[j], c[j]);
#pragma unroll
        for (int j = 0; j < SPEC_SUM_UNROLL; ++j) {
            if (k + j >= wch) break;
            accumulate4<RES>(acc, a[j], c[j]);
            if (--left == 0) {                         // the segment's last chunk
                acc = ds_add(acc, DSum{0.f, 0.f});
#pragma unroll
                for (int m = 16; m > 0; m >>= 1) acc = ds_add(acc, shfl_xor_ds(acc, m));
                if (lane == 0) s_seg[sg] = acc;
                ++sg;
                left = nch;
                acc = DSum{0.f, 0.f};
            }
        }
    }
}

template <bool kBulk>
__global__ void __launch_bounds__(SPEC_THREADS, 1) spec_verify_kernel(const float *p, const float *q,
                                                                    const int32_t *draft, const float *u,
                                                                    const float *v, int K, int64_t V, int32_t *out,
                                                                    int32_t *n_out, int *status) {
    extern __shared__ __align__(128) uint8_t spec_smem[];
    __shared__ DSum s_seg[SPEC_SEGS];
    __shared__ DSum s_before;
    __shared__ DSum s_target;
    __shared__ int s_rej, s_sel, s_abort;
    __shared__ DSum s_wsum[SPEC_WARPS], s_wpre[SPEC_WARPS], s_btotal;
    __shared__ int s_hit, s_last;
    const int64_t b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *o = out + b * (K + 1);
    const uint32_t bars = smem_u32(spec_smem + SPEC_RING_BYTES) + warp * SPEC_NS * 8;
    if (kBulk && lane == 0) {
        for (int st = 0; st < SPEC_NS; ++st) mbar_init(bars + st * 8, 1);
        fence_barrier_init();
    }
    if (tid == 0) s_abort = 0;

    const float vb = warp == 0 ? v[b] : 0.f;            // in flight during the accept tests
    if (warp == 0) {
        // accept tests, 32 drafts at a time; the first failure (or out-of-vocabulary draft) ends them
        int rej = K;
        for (int i0 = 0; i0 < K; i0 += 32) {
            const int i = i0 + lane;
            int32_t x = 0;
            bool inb = true, ok = false;
            if (i < K) {
                x = draft[b * K + i];
                inb = x >= 0 && x < V;
                if (inb) {
                    const float pi = p[(b * (K + 1) + i) * V + x];
                    const float qi = q[(b * K + i) * V + x];
                    ok = __fmul_rn(u[b * K + i], qi) < pi;
                }
            }
            const unsigned fail = __ballot_sync(0xffffffffu, i < K && !ok);
            const int first = fail ? i0 + __ffs(fail) - 1 : K;
            if (i < first) o[i] = x;
            if (i == first && !inb) set_status(status, STATUS_BOUNDS);
            if (fail) {
                rej = first;
                break;
            }
        }
        if (lane == 0) s_rej = rej;
    }
    __syncthreads();
    const int n_kept = s_rej;                          // == K when every draft is kept
    for (int i = n_kept + 1 + tid; i <= K; i += SPEC_THREADS) o[i] = -1;

    SpecRow row;
    row.p = p + (b * (K + 1) + n_kept) * V;
    row.q = n_kept < K ? q + (b * K + n_kept) * V : row.p;
    row.residual = n_kept < K;
    row.vec = kBulk;                                   // the bulk variant runs on 16-byte aligned rows only
    // segments: whole copy chunks (bulk) or whole 128-value chunks, 256 of them covering the row
    constexpr int64_t unit = kBulk ? SPEC_CH : 128;
    const int64_t seg_len = ((V + SPEC_SEGS - 1) / SPEC_SEGS + unit - 1) / unit * unit;
    uint32_t issued = 0;

    for (int pass = 0; pass < 2; ++pass) {
        // level 1: segment sums
        if constexpr (kBulk) {
            uint8_t *ring = spec_smem + warp * SPEC_NS * SPEC_STAGE_BYTES;
            const bool ok = row.residual ? segment_sums_bulk<true>(row, V, seg_len, ring, bars, issued, s_seg, warp, lane)
                                         : segment_sums_bulk<false>(row, V, seg_len, ring, bars, issued, s_seg, warp,
                                                                    lane);
            if (!ok && lane == 0) atomicExch(&s_abort, 1);
        } else if (row.residual) {
            segment_sums_direct<true>(row, V, seg_len, s_seg, warp, lane);
        } else {
            segment_sums_direct<false>(row, V, seg_len, s_seg, warp, lane);
        }
        __syncthreads();
        if (s_abort) {
            // a copy never completed: no token is drawn, and n_out = 0 reports it
            if (tid == 0) {
                o[n_kept] = -1;
                n_out[b] = 0;
            }
            return;
        }
        // level 2: the first segment whose running sum passes v * total
        if (warp == 0) {
            static_assert(SPEC_SEGS_LANE == 8, "level 2 sums a lane's segments as a tree of 8");
            DSum sv[SPEC_SEGS_LANE];
#pragma unroll
            for (int j = 0; j < SPEC_SEGS_LANE; ++j) sv[j] = s_seg[lane * SPEC_SEGS_LANE + j];
            const DSum mine = ds_add(ds_add(ds_add(sv[0], sv[1]), ds_add(sv[2], sv[3])),
                                     ds_add(ds_add(sv[4], sv[5]), ds_add(sv[6], sv[7])));
            DSum incl, excl;
            warp_scan(mine, lane, incl, excl);
            const DSum target = ds_scale(vb, shfl_ds(incl, 31));
            DSum c = excl, before{0.f, 0.f};
            int first = -1, last = -1;
#pragma unroll
            for (int j = 0; j < SPEC_SEGS_LANE; ++j) {
                const DSum nc = ds_add(c, sv[j]);
                if (sv[j].hi > 0.f) {
                    if (first < 0 && ds_gt(nc, target)) {
                        first = j;
                        before = c;
                    }
                    last = j;
                }
                c = nc;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, first >= 0);
            const unsigned any = __ballot_sync(0xffffffffu, last >= 0);
            if (hit) {
                // the token lies in this segment
                const int fl = __ffs(hit) - 1;
                if (lane == fl) {
                    s_sel = lane * SPEC_SEGS_LANE + first;
                    s_before = before;
                    s_target = target;
                }
            } else if (any) {
                // v * total rounded to (or above) the total: the last token of positive weight
                const int ll = 31 - __clz(any);
                if (lane == ll) {
                    s_sel = lane * SPEC_SEGS_LANE + last;
                    s_before = DSum{0.f, 0.f};
                    s_target = DSum{__int_as_float(0x7f800000), 0.f};  // +inf: nothing passes it
                }
            } else if (lane == 0) {
                s_sel = -1;                            // no mass at all
            }
        }
        __syncthreads();
        if (s_sel >= 0 || !row.residual) break;
        row.residual = false;                          // the residual has no mass: draw from p
        __syncthreads();
    }

    // level 3: the chosen segment, SPEC_THREADS values at a time, one per thread: a warp scan, a scan
    // of the warp sums, and the first value whose running sum passes the target (else, after rounding,
    // the segment's last value of positive weight)
    const int sel = s_sel;
    int tok = -1;
    if (sel >= 0) {
        const DSum target = s_target;
        const int64_t s0 = sel * seg_len;
        const int64_t s1 = s0 + seg_len < V ? s0 + seg_len : V;
        DSum before = s_before;
        if (tid == 0) {
            s_hit = 0x7fffffff;
            s_last = -1;
        }
        for (int64_t blk = s0; blk < s1; blk += SPEC_THREADS) {
            const int64_t i = blk + tid;
            const DSum w = i < s1 ? weight(__ldg(row.p + i), row.residual ? __ldg(row.q + i) : 0.f, row.residual)
                                  : DSum{0.f, 0.f};
            DSum incl, excl;
            warp_scan(w, lane, incl, excl);
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            if (warp == 0) {
                const DSum x = lane < SPEC_WARPS ? s_wsum[lane] : DSum{0.f, 0.f};
                DSum wi, we;
                warp_scan(x, lane, wi, we);
                if (lane < SPEC_WARPS) s_wpre[lane] = we;
                if (lane == SPEC_WARPS - 1) s_btotal = wi;
            }
            __syncthreads();
            const bool pos = w.hi > 0.f;
            const bool hit = pos && ds_gt(ds_add(ds_add(before, s_wpre[warp]), incl), target);
            const unsigned hb = __ballot_sync(0xffffffffu, hit), pb = __ballot_sync(0xffffffffu, pos);
            if (lane == 0) {
                if (hb) atomicMin(&s_hit, warp * 32 + __ffs(hb) - 1);
                if (pb) atomicMax(&s_last, (int)(blk - s0) + warp * 32 + 31 - __clz(pb));
            }
            __syncthreads();
            if (s_hit != 0x7fffffff) {
                tok = (int)(blk + s_hit);
                break;
            }
            before = ds_add(before, s_btotal);
            __syncthreads();                             // s_wsum, s_wpre, s_btotal are rewritten next
        }
        if (tok < 0 && s_last >= 0) tok = (int)(s0 + s_last);   // the running sums fell short by rounding
    }
    if (tid == 0) {
        o[n_kept] = tok;
        n_out[b] = n_kept + 1;
    }
}

cudaError_t launch_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                               int B, int K, int64_t V, int32_t *out, int32_t *n_out, int *status,
                               cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    const bool bulk = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(q)) & 15) == 0;
    if (!bulk) {
        spec_verify_kernel<false><<<B, SPEC_THREADS, 0, stream>>>(p, q, draft, u, v, K, V, out, n_out, status);
        return cudaGetLastError();
    }
    // set on every call: the attribute belongs to the current device, and callers may use several
    const cudaError_t e =
        cudaFuncSetAttribute(spec_verify_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SPEC_SMEM);
    if (e != cudaSuccess) return e;
    spec_verify_kernel<true><<<B, SPEC_THREADS, SPEC_SMEM, stream>>>(p, q, draft, u, v, K, V, out, n_out, status);
    return cudaGetLastError();
}

}  // namespace pa
