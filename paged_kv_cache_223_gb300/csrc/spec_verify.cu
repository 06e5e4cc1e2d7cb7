// spec_verify.cu -- speculative rejection sampling after the target's one-pass verify of K
// draft tokens (yangyu.win blog #54, section 5 question 3; maths.nthquan ch. 17 "Speculative
// decoding", algorithm steps 3-4): draft x_i is kept with probability min(1, p_i(x_i) / q_i(x_i));
// the first rejected position is resampled from max(0, p_i - q_i) renormalised and later drafts
// are dropped; when every draft is kept, one more token is drawn from p_K.
//
// One CTA per sequence. Thread 0 runs the K accept tests (fp32: u * q < p). The draw is an inverse
// CDF over the vocabulary: each thread sums a contiguous chunk in fp64, a block scan of the chunk
// sums locates the chunk where the running sum first exceeds v * total, and that thread walks its
// chunk. Reads: K (p, q) pairs and one or two rows of V floats per sequence.
#include <cub/block/block_scan.cuh>

#include "pa_device.cuh"

namespace pa {

constexpr int SPEC_THREADS = 256;

__global__ void __launch_bounds__(SPEC_THREADS) spec_verify_kernel(const float *p, const float *q,
                                                                    const int32_t *draft, const float *u,
                                                                    const float *v, int K, int64_t V, int32_t *out,
                                                                    int32_t *n_out, int *status) {
    using Scan = cub::BlockScan<double, SPEC_THREADS>;
    __shared__ typename Scan::TempStorage scan_tmp;
    __shared__ int s_rej, s_tok;
    __shared__ double s_total;
    const int64_t b = blockIdx.x;
    const int tid = threadIdx.x;
    int32_t *o = out + b * (K + 1);

    if (tid == 0) {
        int rej = -1;
        for (int i = 0; i < K; ++i) {
            int32_t x = draft[b * K + i];
            if (x < 0 || x >= V) {                       // outside the vocabulary: flag and reject here
                set_status(status, STATUS_BOUNDS);
                rej = i;
                break;
            }
            const float pi = p[(b * (K + 1) + i) * V + x];
            const float qi = q[(b * K + i) * V + x];
            if (__fmul_rn(u[b * K + i], qi) < pi) {
                o[i] = x;
            } else {
                rej = i;
                break;
            }
        }
        s_rej = rej;
        s_tok = -1;
    }
    __syncthreads();
    const int rej = s_rej;
    const int n_kept = rej >= 0 ? rej : K;
    for (int i = n_kept + 1 + tid; i <= K; i += SPEC_THREADS) o[i] = -1;

    const float *pr = p + (b * (K + 1) + (rej >= 0 ? rej : K)) * V;
    const float *qr = rej >= 0 ? q + (b * K + rej) * V : nullptr;
    const int64_t chunk = (V + SPEC_THREADS - 1) / SPEC_THREADS;
    const int64_t t0 = tid * chunk < V ? tid * chunk : V;
    const int64_t t1 = t0 + chunk < V ? t0 + chunk : V;
    // weight of token t: the residual max(0, p - q) after a rejection, else max(0, p)
    auto weight = [&](int64_t t, bool residual) -> double {
        return residual ? fmax((double)pr[t] - (double)qr[t], 0.0) : fmax((double)pr[t], 0.0);
    };
    bool residual = qr != nullptr;
    double local = 0.0, before = 0.0, total = 0.0;
    for (int pass = 0; pass < 2; ++pass) {
        local = 0.0;
        for (int64_t t = t0; t < t1; ++t) local += weight(t, residual);
        Scan(scan_tmp).ExclusiveSum(local, before, total);
        if (tid == 0) s_total = total;
        __syncthreads();
        total = s_total;
        __syncthreads();
        if (total > 0.0 || !residual) break;
        residual = false;                                // the residual has no mass: draw from p
    }
    if (tid == 0) s_tok = 0x7fffffff;
    __syncthreads();
    const double target = (double)v[b] * total;
    if (total > 0.0 && local > 0.0 && before <= target && before + local > target) {
        double c = before;
        for (int64_t t = t0; t < t1; ++t) {
            c += weight(t, residual);
            if (c > target) {
                atomicMin(&s_tok, (int)t);
                break;
            }
        }
    }
    __syncthreads();
    if (tid == 0 && s_tok == 0x7fffffff) {
        // rounding left the target between two chunks' sums: walk the whole row in order
        double c = 0.0;
        int tok = -1;
        for (int64_t t = 0; t < V && tok < 0; ++t) {
            c += weight(t, residual);
            if (c > target) tok = (int)t;
        }
        for (int64_t t = V - 1; t >= 0 && tok < 0; --t)  // v * total rounded up to the total
            if (weight(t, residual) > 0.0) tok = (int)t;
        s_tok = tok;
    }
    __syncthreads();
    if (tid == 0) {
        o[n_kept] = s_tok;
        n_out[b] = n_kept + 1;
    }
}

cudaError_t launch_spec_verify(const float *p, const float *q, const int32_t *draft, const float *u, const float *v,
                               int B, int K, int64_t V, int32_t *out, int32_t *n_out, int *status,
                               cudaStream_t stream) {
    if (B == 0) return cudaSuccess;
    spec_verify_kernel<<<B, SPEC_THREADS, 0, stream>>>(p, q, draft, u, v, K, V, out, n_out, status);
    return cudaGetLastError();
}

}  // namespace pa
