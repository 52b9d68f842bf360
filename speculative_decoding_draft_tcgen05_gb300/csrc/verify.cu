// Greedy accept check of a draft path against the target's argmax tokens.
//
// Blog "DFlash 2: Keep Drafting Parallel" (introduction): the target model
// verifies the whole drafted block in one forward pass; good guesses are kept
// and bad ones thrown away. With greedy decoding the kept guesses are the
// longest prefix of the path that equals the target's own argmax tokens, and
// the target contributes one more token (its argmax after that prefix).
// One warp per sequence: lane t compares position t, a ballot finds the first
// mismatch.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

__global__ void __launch_bounds__(256) verify_kernel(const int32_t *__restrict__ path,
                                                     const int32_t *__restrict__ target, int B, int L,
                                                     int32_t *__restrict__ accept, int32_t *__restrict__ emitted)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t *pb = path + static_cast<size_t>(b) * L;
    const int32_t *tb = target + static_cast<size_t>(b) * (L + 1);
    const int32_t pt = lane < L ? pb[lane] : 0;
    const int32_t tt = lane <= L ? tb[lane] : 0;
    const unsigned in_block = (L >= 32) ? 0xFFFFFFFFu : ((1u << L) - 1u);
    const unsigned mismatch = ~__ballot_sync(0xFFFFFFFFu, lane < L && pt == tt) & in_block;
    const int n = mismatch ? __ffs(mismatch) - 1 : L;
    if (lane == 0) accept[b] = n;
    if (emitted && lane <= L) emitted[static_cast<size_t>(b) * (L + 1) + lane] = lane < n ? pt : (lane == n ? tt : -1);
}

}  // namespace

cudaError_t launch_verify(const int32_t *path, const int32_t *target, int B, int L, int32_t *accept,
                          int32_t *emitted, cudaStream_t s)
{
    const int per_cta = 8;
    return launch_ex(verify_kernel, dim3((B + per_cta - 1) / per_cta), dim3(per_cta * 32), 0, s, 1, path, target, B,
                     L, accept, emitted);
}

}  // namespace dfl

// Rejection-sampling verification of a sampled draft (blog "DFlash 2: Keep
// Drafting Parallel", section "A Lightweight Path Selector": rejection
// sampling restores the exact target distribution). Draft token x_t is kept
// when u_acc_t < min(1, p_t(x_t) / q_t(x_t)); at the first rejection the
// emitted token is drawn from the residual max(0, p_t - q_t) (q_t is zero off
// the K candidates), normalised, by inverting its CDF in vocabulary order
// with u_res; when all L drafts are kept the bonus token is drawn from p_L.
// One CTA of 1024 threads per sequence: lanes decide the L acceptances in
// parallel, then each thread sums a contiguous slice of the vocabulary, a
// block scan locates the slice holding u_res * Z, and its owner walks it.
// The ratio and the residual's running sums are taken in double precision, so
// each decision matches an exact computation unless the uniform lies within
// about 1e-12 of a boundary (the CDF steps of a 150k-token vocabulary are
// ~1e-5, as small as fp32 summation error).
namespace dfl {

namespace {

constexpr int kRejThreads = 1024;

__global__ void __launch_bounds__(kRejThreads) verify_rejection_kernel(
    const int32_t *__restrict__ path, const int32_t *__restrict__ ids, const float *__restrict__ q,
    const float *__restrict__ p, const float *__restrict__ u_acc, const float *__restrict__ u_res, int L, int K,
    int64_t V, int32_t *__restrict__ accept, int32_t *__restrict__ emitted)
{
    __shared__ int s_n;
    __shared__ int32_t s_cand[32];
    __shared__ float s_q[32];
    __shared__ double s_warp[32];
    __shared__ int s_owner;
    __shared__ int32_t s_draw;
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *pb = path + static_cast<size_t>(b) * L;
    const int32_t *ib = ids + static_cast<size_t>(b) * L * K;
    const float *qb = q + static_cast<size_t>(b) * L * K;
    const float *prow0 = p + static_cast<size_t>(b) * (L + 1) * V;

    if (warp == 0) {
        bool keep = false;
        if (lane < L) {
            const int32_t x = pb[lane];
            float qx = 0.f;
            for (int j = 0; j < K; ++j)
                if (__ldg(ib + lane * K + j) == x) qx = __ldg(qb + lane * K + j);
            const double px = (x >= 0 && x < V) ? __ldg(prow0 + static_cast<size_t>(lane) * V + x) : 0.0;
            const double a = (qx > 0.f) ? fmin(1.0, px / static_cast<double>(qx)) : 0.0;
            keep = static_cast<double>(__ldg(u_acc + static_cast<size_t>(b) * L + lane)) < a;
        }
        const unsigned rejected = ~__ballot_sync(0xFFFFFFFFu, keep) & ((L >= 32) ? 0xFFFFFFFFu : ((1u << L) - 1u));
        const int n = rejected ? __ffs(rejected) - 1 : L;
        if (lane == 0) s_n = n;
        if (n < L && lane < K) {
            s_cand[lane] = __ldg(ib + n * K + lane);
            s_q[lane] = __ldg(qb + n * K + lane);
        }
    }
    __syncthreads();
    const int n = s_n;
    const bool residual = n < L;
    const float *row = prow0 + static_cast<size_t>(n) * V;

    // this thread's slice of the vocabulary and its mass
    const int64_t chunk = (V + kRejThreads - 1) / kRejThreads;
    const int64_t y0 = tid * chunk, y1 = (y0 + chunk < V) ? y0 + chunk : V;
    auto mass = [&](int64_t y, double py) -> double {
        if (residual)
            for (int j = 0; j < K; ++j)
                if (s_cand[j] == y) return fmax(0.0, py - static_cast<double>(s_q[j]));
        return py;
    };
    double part = 0.0;
    for (int64_t y = y0; y < y1; ++y) part += mass(y, __ldg(row + y));
    // block-wide exclusive scan of the slice masses
    double incl = part;
    for (int off = 1; off < 32; off <<= 1) {
        const double v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    if (tid == 0) s_owner = -1;
    __syncthreads();
    if (warp == 0) {
        double w = s_warp[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const double v = __shfl_up_sync(0xFFFFFFFFu, w, off);
            if (lane >= off) w += v;
        }
        s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const double Z = s_warp[31];
    const double excl = incl - part + (warp > 0 ? s_warp[warp - 1] : 0.0);
    const double target = static_cast<double>(__ldg(u_res + b)) * Z;
    if (part > 0.0 && target >= excl && target < excl + part) s_owner = tid;
    __syncthreads();
    if (s_owner < 0) {  // target at the very top (rounding): the last slice with mass owns it
        const unsigned has = __ballot_sync(0xFFFFFFFFu, part > 0.0);
        if (lane == 0 && has) atomicMax(&s_owner, warp * 32 + 31 - __clz(has));
        __syncthreads();
    }
    if (tid == s_owner) {
        double c = excl;
        int32_t draw = -1, last = -1;
        for (int64_t y = y0; y < y1; ++y) {
            const double m = mass(y, __ldg(row + y));
            if (m <= 0.0) continue;
            last = static_cast<int32_t>(y);
            c += m;
            if (c > target) {
                draw = static_cast<int32_t>(y);
                break;
            }
        }
        s_draw = draw >= 0 ? draw : last;
    }
    __syncthreads();
    if (tid <= L) {
        int32_t e = -1;
        if (tid < n)
            e = pb[tid];
        else if (tid == n)
            e = s_owner >= 0 ? s_draw : -1;
        emitted[static_cast<size_t>(b) * (L + 1) + tid] = e;
    }
    if (tid == 0) accept[b] = n;
}

}  // namespace

cudaError_t launch_verify_rejection(const int32_t *path, const int32_t *ids, const float *q, const float *p,
                                    const float *u_acc, const float *u_res, int B, int L, int K, int64_t V,
                                    int32_t *accept, int32_t *emitted, cudaStream_t s)
{
    return launch_ex(verify_rejection_kernel, dim3(B), dim3(kRejThreads), 0, s, 1, path, ids, q, p, u_acc, u_res,
                     L, K, V, accept, emitted);
}

}  // namespace dfl
