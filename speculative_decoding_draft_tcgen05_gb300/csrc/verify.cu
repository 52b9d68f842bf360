// Greedy accept check of a draft path against the target's argmax tokens.
//
// Blog "DFlash 2: Keep Drafting Parallel" (introduction): one pass of the
// target checks a whole drafted block, retaining the drafts it agrees with.
// Under greedy decoding those are the longest prefix of the path equal to the
// target's own argmax tokens, and the target adds one token of its own (its
// argmax after that prefix).
// One warp per sequence: lane t compares position t, a ballot finds the first
// mismatch.
#include <cooperative_groups.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

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
// Drafting Parallel", section "A Lightweight Path Selector": verified by
// rejection sampling, the output follows the target's distribution exactly).
// Draft token x_t is kept when u_acc_t < min(1, p_t(x_t) / q_t(x_t)), i.e.
// u_acc_t * q_t(x_t) < p_t(x_t) (a product of two floats, exact in double
// precision); at the first rejection the emitted token is drawn from the
// residual max(0, p_t - q_t) (q_t is zero off the K candidates), normalised,
// by inverting its CDF in vocabulary order with u_res; when all L drafts are
// kept the bonus token is drawn from p_L. A residual with no mass at all falls
// back to p_t itself.
//
// The draw reads one whole vocabulary row per sequence: a thread-block
// cluster of C CTAs per sequence shares it (C from 1 to 16, chosen by the
// number of sequences). Every CTA decides the L
// acceptances (a warp per position) and takes kRejWarps consecutive warp
// sub-slices of the row. Phase 1: each warp sums the masses of its sub-slice
// with coalesced loads, many in flight. Each CTA pushes its totals into every
// peer's shared memory, and after one cluster barrier each knows Z and which
// CTA holds u_res * Z. Phase 2 runs in that CTA only: its warp totals locate
// the warp whose sub-slice holds the target; the CTA's warps sum that
// sub-slice (now in L1/L2) a chunk of 32 consecutive tokens each, and a scan
// over the chunk sums and one inside the chunk holding the target find the
// token. At every level the owner is the last unit with mass whose exclusive
// start does not exceed the target, else the first unit with mass.
//
// Masses are summed in 64-bit fixed point: a probability becomes
// floor(p * 2^54), computed from its exponent and mantissa bits with integer
// instructions. Integer sums do not depend on their order, so both phases see
// the same running sums, and the CDF is exact to V * 2^-54 (8e-12 at a 150k
// vocabulary), far below the ~1e-5 CDF steps, where fp32 sums would not be.
// Double precision would also do, but it is the slowest arithmetic on this
// GPU. Probabilities must lie in [0, 1] and a row must sum to less than 1024.
namespace dfl {

namespace {

#ifndef DFL_REJ_THREADS
#define DFL_REJ_THREADS 1024
#endif
#ifndef DFL_REJ_BATCH
#define DFL_REJ_BATCH 16
#endif
constexpr int kRejThreads = DFL_REJ_THREADS;
constexpr int kRejWarps = kRejThreads / 32;
constexpr int kRejMaxCluster = 16;           // CTAs per sequence: 1 to 16, chosen per launch
constexpr int kRejBatch = DFL_REJ_BATCH;      // loads a lane keeps in flight (phase 1)
static_assert(kRejWarps <= 32, "one warp scans the warp totals");

// floor(x * 2^54) for 0 <= x < 2 (larger values saturate); zero for zero,
// subnormal, negative, infinite and NaN inputs.
__device__ __forceinline__ uint64_t fixed54(float x)
{
    const uint32_t b = __float_as_uint(x);
    const uint32_t ex = b >> 23;  // the sign bit pushes negatives above 255
    if (ex - 1u >= 254u) return 0;
    const uint32_t m = (b & 0x7FFFFFu) | 0x800000u;  // x = m * 2^(ex - 150)
    const int sh = static_cast<int>(ex < 127u ? ex : 127u) - 96;  // x * 2^54 = m * 2^(ex - 96)
    if (sh >= 0) return static_cast<uint64_t>(m) * (1u << sh);
    return m >> (-sh < 31 ? -sh : 31);
}

struct RejShared {
    unsigned long long warp_p[kRejWarps];   // mass of p_t over each warp's sub-slice
    unsigned long long warp_r[kRejWarps];   // mass of the residual over it
    unsigned long long tot_p[kRejMaxCluster];  // every CTA's totals, pushed by the CTAs
    unsigned long long tot_r[kRejMaxCluster];
    unsigned long long chunk[kRejWarps];    // phase 2: chunk sums
    unsigned long long warp_excl;           // phase 2: mass before the owner warp's sub-slice
    unsigned warp_cand[kRejWarps];          // candidates (bit j) inside each warp's sub-slice
    int32_t cand[16][32];                   // candidates of every position
    uint64_t qfx[16][32];                   // their draft probabilities, fixed point
    unsigned long long target;              // u_res * Z
    int keep[16];
    int owner_warp, use_r, done;
};

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += y;
    }
    return v;
}

// Residual mass of token y (fixed point pf): candidates (the set bits of
// `mask`, indices into cand/qfx of the rejected position) subtract their draft
// probability.
__device__ __forceinline__ uint64_t residual_mass(int64_t y, uint64_t pf, unsigned mask, const int32_t *cand,
                                                  const uint64_t *qfx)
{
    while (mask) {
        const int j = __ffs(mask) - 1;
        mask &= mask - 1;
        if (cand[j] == y) pf = pf > qfx[j] ? pf - qfx[j] : 0;
    }
    return pf;
}

// The owner among 32 units (lane = unit) given each unit's mass and exclusive
// start: the last unit with mass whose start is <= target, else the first
// unit with mass; -1 when no unit has mass.
__device__ __forceinline__ int owner_of(uint64_t mass, uint64_t excl, uint64_t target)
{
    const unsigned has = __ballot_sync(0xFFFFFFFFu, mass > 0);
    const unsigned below = __ballot_sync(0xFFFFFFFFu, mass > 0 && excl <= target);
    if (below) return 31 - __clz(below);
    return has ? __ffs(has) - 1 : -1;
}

// Phase 1 over the sub-slice [w0, w1): lane l reads the tokens w0 + 32 c + l
// (16-byte loads measured no faster here: a lane holds only a few tokens).
// kResidual: the warp holds candidates, whose residual differs from p_t.
template <bool kResidual>
__device__ __forceinline__ void slice_masses(const float *row, int64_t w0, int64_t w1, int lane, unsigned mask,
                                             const int32_t *cand, const uint64_t *qfx, uint64_t &sp, uint64_t &sr)
{
    const int64_t nchunks = (w1 - w0 + 31) / 32;
    for (int64_t c0 = 0; c0 < nchunks; c0 += kRejBatch) {
        float v[kRejBatch];
#pragma unroll
        for (int u = 0; u < kRejBatch; ++u) {
            const int64_t y = w0 + (c0 + u) * 32 + lane;
            v[u] = (y < w1) ? __ldg(row + y) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kRejBatch; ++u) {
            const uint64_t f = fixed54(v[u]);
            sp += f;
            if (kResidual) sr += residual_mass(w0 + (c0 + u) * 32 + lane, f, mask, cand, qfx);
        }
    }
    if (!kResidual) sr = sp;
}

__global__ void __launch_bounds__(kRejThreads) verify_rejection_kernel(
    const int32_t *__restrict__ path, const int32_t *__restrict__ ids, const float *__restrict__ q,
    const float *__restrict__ p, const float *__restrict__ u_acc, const float *__restrict__ u_res, int L, int K,
    int64_t V, int32_t *__restrict__ accept, int32_t *__restrict__ emitted)
{
    __shared__ RejShared s;
    pdl_wait();
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int C = static_cast<int>(cluster.num_blocks());
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *pb = path + static_cast<size_t>(b) * L;
    const int32_t *ib = ids + static_cast<size_t>(b) * L * K;
    const float *qb = q + static_cast<size_t>(b) * L * K;
    const float *prow0 = p + static_cast<size_t>(b) * (L + 1) * V;

    // the L acceptance decisions, a warp per position: candidates and draft
    // probabilities of position t are loaded coalesced and kept in shared
    // memory for the draw
    for (int t = warp; t < L; t += kRejWarps) {
        const int32_t x = __ldg(pb + t);
        const int32_t id = lane < K ? __ldg(ib + t * K + lane) : -1;
        const float qv = lane < K ? __ldg(qb + t * K + lane) : 0.f;
        const float ua = __ldg(u_acc + static_cast<size_t>(b) * L + t);
        const float px = (x >= 0 && x < V) ? __ldg(prow0 + static_cast<size_t>(t) * V + x) : 0.f;
        const unsigned match = __ballot_sync(0xFFFFFFFFu, lane < K && id == x);
        const float qx = match ? __shfl_sync(0xFFFFFFFFu, qv, 31 - __clz(match)) : 0.f;  // the last match counts
        s.cand[t][lane] = id;
        s.qfx[t][lane] = fixed54(qv);
        if (lane == 0) s.keep[t] = qx > 0.f && static_cast<double>(ua) * static_cast<double>(qx) < static_cast<double>(px);
    }
    __syncthreads();
    int n = L;
    for (int t = L - 1; t >= 0; --t)
        if (!s.keep[t]) n = t;
    const float *row = prow0 + static_cast<size_t>(n) * V;
    const int32_t *cand = s.cand[n < L ? n : 0];
    const uint64_t *qfx = s.qfx[n < L ? n : 0];

    // this warp's sub-slice [w0, w1): the row split into C * kRejWarps pieces
    // whose length is a multiple of 32 (whole 128-byte lines when the row
    // starts on one)
    const int64_t sub = ((V + C * kRejWarps - 1) / (C * kRejWarps) + 31) & ~int64_t(31);
    auto slice_of = [&](int w, int64_t &a, int64_t &e) {
        a = (static_cast<int64_t>(rank) * kRejWarps + w) * sub;
        e = (a + sub < V) ? a + sub : V;
        if (e < a) e = a;
    };
    int64_t w0, w1;
    slice_of(warp, w0, w1);
    unsigned mask;
    {
        bool in = false;
        if (lane < K && n < L) {  // the last occurrence of each candidate id counts
            const int32_t c = cand[lane];
            bool last = true;
            for (int j = lane + 1; j < K; ++j) last &= cand[j] != c;
            in = last && c >= w0 && c < w1;
        }
        mask = __ballot_sync(0xFFFFFFFFu, in);
    }

    // phase 1
    uint64_t sp = 0, sr = 0;
    if (mask)
        slice_masses<true>(row, w0, w1, lane, mask, cand, qfx, sp, sr);
    else
        slice_masses<false>(row, w0, w1, lane, mask, cand, qfx, sp, sr);
    sp = warp_sum_u64(sp);
    sr = warp_sum_u64(sr);
    if (lane == 0) {
        s.warp_p[warp] = sp;
        s.warp_r[warp] = sr;
        s.warp_cand[warp] = mask;
    }
    __syncthreads();
    if (warp == 0) {  // this CTA's totals, pushed into every CTA of the cluster
        const uint64_t cp = warp_sum_u64(lane < kRejWarps ? s.warp_p[lane] : 0ull);
        const uint64_t cr = warp_sum_u64(lane < kRejWarps ? s.warp_r[lane] : 0ull);
        if (lane < C) {
            RejShared *peer = cluster.map_shared_rank(&s, lane);
            peer->tot_p[rank] = cp;
            peer->tot_r[rank] = cr;
        }
    }
    cluster.sync();  // the only one: no CTA touches another's shared memory after it
    // the rows are read: the next kernel (the next lm_head pass) may be
    // scheduled without its early weight loads competing with those reads
    pdl_trigger();

    if (warp == 0) {  // every CTA: Z, the target and the CTA that holds it (the same arithmetic everywhere)
        const uint64_t mp = lane < C ? s.tot_p[lane] : 0ull;
        const uint64_t mr = lane < C ? s.tot_r[lane] : 0ull;
        const uint64_t ip = warp_incl_scan_u64(mp, lane), ir = warp_incl_scan_u64(mr, lane);
        const uint64_t zp = __shfl_sync(0xFFFFFFFFu, ip, 31), zr = __shfl_sync(0xFFFFFFFFu, ir, 31);
        const bool use_r = n < L && zr > 0;
        const uint64_t z = use_r ? zr : zp;
        const uint64_t target =
            static_cast<uint64_t>(static_cast<double>(z) * static_cast<double>(__ldg(u_res + b)));
        const uint64_t m = use_r ? mr : mp, e = (use_r ? ir : ip) - m;
        const int owner_rank = owner_of(m, e, target);
        const uint64_t cta_excl = __shfl_sync(0xFFFFFFFFu, e, rank);
        if (rank == 0) {  // everything but the drawn token
            const size_t eb = static_cast<size_t>(b) * (L + 1);
            if (lane <= L && lane != n) emitted[eb + lane] = lane < n ? __ldg(pb + lane) : -1;
            if (lane == 0 && owner_rank < 0) emitted[eb + n] = -1;  // no mass anywhere in the row
            if (lane == 0) accept[b] = n;
        }
        int ow = -1;
        if (rank == owner_rank) {  // the warp whose sub-slice holds the target
            const uint64_t wm = lane >= kRejWarps ? 0ull : use_r ? s.warp_r[lane] : s.warp_p[lane];
            const uint64_t we = cta_excl + warp_incl_scan_u64(wm, lane) - wm;
            ow = owner_of(wm, we, target);
            if (lane == ow) s.warp_excl = we;
        }
        if (lane == 0) {
            s.owner_warp = ow;
            s.use_r = use_r;
            s.target = target;
        }
    }
    __syncthreads();
    const int ow = s.owner_warp;
    if (ow < 0) return;  // not the owner CTA (uniform over the CTA)

    // phase 2: the owner warp's sub-slice, kRejWarps chunks of 32 tokens at a
    // time (a warp per chunk), then a scan over the chunk sums and one inside
    // the chunk that holds the target
    const uint64_t target = s.target;
    int64_t v0, v1;
    slice_of(ow, v0, v1);
    const unsigned wmask = s.use_r ? s.warp_cand[ow] : 0u;
    const int64_t nch = (v1 - v0 + 31) / 32;
    uint64_t base = s.warp_excl;  // warp 0's running start
    int64_t chosen = -1;
    for (int64_t g0 = 0; g0 < nch; g0 += kRejWarps) {
        const int64_t c = g0 + warp;
        uint64_t cs = 0;
        if (c < nch) {
            const int64_t y = v0 + c * 32 + lane;
            cs = warp_sum_u64(y < v1 ? residual_mass(y, fixed54(__ldg(row + y)), wmask, cand, qfx) : 0ull);
        }
        if (lane == 0) s.chunk[warp] = cs;
        __syncthreads();
        if (warp == 0) {
            const uint64_t ch = lane < kRejWarps ? s.chunk[lane] : 0ull;
            const uint64_t incl = warp_incl_scan_u64(ch, lane);
            const uint64_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            bool done = false;
            if (total > 0) {
                const int oc = owner_of(ch, base + incl - ch, target);
                const uint64_t cbase = base + __shfl_sync(0xFFFFFFFFu, incl - ch, oc);
                const int64_t y0 = v0 + (g0 + oc) * 32;
                const int64_t y = y0 + lane;
                const uint64_t m = y < v1 ? residual_mass(y, fixed54(__ldg(row + y)), wmask, cand, qfx) : 0ull;
                const int o = owner_of(m, cbase + warp_incl_scan_u64(m, lane) - m, target);
                if (base > target) {  // the target lies before this group's mass
                    if (chosen < 0) chosen = y0 + o;
                    done = true;
                } else {
                    chosen = y0 + o;
                    base += total;
                    done = base > target;
                }
            }
            if (lane == 0) s.done = done;
        }
        __syncthreads();
        if (s.done) break;
    }
    if (warp == 0 && lane == 0) emitted[static_cast<size_t>(b) * (L + 1) + n] = static_cast<int32_t>(chosen);
}

}  // namespace

cudaError_t launch_verify_rejection(const int32_t *path, const int32_t *ids, const float *q, const float *p,
                                    const float *u_acc, const float *u_res, int B, int L, int K, int64_t V,
                                    int32_t *accept, int32_t *emitted, cudaStream_t s)
{
    // per device, once: the SM count, the shared memory that keeps one CTA per
    // SM, and the opt-ins to clusters of 16 and to that much shared memory
    static std::atomic<int> sms_of[64], spread_of[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = (dev >= 0 && dev < 64) ? sms_of[dev].load(std::memory_order_acquire) : 0;
    int spread = (sms != 0) ? spread_of[dev].load(std::memory_order_relaxed) : 0;
    if (sms == 0) {
        int per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(verify_rejection_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        spread = static_cast<int>(ctas_per_sm_smem(static_cast<size_t>(per_sm), 1));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(verify_rejection_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, spread);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) {
            spread_of[dev].store(spread, std::memory_order_relaxed);
            sms_of[dev].store(sms, std::memory_order_release);  // publishes spread
        }
    }
#ifndef DFL_REJ_FIXED_C
    // CTAs per sequence: 16 for up to 4 sequences (clusters of 16 need a whole
    // GPC each), else as many as keep all sequences in one wave of one CTA per SM
    int C = B <= 4 ? kRejMaxCluster : 8;
    while (C > 1 && static_cast<int64_t>(C) * B > sms) C >>= 1;
#else
    const int C = DFL_REJ_FIXED_C;
#endif
    // While all CTAs fit one per SM, reserved (unused) shared memory keeps two of
    // these 1024-thread CTAs from sharing an SM when the kernel is scheduled
    // early, beside its predecessor's last CTAs.
    const size_t smem = (static_cast<int64_t>(C) * B <= sms) ? static_cast<size_t>(spread) : 0;
    return launch_ex(verify_rejection_kernel, dim3(B, 1, C), dim3(kRejThreads), smem, s, C, path, ids, q, p, u_acc,
                     u_res, L, K, V, accept, emitted);
}

}  // namespace dfl
