// Two-tap dynamic depthwise convolution of the DFlash 2 drafter.
//
// Blog "DFlash 2: Keep Drafting Parallel", section "A Lightweight Local
// Convolution": Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}, each
// coefficient a base kernel plus a correction computed from the current
// hidden state, one correction per 16 channels; block-local and stateless.
// With the correction a linear map, corr_t = Wc x_t ([d/8] values: two taps
// of d/16 groups), the operation is a small GEMM followed by an elementwise
// epilogue:
//   1. corr = X Wc^T  ([P, d] x [d, d/8], P = B * S rows): tcgen05 with the
//      "swap-AB" tiling of the lm_head kernel -- 128 rows of Wc (64 groups,
//      both taps interleaved) are the MMA's M, NT rows of X are N, d is
//      streamed 64 columns per stage by TMA into 128-byte-swizzled shared
//      memory. Small P splits d over a thread-block cluster of up to 8 CTAs:
//      each sends the partial sums of every CTA's share of the rows to that
//      CTA by a bulk shared-to-shared copy (counted on the receiver's
//      mbarrier), and each sums its ks partials in rank order.
//   2. Y[p, c] = (base0[c] + corr[p, 2g]) X[p, c] + (base1[c] + corr[p, 2g+1]) X[p-1, c]
//      (g = c / 16; X[p-1] = 0 at a block's first row): two threads per
//      (row, group), 8 channels each, 16-byte loads and stores, so a warp
//      reads and writes 512 contiguous bytes of a row.
// With at most 8 rows (one block) corr is a matrix-vector product bound by the
// Wc read, and conv2_small_kernel does it on CUDA cores instead (see there).
// Warp roles of conv2_kernel: warp 0 lane 0 issues TMA copies, warp 1 lane 0 owns TMEM and
// issues the MMAs, warps 0-3 move the accumulator from TMEM to shared memory,
// and all 8 warps run the epilogue. Every pipeline wait is bounded.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <cstdio>

#include "common.cuh"
#include "dflash_conv2.h"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dfl {
dflash_status host_fail(dflash_status st, const char *msg);
dflash_status host_make_tmap(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, int box_rows);
}  // namespace dfl

namespace dfl {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTileM = 128;                                  // Wc rows per tile: 64 groups x 2 taps
constexpr uint32_t kConvABytes = kConvTileM * kLmTileK * 2;      // 16 KB of Wc per stage
constexpr int kConvMaxStages = 8;
constexpr int kConvMaxSplit = 8;
constexpr int kConvEpiBatch = 8;  // X rows a thread keeps in flight in the epilogue

struct ConvParams {
    CUtensorMap tm_wc;  // [d/8, d], box 128 x 64
    CUtensorMap tm_x;   // [P, d], box NT x 64
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *base;  // [2, d]
    __nv_bfloat16 *y;
    int P, S, d, rows;  // rows = d / 8
    int NT, ksplit, stages;
    int *err;
};

struct ConvLayout {
    uint32_t stage_bytes, ring_bytes, red_bytes, off_bar, total;
};

__host__ __device__ inline ConvLayout conv_layout(int NT, int ksplit, int stages)
{
    ConvLayout l;
    l.stage_bytes = kConvABytes + static_cast<uint32_t>(NT) * kLmTileK * 2;
    const uint32_t ring = static_cast<uint32_t>(stages) * l.stage_bytes;
    const uint32_t dump = static_cast<uint32_t>(kConvTileM) * (NT + 1) * 4;  // fp32 accumulator, padded rows
    l.ring_bytes = ring > dump ? ring : dump;
    l.red_bytes = ksplit > 1 ? static_cast<uint32_t>(kConvTileM) * NT * 4 : 0;  // ksplit slots of 128/ksplit rows
    l.off_bar = (l.ring_bytes + l.red_bytes + 7u) & ~7u;
    // full[S], empty[S], done, red, then the TMEM base and the abort flag
    l.total = l.off_bar + 8u * (2u * stages + 2u) + 8u;
    return l;
}

__host__ __device__ inline uint32_t conv_tmem_cols(int NT)
{
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(NT)) c <<= 1;
    return c;
}

// Split cluster barrier (all threads of every CTA take part): arrive
// (relaxed: no memory ordering), later wait for the other CTAs' arrivals.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// The shared::cluster address of `addr` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to a
// CTA of the cluster, counted in bytes on that CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// Orders this thread's shared-memory writes before later async-proxy (bulk
// copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__global__ void __launch_bounds__(kConvThreads, 1) conv2_kernel(const __grid_constant__ ConvParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzled tiles need 1024 B alignment
    uint8_t *const gbase = smem_raw + (base - raw);

    const int NT = p.NT, S = p.stages, ks = p.ksplit;
    const ConvLayout lay = conv_layout(NT, ks, S);
    float *const acc = reinterpret_cast<float *>(gbase);  // reuses the ring after the K loop (no split)
    // with a split d: the partial sums of this CTA's rows from every CTA of the
    // cluster, written by them (a region of its own: they may write while this
    // CTA is still in its K loop)
    float *const red = reinterpret_cast<float *>(gbase + lay.ring_bytes);
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_empty = bar_full + 8u * S;
    const uint32_t bar_done = bar_empty + 8u * S;
    const uint32_t bar_red = bar_done + 8u;  // the partial sums of the cluster have arrived
    uint32_t *const tmem_holder = reinterpret_cast<uint32_t *>(gbase + lay.off_bar + 8u * (2u * S + 2u));
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x, n_tile = blockIdx.y;
    cg::cluster_group cluster = cg::this_cluster();
    const int z = static_cast<int>(cluster.block_rank());  // d-slice of this CTA (0 without a cluster)
    const int KBc = p.d / kLmTileK / ks;
    const int kb0 = z * KBc;
    const uint32_t tmem_cols = conv_tmem_cols(NT);
    // row stride of the accumulator copies: padded against bank conflicts, or
    // dense with a split d (a CTA's rows for one owner are then one block)
    const int ld = ks > 1 ? NT : NT + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_red, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // the cluster's partial sums of this CTA's rows, announced before any
        // CTA can send them (they send after the cluster barrier below)
        if (ks > 1) mbar_arrive_expect_tx(bar_red, static_cast<uint32_t>(kConvTileM) * NT * 4);
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_wc);
        tma_prefetch_desc(&p.tm_x);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(tmem_holder), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (ks > 1) cluster_arrive_relaxed();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    // The weights may be read before the previous kernel on the stream ends;
    // X (its output, typically) and Y only after it.
    pdl_trigger();
    if (!(warp == 0 && lane == 0)) pdl_wait();

    bool timed_out = false;
    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t pol_w = l2_policy_evict_normal();  // shared by the CTAs of other row tiles
        const uint64_t pol_x = l2_policy_evict_last();    // read again by the epilogue
        const int pre = KBc < S ? KBc : S;
        for (int it = 0; it < pre; ++it) {
            mbar_arrive_expect_tx(bar_full + 8u * it, lay.stage_bytes);
            tma_load_2d(base + it * lay.stage_bytes, &p.tm_wc, (kb0 + it) * kLmTileK, m_tile * kConvTileM,
                        bar_full + 8u * it, pol_w);
        }
        pdl_wait();
        for (int it = 0; it < pre; ++it)
            tma_load_2d(base + it * lay.stage_bytes + kConvABytes, &p.tm_x, (kb0 + it) * kLmTileK, n_tile * NT,
                        bar_full + 8u * it, pol_x);
        int it = pre;
        for (; it < KBc; ++it) {
            const int s = it % S;
            const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
            if (!mbar_wait(bar_empty + 8u * s, ph ^ 1u, abort_flag)) {
                timed_out = true;
                break;
            }
            const uint32_t sa = base + s * lay.stage_bytes;
            mbar_arrive_expect_tx(bar_full + 8u * s, lay.stage_bytes);
            tma_load_2d(sa, &p.tm_wc, (kb0 + it) * kLmTileK, m_tile * kConvTileM, bar_full + 8u * s, pol_w);
            tma_load_2d(sa + kConvABytes, &p.tm_x, (kb0 + it) * kLmTileK, n_tile * NT, bar_full + 8u * s, pol_x);
        }
        if (timed_out)  // let the copies already issued land before the CTA can exit
            for (int j = (it > S ? it - S : 0); j < it; ++j)
                mbar_wait(bar_full + 8u * (j % S), static_cast<uint32_t>(j / S) & 1u, abort_flag, false);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_bf16_f32(kConvTileM, NT);
        for (int it = 0; it < KBc; ++it) {
            const int s = it % S;
            if (!mbar_wait(bar_full + 8u * s, static_cast<uint32_t>(it / S) & 1u, abort_flag)) {
                timed_out = true;
                break;
            }
            tc_fence_after_sync();
            const uint32_t sa = base + s * lay.stage_bytes;
#pragma unroll
            for (int k = 0; k < kLmTileK / 16; ++k)
                umma_bf16(tmem_base, smem_desc_sw128(sa + 32u * k), smem_desc_sw128(sa + kConvABytes + 32u * k), idesc,
                          (it > 0 || k > 0) ? 1u : 0u);
            umma_commit(bar_empty + 8u * s);  // frees the stage once these MMAs have read it
        }
        umma_commit(bar_done);  // also after a timeout: every issued MMA must finish before TMEM is freed
    }
    __syncwarp();

    // ---------------------------------------------------- epilogue operands
    // Thread -> (channel group gl, half h) of this CTA's rows, and a run of Q
    // consecutive positions; 2 * ng threads cover one position row, so a warp
    // reads and writes contiguous bytes. The base kernels and the first batch
    // of X rows are loaded before the accumulator is ready.
    const int nr = kConvTileM / ks;                     // accumulator rows this CTA finishes
    const int r0 = z * nr;
    const int ng = nr / 2;                              // channel groups of this CTA
    const int per_pos = 2 * ng;                         // threads per position row (16 .. 128)
    const int Q = NT / (kConvThreads / per_pos);        // positions per thread
    const int gl = (threadIdx.x % per_pos) >> 1, h = threadIdx.x & 1;
    const int g = m_tile * (kConvTileM / 2) + r0 / 2 + gl;
    const bool gok = g < p.rows / 2;
    const int nb = (threadIdx.x / per_pos) * Q;         // first position of the run (tile-local)
    const size_t ch = static_cast<size_t>(gok ? g : 0) * 16 + 8 * h;
    float b0[8], b1[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(p.base + ch)), b0);
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(p.base + p.d + ch)), b1);
    uint4 xv[kConvEpiBatch], pv = make_uint4(0u, 0u, 0u, 0u);
    auto load_batch = [&](int j0) {
#pragma unroll
        for (int j = 0; j < kConvEpiBatch; ++j) {
            const int pos = n_tile * NT + nb + j0 + j;
            xv[j] = (gok && j0 + j < Q && pos < p.P)
                        ? *reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(pos) * p.d + ch)
                        : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    {
        const int pos = n_tile * NT + nb;
        if (gok && pos < p.P && pos % p.S != 0)
            pv = *reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(pos - 1) * p.d + ch);
        load_batch(0);
    }

    // ---------------------------------------------------- accumulator -> shared memory
    // Only the time bound ends this wait: the MMAs in flight must be drained.
    if (!mbar_wait(bar_done, 0, abort_flag, false)) timed_out = true;
    tc_fence_after_sync();
    if (warp < 4) {  // warp w may read TMEM lanes 32w .. 32w+31 (= Wc rows of the tile)
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        float *const dst = acc + (warp * 32 + lane) * ld;
        for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
            __syncwarp();
            tmem_load16(taddr + static_cast<uint32_t>(c0), v);
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[c0 + j] = v[j];
        }
        if (ks > 1) fence_proxy_async_smem();  // the bulk copies below read these rows
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    if (ks > 1) {
        // Split d: rows [q nr, (q+1) nr) of this CTA's partial sums go to CTA q,
        // slot z, by one bulk copy each; every CTA then waits for its own ks
        // slots. The split barrier makes sure all CTAs run (and have announced
        // their byte counts) before the first copy.
        cluster_wait();
        if (threadIdx.x == 0) {
            const uint32_t blk = static_cast<uint32_t>(nr) * NT * 4;
            for (int q = 0; q < ks; ++q)
                bulk_copy_to_cluster(mapa_shared(smem_u32(red) + static_cast<uint32_t>(z) * blk, q),
                                     smem_u32(acc) + static_cast<uint32_t>(q) * blk, blk, mapa_shared(bar_red, q));
        }
        if (!mbar_wait(bar_red, 0, abort_flag, false)) timed_out = true;
        // arrive once this CTA holds everything it was sent; the wait at the
        // end keeps every CTA (the source of its copies) alive until all have
        cluster_arrive_relaxed();
    }

    // ---------------------------------------------------- epilogue
    // corr of row pair (2 gl, 2 gl + 1) at position n: the accumulator, or with
    // a split d the sum of the ks partial sums in rank order
    auto corr = [&](int rr, int n) -> float {
        if (ks == 1) return acc[rr * ld + n];
        float s = 0.f;
        for (int q = 0; q < ks; ++q) s += red[(q * nr + rr) * ld + n];
        return s;
    };
    for (int j0 = 0; j0 < Q; j0 += kConvEpiBatch) {
        if (j0 > 0) {
            pv = xv[kConvEpiBatch - 1];
            load_batch(j0);
        }
#pragma unroll
        for (int j = 0; j < kConvEpiBatch; ++j) {
            const int n = nb + j0 + j;
            const int pos = n_tile * NT + n;
            if (!gok || j0 + j >= Q || pos >= p.P) continue;
            const float c0 = corr(2 * gl, n), c1 = corr(2 * gl + 1, n);
            float x[8], xp[8];
            bf16x8_to_f32(xv[j], x);
            bf16x8_to_f32(j == 0 ? pv : xv[j - 1], xp);
            const float keep = (pos % p.S != 0) ? 1.f : 0.f;  // a block's first row has no predecessor
            uint32_t out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float y0 = (b0[2 * k] + c0) * x[2 * k] + keep * ((b1[2 * k] + c1) * xp[2 * k]);
                const float y1 = (b0[2 * k + 1] + c0) * x[2 * k + 1] + keep * ((b1[2 * k + 1] + c1) * xp[2 * k + 1]);
                const __nv_bfloat162 v = __floats2bfloat162_rn(y0, y1);
                out[k] = *reinterpret_cast<const uint32_t *>(&v);
            }
            *reinterpret_cast<uint4 *>(p.y + static_cast<size_t>(pos) * p.d + ch) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
    if (timed_out) atomicOr(p.err, DEV_ERR_TIMEOUT);
    if (ks > 1) cluster_wait();
}

// ---------------------------------------------------------------------------
// Few rows (P <= 8: one block): corr is a matrix-vector product
// bound by reading Wc, so CUDA cores do it without a tensor-core pipeline. A
// CTA takes NG channel groups: their 2 NG Wc rows (contiguous in memory) are
// bulk-copied into shared memory before the dependency wait (they are
// weights), then every thread takes a strided share of d for all P rows and
// all 2 NG rows, and after a fixed-order block reduction one thread per
// (row, group, half) writes 8 channels.
constexpr int kSmallThreads = 256;
constexpr int kSmallAcc = 64;   // PM * 2 NG accumulators per thread
constexpr int kSmallRows = 8;   // the few-row kernel's limit (measured: beyond 8 rows the tcgen05 kernel is faster)
// 16-byte pieces of d per thread whose x loads are in flight together: two up
// to d = 4096 (one pass; two CTAs per SM), else one (three CTAs per SM keep the
// 2 d / 32 CTAs of a larger d in one wave)
constexpr int kSmallUnitsMaxD = 4096;

// 1D bulk copy global -> this CTA's shared memory, counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

template <int PM, int NG, int UPT>
__global__ void __launch_bounds__(kSmallThreads, (UPT > 1) ? 2 : 3) conv2_small_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                    const __nv_bfloat16 *__restrict__ base,
                                                                    const __nv_bfloat16 *__restrict__ Wc,
                                                                    __nv_bfloat16 *__restrict__ y, int P, int S, int d,
                                                                    int *err)
{
    static_assert(PM * 2 * NG <= kSmallAcc, "accumulators per thread");
    extern __shared__ __align__(16) uint8_t wsm[];  // Wc rows [2 NG][d] bf16
    __shared__ float part[kSmallThreads / 32][2 * NG * PM];
    __shared__ float corr[2 * NG * PM];
    __shared__ __align__(8) uint64_t bar_w;
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d / 16;
    const int g0 = blockIdx.x * NG;
    const int ng = G - g0 < NG ? G - g0 : NG;  // groups of this CTA
    const int nu = d / 8;                     // 16-byte pieces of a row
    const uint32_t bar = smem_u32(&bar_w);
    if (tid == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t row_bytes = static_cast<uint32_t>(d) * 2;
        mbar_arrive_expect_tx(bar, 2u * ng * row_bytes);
        for (int r = 0; r < 2 * ng; ++r)
            bulk_copy_g2s(smem_u32(wsm) + r * row_bytes, Wc + static_cast<size_t>(2 * g0 + r) * d, row_bytes, bar);
    }
    // this thread's output piece: row er, group g0 + eg, channels 8 eh .. 8 eh + 7
    const int eh = tid & 1, eg = (tid >> 1) % NG, er = tid / (2 * NG);
    const bool epi = er < P && eg < ng;
    const size_t ch = static_cast<size_t>(g0 + (epi ? eg : 0)) * 16 + 8 * eh;
    const uint4 bv0 = __ldg(reinterpret_cast<const uint4 *>(base + ch));
    const uint4 bv1 = __ldg(reinterpret_cast<const uint4 *>(base + d + ch));
    pdl_trigger();
    pdl_wait();
    uint4 xv = make_uint4(0u, 0u, 0u, 0u), pv = make_uint4(0u, 0u, 0u, 0u);
    if (epi) {
        xv = *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(er) * d + ch);
        if (er % S != 0) pv = *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(er - 1) * d + ch);
    }
    bool timed_out = false;
    if (!mbar_wait(bar, 0, &abort_flag, false)) {  // then wait once more for the copies in flight
        timed_out = true;
        mbar_wait(bar, 0, &abort_flag, false);
    }

    float acc[PM][2 * NG];
#pragma unroll
    for (int r = 0; r < PM; ++r)
#pragma unroll
        for (int q = 0; q < 2 * NG; ++q) acc[r][q] = 0.f;
    const uint4 *w4 = reinterpret_cast<const uint4 *>(wsm);
    // UPT pieces of d per thread and pass, every x load of a pass issued before
    // its first use (one round trip to L2 per pass); the sums still run over u
    // in increasing order
    for (int u0 = tid; u0 < nu; u0 += UPT * kSmallThreads) {
        uint4 xr[UPT][PM];
#pragma unroll
        for (int v = 0; v < UPT; ++v) {
            const int u = u0 + v * kSmallThreads;
#pragma unroll
            for (int r = 0; r < PM; ++r)
                xr[v][r] = (u < nu && r < P) ? *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(r) * d +
                                                                                  8 * static_cast<size_t>(u))
                                             : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int v = 0; v < UPT; ++v) {
            const int u = u0 + v * kSmallThreads;
            if (u >= nu) break;
            float fw[2 * NG][8];
#pragma unroll
            for (int q = 0; q < 2 * NG; ++q)
                bf16x8_to_f32(q < 2 * ng ? w4[q * nu + u] : make_uint4(0u, 0u, 0u, 0u), fw[q]);
#pragma unroll
            for (int r = 0; r < PM; ++r) {
                if (r >= P) break;
                float fx[8];
                bf16x8_to_f32(xr[v][r], fx);
#pragma unroll
                for (int q = 0; q < 2 * NG; ++q)
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[r][q] = fmaf(fw[q][k], fx[k], acc[r][q]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < PM; ++r)
#pragma unroll
        for (int q = 0; q < 2 * NG; ++q) {
            float v = acc[r][q];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) part[warp][r * 2 * NG + q] = v;
        }
    __syncthreads();
    if (tid < 2 * NG * PM) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kSmallThreads / 32; ++w) sum += part[w][tid];  // warp order
        corr[tid] = sum;
    }
    __syncthreads();
    if (epi) {
        const float c0 = corr[er * 2 * NG + 2 * eg], c1 = corr[er * 2 * NG + 2 * eg + 1];
        float fx[8], fp[8], b0[8], b1[8];
        bf16x8_to_f32(bv0, b0);
        bf16x8_to_f32(bv1, b1);
        bf16x8_to_f32(xv, fx);
        bf16x8_to_f32(pv, fp);
        uint32_t out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float y0 = (b0[2 * k] + c0) * fx[2 * k] + (b1[2 * k] + c1) * fp[2 * k];
            const float y1 = (b0[2 * k + 1] + c0) * fx[2 * k + 1] + (b1[2 * k + 1] + c1) * fp[2 * k + 1];
            const __nv_bfloat162 v = __floats2bfloat162_rn(y0, y1);
            out[k] = *reinterpret_cast<const uint32_t *>(&v);
        }
        *reinterpret_cast<uint4 *>(y + static_cast<size_t>(er) * d + ch) = make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (timed_out && tid == 0) atomicOr(err, DEV_ERR_TIMEOUT);
}

template <int PM, int NG, int UPT>
cudaError_t launch_small(const __nv_bfloat16 *x, const __nv_bfloat16 *base, const __nv_bfloat16 *Wc, __nv_bfloat16 *y,
                         int P, int S, int d, int *err, cudaStream_t s)
{
    const size_t smem = static_cast<size_t>(2 * NG) * d * 2;
    const int G = d / 16;
    return launch_ex(conv2_small_kernel<PM, NG, UPT>, dim3((G + NG - 1) / NG), dim3(kSmallThreads), smem, s, 1, x, base, Wc,
                     y, P, S, d, err);
}

// Lets the few-row kernel take the Wc rows it needs (up to 64 KB).
cudaError_t prepare_small()
{
    const cudaError_t e = cudaFuncSetAttribute(conv2_small_kernel<kSmallRows, 1, 2>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(conv2_small_kernel<kSmallRows, 1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                64 * 1024);
}

}  // namespace

}  // namespace dfl

// ------------------------------------------------------------------------ host
struct dflash_conv2_ctx {
    int dev = 0, d = 0, rows = 0, num_sms = 0, smem_optin = 0;
    const void *base = nullptr, *Wc = nullptr;
    CUtensorMap tm_wc;
    int *err = nullptr;
};

namespace {

dflash_status conv_fail(dflash_status st, const char *fmt, long long a = 0, long long b = 0)
{
    char buf[256];
    snprintf(buf, sizeof buf, fmt, a, b);
    return dfl::host_fail(st, buf);
}

bool misaligned(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

}  // namespace

extern "C" dflash_status dflash_conv2_init(const void *base, const void *Wc, int32_t d, dflash_conv2_handle *out)
{
    if (!out) return conv_fail(DFLASH_ERR_INVALID_ARG, "out must not be NULL");
    *out = nullptr;
    if (!base || !Wc) return conv_fail(DFLASH_ERR_INVALID_ARG, "base and Wc must not be NULL");
    if (misaligned(base) || misaligned(Wc)) return conv_fail(DFLASH_ERR_INVALID_ARG, "base and Wc must be 16-byte aligned");
    if (d < 64 || d > 16384 || d % 64 != 0)
        return conv_fail(DFLASH_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 16384] (got %lld)", d);
    dflash_conv2_ctx *c = new (std::nothrow) dflash_conv2_ctx;
    if (!c) return conv_fail(DFLASH_ERR_CUDA, "out of host memory");
    int major = 0, minor = 0;
    if (cudaGetDevice(&c->dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, c->dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, c->dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->dev) != cudaSuccess) {
        delete c;
        return conv_fail(DFLASH_ERR_CUDA, "querying the current device failed");
    }
    if (major != 10 || minor != 3) {
        delete c;
        return conv_fail(DFLASH_ERR_UNSUPPORTED, "built for sm_103 (GB300); device is sm_%lld%lld", major, minor);
    }
    c->d = d;
    c->rows = d / 8;
    c->base = base;
    c->Wc = Wc;
    dflash_status st = dfl::host_make_tmap(&c->tm_wc, Wc, c->rows, d, dfl::kConvTileM);
    if (st != DFLASH_OK) {
        delete c;
        return st;
    }
    if (dfl::set_max_dynamic_smem(dfl::conv2_kernel, c->smem_optin) != cudaSuccess || dfl::prepare_small() != cudaSuccess ||
        cudaMalloc(&c->err, sizeof(int)) != cudaSuccess || cudaMemset(c->err, 0, sizeof(int)) != cudaSuccess) {
        if (c->err) cudaFree(c->err);
        delete c;
        return conv_fail(DFLASH_ERR_CUDA, "setting up the convolution failed");
    }
    *out = c;
    return DFLASH_OK;
}

extern "C" dflash_status dflash_conv2_run(dflash_conv2_handle h, const void *X, int32_t B, int32_t S, void *Y,
                                          void *stream)
{
    if (!h) return conv_fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    if (B < 0 || S < 1) return conv_fail(DFLASH_ERR_INVALID_ARG, "need B >= 0 and S >= 1 (got %lld, %lld)", B, S);
    const int64_t P64 = static_cast<int64_t>(B) * S;
    if (P64 >= (int64_t(1) << 31)) return conv_fail(DFLASH_ERR_INVALID_ARG, "B * S = %lld rows is too many", P64);
    if (P64 == 0) return DFLASH_OK;
    if (!X || !Y) return conv_fail(DFLASH_ERR_INVALID_ARG, "X and Y must not be NULL");
    if (misaligned(X) || misaligned(Y)) return conv_fail(DFLASH_ERR_INVALID_ARG, "X and Y must be 16-byte aligned");
    const int d = h->d;
    const size_t bytes = static_cast<size_t>(P64) * d * 2;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(X), ya = reinterpret_cast<uintptr_t>(Y);
    if (xa < ya + bytes && ya < xa + bytes) return conv_fail(DFLASH_ERR_INVALID_ARG, "Y must not overlap X");
    const int P = static_cast<int>(P64);

    if (P <= dfl::kSmallRows) {  // a matrix-vector product: CUDA cores, one channel group per CTA
        const auto *x = static_cast<const __nv_bfloat16 *>(X);
        const auto *base = static_cast<const __nv_bfloat16 *>(h->base);
        const auto *Wc = static_cast<const __nv_bfloat16 *>(h->Wc);
        auto *y = static_cast<__nv_bfloat16 *>(Y);
        const auto st = static_cast<cudaStream_t>(stream);
        const cudaError_t e = (d <= dfl::kSmallUnitsMaxD)
                                  ? dfl::launch_small<dfl::kSmallRows, 1, 2>(x, base, Wc, y, P, S, d, h->err, st)
                                  : dfl::launch_small<dfl::kSmallRows, 1, 1>(x, base, Wc, y, P, S, d, h->err, st);
        if (e != cudaSuccess) return conv_fail(DFLASH_ERR_CUDA, "convolution launch failed (error %lld)", e);
        return DFLASH_OK;
    }

    dfl::ConvParams prm;
    const int m_tiles = (h->rows + dfl::kConvTileM - 1) / dfl::kConvTileM;
    // The position-tile width NT (halved from the rows, down to 16) and the
    // split of d over a cluster (ks of 1, 2, 4, 8 dividing the k-blocks) that,
    // within one CTA per SM and the shared memory, stream the fewest bytes per
    // CTA: KB / ks stages of 16 KB of Wc and NT rows of X (a CTA's load time
    // sets the call's length; narrower tiles re-read Wc once per tile).
    // Ties go to the larger grid. With no pair in one wave: NT = 256, no split.
    const int KB = d / dfl::kLmTileK;
    int NT = 256, ks = 1;
    {
        int64_t best = -1, best_grid = 0;
        for (int nt = P <= 256 ? ((P + 15) / 16) * 16 : 256;; nt = ((nt / 2 + 15) / 16) * 16) {
            for (int k = 1; k <= dfl::kConvMaxSplit; k <<= 1) {
                const int64_t grid = static_cast<int64_t>(m_tiles) * ((P + nt - 1) / nt) * k;
                if (KB % k != 0 || grid > h->num_sms ||
                    dfl::conv_layout(nt, k, 1).total + 1024u > static_cast<uint32_t>(h->smem_optin))
                    continue;
                const int64_t bytes = static_cast<int64_t>(KB / k) * dfl::conv_layout(nt, k, 1).stage_bytes;
                if (best < 0 || bytes < best || (bytes == best && grid > best_grid)) {
                    best = bytes;
                    best_grid = grid;
                    NT = nt;
                    ks = k;
                }
            }
            if (nt <= 16) break;
        }
    }
    prm.NT = NT;
    const int n_tiles = (P + NT - 1) / NT;
    prm.ksplit = ks;
    const int KBc = KB / ks;
    int stages = KBc < dfl::kConvMaxStages ? KBc : dfl::kConvMaxStages;  // as deep as shared memory allows
    while (stages > 1 && dfl::conv_layout(prm.NT, ks, stages).total + 1024u > static_cast<uint32_t>(h->smem_optin))
        --stages;
    const size_t smem = dfl::conv_layout(prm.NT, ks, stages).total + 1024u;  // + alignment slack
    if (smem > static_cast<size_t>(h->smem_optin))
        return conv_fail(DFLASH_ERR_UNSUPPORTED, "shared memory: need %lld bytes, have %lld", static_cast<long long>(smem),
                         h->smem_optin);
    prm.stages = stages;

    prm.tm_wc = h->tm_wc;
    dflash_status st = dfl::host_make_tmap(&prm.tm_x, X, P, d, prm.NT);
    if (st != DFLASH_OK) return st;
    prm.x = static_cast<const __nv_bfloat16 *>(X);
    prm.base = static_cast<const __nv_bfloat16 *>(h->base);
    prm.y = static_cast<__nv_bfloat16 *>(Y);
    prm.P = P;
    prm.S = S;
    prm.d = d;
    prm.rows = h->rows;
    prm.err = h->err;
    const cudaError_t e = dfl::launch_ex(dfl::conv2_kernel, dim3(m_tiles, n_tiles, ks), dim3(dfl::kConvThreads), smem,
                                         static_cast<cudaStream_t>(stream), ks, prm);
    if (e != cudaSuccess) return conv_fail(DFLASH_ERR_CUDA, "convolution launch failed (error %lld)", e);
    return DFLASH_OK;
}

extern "C" dflash_status dflash_conv2_sync_status(dflash_conv2_handle h, void *stream)
{
    if (!h) return conv_fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int e = 0;
    if (cudaMemcpyAsync(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return conv_fail(DFLASH_ERR_CUDA, "reading the device error word failed");
    if (e == 0) return DFLASH_OK;
    if (cudaMemsetAsync(h->err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return conv_fail(DFLASH_ERR_CUDA, "clearing the device error word failed");
    return conv_fail(DFLASH_ERR_TIMEOUT, "a convolution pipeline wait exceeded its time bound (error word %lld)", e);
}

extern "C" dflash_status dflash_conv2_destroy(dflash_conv2_handle h)
{
    if (!h) return DFLASH_OK;
    cudaDeviceSynchronize();
    cudaFree(h->err);
    delete h;
    return DFLASH_OK;
}
