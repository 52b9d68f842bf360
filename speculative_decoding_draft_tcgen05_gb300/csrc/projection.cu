// Candidate projections A|B = [W_A; W_B] E[row] on the 5th-generation tensor
// cores, for the selector's larger-batch path and for building the
// precomputed A|B tables.
//
// Blog "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path
// Selector": A and B give every token a 256-wide embedding, A(a) = W_A E[a]
// and B(b) = W_B E[b] here. For every sequence the rows {x0, c_{0,*}, ...,
// c_{L-1,*}} of E are gathered and multiplied by W_A (first half of the
// output row) and W_B (second half).
//
// One CTA computes 128 gathered rows x NC outputs (NC = 64, 128 or 256 of the
// 512, chosen so that the grid fills the SMs):
//   - the 128 rows are the MMA's M (TMEM lanes), NC weight rows its N (TMEM
//     columns), d is streamed 64 columns per stage;
//   - the weight tile comes by TMA (128-byte swizzle); the gathered rows are
//     fetched by 256 threads with cp.async into the same swizzled layout
//     (16-byte chunk c of row r at r * 128 + ((c ^ (r % 8)) * 16));
//   - a stage is full when the TMA bytes have landed and all 256 gathering
//     threads have arrived (each after its copies completed and a proxy
//     fence), and free again when the MMAs that read it complete.
// Warp roles: warp 0 lane 0 TMA, warp 1 TMEM owner and MMA issuer, warps 2-9
// gather, then warps 2-5 move the accumulator from TMEM to global memory.
// Every pipeline wait is bounded.
//
// With few rows (a grid that would fill at most half the SMs) d is split in
// two: CTA z of a tile streams the z-th half of d and writes a partial sum;
// the tile's second CTA to finish (an atomic ticket, no waiting) adds the two
// halves in order and writes A|B, so results do not depend on timing.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kPrRows = 128;     // gathered rows per CTA
constexpr int kPrThreads = 320;  // 10 warps
constexpr int kPrGather = 256;   // gathering threads (warps 2-9)
constexpr uint32_t kPrEBytes = kPrRows * 64 * 2;  // 16 KB

template <int NC>
struct PrShape {
    static constexpr uint32_t kWBytes = NC * 64 * 2;
    static constexpr uint32_t kStageBytes = kPrEBytes + kWBytes;
    static constexpr int kStages = (192 * 1024) / kStageBytes < 8 ? (192 * 1024) / kStageBytes : 8;
    static constexpr uint32_t kOffTok = kStages * kStageBytes;
    static constexpr uint32_t kOffBar = kOffTok + kPrRows * 4;
    // full[S], empty[S], done, then the TMEM base and the abort flag
    static constexpr uint32_t kSmem = kOffBar + 8u * (2u * kStages + 1u) + 8u + 1024u;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk)
{
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's completed shared-memory writes before the tensor
// cores' (async proxy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// grid (512 / NC output tiles, ceil(R_total / 128) row tiles, p.ksplit), 320
// threads. p.tm_wa / p.tm_wb have boxes of 64 columns x NC rows.
template <int NC>
__global__ void __launch_bounds__(kPrThreads, 1) projection_tc_kernel(const __grid_constant__ ProjParams p)
{
    using Sh = PrShape<NC>;
    constexpr int kPrStages = Sh::kStages;
    constexpr uint32_t kPrWBytes = Sh::kWBytes;
    constexpr uint32_t kPrStageBytes = Sh::kStageBytes;
    constexpr uint32_t kPrOffTok = Sh::kOffTok;
    constexpr uint32_t kPrOffBar = Sh::kOffBar;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzled tiles need 1024 B alignment
    uint8_t *const gbase = smem_raw + (base - raw);
    int32_t *const tok = reinterpret_cast<int32_t *>(gbase + kPrOffTok);
    const uint32_t bar_full = base + kPrOffBar;
    const uint32_t bar_empty = bar_full + 8u * kPrStages;
    const uint32_t bar_done = bar_empty + 8u * kPrStages;
    uint32_t *const tmem_holder = reinterpret_cast<uint32_t *>(gbase + kPrOffBar + 8u * (2u * kPrStages + 1u));
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int ct = blockIdx.x;               // output columns [ct NC, (ct + 1) NC) of the 512
    const int half = ct / (256 / NC);        // 0: A = W_A E, 1: B = W_B E
    const int wrow0 = (ct % (256 / NC)) * NC;  // first weight row of this tile
    const int row0 = blockIdx.y * kPrRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's k-blocks of 64 columns: [kb0, kb0 + KB)
    const int KB_all = p.d / 64;
    const int KB_per = (KB_all + p.ksplit - 1) / p.ksplit;
    const int kb0 = static_cast<int>(blockIdx.z) * KB_per;
    const int KB = min(KB_all, kb0 + KB_per) - kb0;
    const CUtensorMap *const tmw = half ? &p.tm_wb : &p.tm_wa;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrStages; ++s) {
            mbar_init(bar_full + 8u * s, kPrGather + 1);  // every gathering thread + the TMA's expect_tx
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(tmem_holder), NC);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    pdl_trigger();
    // Deduplicated rows: their count comes from the previous kernel, so every
    // role waits for it first; a tile past the count does no work.
    int n_rows = p.R_total;
    if (p.uniq) {
        pdl_wait();
        n_rows = static_cast<int>(*reinterpret_cast<const volatile unsigned *>(p.count));
    }
    const bool active = row0 < n_rows;
    const int KBe = active ? KB : 0;

    bool timed_out = false;
    if (warp == 0) {
        // ------------------------------------------------ TMA: weight tiles
        if (lane == 0) {
            tma_prefetch_desc(tmw);
            const uint64_t pol = l2_policy_evict_last();  // every row tile reads the same weights
            const int pre = KBe < kPrStages ? KBe : kPrStages;
            for (int kb = 0; kb < pre; ++kb) {  // weights: before the dependency wait
                mbar_arrive_expect_tx(bar_full + 8u * kb, kPrWBytes);
                tma_load_2d(base + kb * kPrStageBytes + kPrEBytes, tmw, (kb0 + kb) * 64, wrow0, bar_full + 8u * kb, pol);
            }
            int kb = pre;
            for (; kb < KBe; ++kb) {
                const int s = kb % kPrStages;
                if (!mbar_wait(bar_empty + 8u * s, (static_cast<uint32_t>(kb / kPrStages) & 1u) ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                mbar_arrive_expect_tx(bar_full + 8u * s, kPrWBytes);
                tma_load_2d(base + s * kPrStageBytes + kPrEBytes, tmw, (kb0 + kb) * 64, wrow0, bar_full + 8u * s, pol);
            }
            if (timed_out)  // let the copies already issued land before the CTA can exit
                for (int j = (kb > kPrStages ? kb - kPrStages : 0); j < kb; ++j)
                    mbar_wait(bar_full + 8u * (j % kPrStages), static_cast<uint32_t>(j / kPrStages) & 1u, abort_flag,
                              false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPrRows, NC);
            for (int kb = 0; kb < KBe; ++kb) {
                const int s = kb % kPrStages;
                if (!mbar_wait(bar_full + 8u * s, static_cast<uint32_t>(kb / kPrStages) & 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = base + s * kPrStageBytes;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_bf16(tmem_base, smem_desc_sw128(st + 32u * k), smem_desc_sw128(st + kPrEBytes + 32u * k),
                              idesc, (kb > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar_empty + 8u * s);  // frees the stage once these MMAs have read it
            }
            if (active)
                umma_commit(bar_done);  // also after a timeout: every issued MMA must finish before TMEM is freed
            else
                mbar_arrive(bar_done);  // no MMA was issued
        }
    } else {
        // ------------------------------------------------ gather the E rows
        const int gt = threadIdx.x - 64;  // 0..255
        pdl_wait();                      // the candidates come from the previous kernel
        if (gt < kPrRows) {
            const int gr = row0 + gt;
            int32_t t = -1;
            if (gr < n_rows) {
                const int b = gr / p.R, rr = gr % p.R;
                t = p.uniq ? p.uniq[gr]
                           : ((rr == 0) ? p.anchor[b] : p.ids[static_cast<size_t>(b) * p.L * p.K + (rr - 1)]);
                if (t < 0 || static_cast<int64_t>(t) >= p.V) {
                    atomicOr(p.err, DEV_ERR_TOKEN);
                    t = 0;
                }
            }
            tok[gt] = t;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the gathering warps only
        int arrived = 0;  // k-blocks this thread has signalled
        for (int kb = 0; kb < KBe; ++kb) {
            const int s = kb % kPrStages;
            if (kb >= kPrStages &&
                !mbar_wait(bar_empty + 8u * s, (static_cast<uint32_t>(kb / kPrStages) & 1u) ^ 1u, abort_flag)) {
                timed_out = true;
                break;
            }
            const uint32_t et = base + s * kPrStageBytes;
#pragma unroll
            for (int u = 0; u < (kPrRows * 8) / kPrGather; ++u) {
                const int i = gt + u * kPrGather;
                const int r = i >> 3, c = i & 7;
                const int32_t t = tok[r];
                const uint16_t *src = p.E + static_cast<size_t>(t < 0 ? 0 : t) * p.d + (kb0 + kb) * 64 + c * 8;
                cp_async16(et + swz128(r, c), src, t < 0 ? 0u : 16u);  // rows past the end read as zero
            }
            cp_async_commit();
            if (kb >= kPrStages - 1) {  // the copies of k-block kb - (S - 1) are complete
                cp_async_wait<kPrStages - 1>();
                fence_proxy_async_smem();
                mbar_arrive(bar_full + 8u * (arrived % kPrStages));
                ++arrived;
            }
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        if (!timed_out)
            for (; arrived < KBe; ++arrived) mbar_arrive(bar_full + 8u * (arrived % kPrStages));
    }
    __syncwarp();

    // ---------------------------------------------------- epilogue: TMEM -> AB
    if (!mbar_wait(bar_done, 0, abort_flag, false)) timed_out = true;
    tc_fence_after_sync();
    if (active && warp >= 2 && warp < 6) {
        const int q = warp & 3;  // warp w may read TMEM lanes 32 (w % 4) ..
        const int r = q * 32 + lane;
        const int gr = row0 + r;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        float *const out = p.ksplit > 1 ? p.part + static_cast<size_t>(blockIdx.z) * p.R_total * 512 : p.AB;
        float *const dst = out + static_cast<size_t>(gr < p.R_total ? gr : 0) * 512 + ct * NC;
        for (int c0 = 0; c0 < NC; c0 += 16) {
            float v[16];
            __syncwarp();
            tmem_load16(taddr + static_cast<uint32_t>(c0), v);
            if (gr < n_rows) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
    }
    if (timed_out) atomicOr(p.err, DEV_ERR_TIMEOUT);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, NC);
    }
    if (p.ksplit > 1) {
        // the tile's last CTA adds the partial sums in split order
        __shared__ int last;
        __threadfence();  // this thread's partial sums before the ticket
        __syncthreads();
        unsigned *const tk = p.ticket + blockIdx.y * gridDim.x + blockIdx.x;
        if (threadIdx.x == 0) {
            last = atomicAdd(tk, 1u) == static_cast<unsigned>(p.ksplit - 1);
            if (last) *tk = 0;  // ready for the next run
        }
        __syncthreads();
        if (last) {
            // d is split in two halves (projection_ksplit); the loads of a
            // batch of items are all issued before any sum is stored, so a
            // batch costs one round trip to L2
            __threadfence();
            constexpr int nc4 = NC / 4;
            constexpr int kSumBatch = 8;
            const size_t zstride = static_cast<size_t>(p.R_total) * 512;
            const int n_items = max(0, min(kPrRows, n_rows - row0)) * nc4;
            for (int e0 = threadIdx.x; e0 < n_items; e0 += kSumBatch * kPrThreads) {
                float4 h0[kSumBatch], h1[kSumBatch];
#pragma unroll
                for (int u = 0; u < kSumBatch; ++u) {
                    const int e = e0 + u * kPrThreads;
                    if (e < n_items) {
                        const size_t off = static_cast<size_t>(row0 + e / nc4) * 512 + ct * NC + (e % nc4) * 4;
                        h0[u] = __ldcg(reinterpret_cast<const float4 *>(p.part + off));
                        h1[u] = __ldcg(reinterpret_cast<const float4 *>(p.part + zstride + off));
                    }
                }
#pragma unroll
                for (int u = 0; u < kSumBatch; ++u) {
                    const int e = e0 + u * kPrThreads;
                    if (e < n_items) {
                        const size_t off = static_cast<size_t>(row0 + e / nc4) * 512 + ct * NC + (e % nc4) * 4;
                        *reinterpret_cast<float4 *>(p.AB + off) = make_float4(h0[u].x + h1[u].x, h0[u].y + h1[u].y,
                                                                              h0[u].z + h1[u].z, h0[u].w + h1[u].w);
                    }
                }
            }
        }
    }
}

// One thread per gathered row: the row that holds the newest mark of its
// token takes the next index of the distinct-token list.
__global__ void __launch_bounds__(256) dedup_compact_kernel(const DedupParams d, const int32_t *__restrict__ ids,
                                                            int R_total)
{
    pdl_trigger();
    pdl_wait();
    const int gr = blockIdx.x * blockDim.x + threadIdx.x;
    if (gr >= R_total) return;
    const int b = gr / d.R, rr = gr % d.R;
    int32_t tok = (rr == 0) ? d.anchor[b] : ids[static_cast<size_t>(b) * d.L * d.K + (rr - 1)];
    if (tok < 0 || static_cast<int64_t>(tok) >= d.V) {
        atomicOr(d.err, DEV_ERR_TOKEN);
        tok = 0;
    }
    const uint64_t mine = (static_cast<uint64_t>(d.epoch) << 32) | ~static_cast<uint32_t>(gr);
    if (__ldcg(reinterpret_cast<const unsigned long long *>(d.tab + tok)) == mine) {
        const unsigned u = atomicAdd(d.count, 1u);
        d.uniq[u] = tok;
        d.rep[gr] = static_cast<int32_t>(u);
    }
}

template <int NC>
cudaError_t set_smem()
{
    return cudaFuncSetAttribute(projection_tc_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(PrShape<NC>::kSmem));
}

}  // namespace

cudaError_t prepare_projection(int smem_optin)
{
    (void)smem_optin;
    cudaError_t e = set_smem<64>();
    if (e == cudaSuccess) e = set_smem<128>();
    if (e == cudaSuccess) e = set_smem<256>();
    return e;
}

int projection_ksplit(int R_total, int NC, int d, int num_sms)
{
    const int rt = (R_total + kPrRows - 1) / kPrRows;
    // halves of equal length only: an odd count of 64-column blocks keeps one
    // CTA per tile (with d a multiple of 64 but not of 128 the small-batch
    // tail runs clusters of one CTA, so the three-kernel tail, the only user of
    // the split, never sees so few rows there anyway)
    return (2 * (512 / NC) * rt <= num_sms && d / 64 >= 8 && (d / 64) % 2 == 0) ? 2 : 1;
}

int projection_split_rows(int num_sms)
{
    // the split needs 2 x 8 CTAs per row tile (64 output columns: the narrowest tiles)
    return (num_sms / 16) * kPrRows;
}

int projection_cols(int R_total, int num_sms)
{
    const int rt = (R_total + kPrRows - 1) / kPrRows;
    if (8 * rt <= num_sms) return 64;
    if (4 * rt <= num_sms) return 128;
    return 256;
}

cudaError_t launch_dedup_compact(const DedupParams &d, const int32_t *ids, int R_total, cudaStream_t s)
{
    return launch_ex(dedup_compact_kernel, dim3((R_total + 255) / 256), dim3(256), 0, s, 1, d, ids, R_total);
}

cudaError_t launch_projection(const ProjParams &p, int NC, cudaStream_t s)
{
    if (p.ksplit < 1 || p.ksplit > 2) return cudaErrorInvalidValue;  // the sum adds two halves
    const dim3 grid(512 / NC, (p.R_total + kPrRows - 1) / kPrRows, p.ksplit);
    if (NC == 64) return launch_ex(projection_tc_kernel<64>, grid, dim3(kPrThreads), PrShape<64>::kSmem, s, 1, p);
    if (NC == 128) return launch_ex(projection_tc_kernel<128>, grid, dim3(kPrThreads), PrShape<128>::kSmem, s, 1, p);
    return launch_ex(projection_tc_kernel<256>, grid, dim3(kPrThreads), PrShape<256>::kSmem, s, 1, p);
}

}  // namespace dfl
