// Fused selector tail for small batches: merge, projections, pair tables and
// the walk in one kernel, one thread-block cluster per draft position.
//
// Blog "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path
// Selector": the pair score S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) > of
// every adjacent candidate pair, then one walk from the last verified token.
// With A(a) = W_A E[a], B(b) = W_B E[b] and g_t = H(h_t) (from the lm_head
// kernel), the table of position t needs the candidates of t and of t-1 (or
// the anchor x0 at t = 0).
//
// When batch x positions is small, the separate merge / projection / pair
// kernels are latency chains (a kernel boundary and a memory round trip
// each). Here a cluster of CS CTAs owns one position (b, t):
//   1. each CTA TMA-prefetches its hidden-dimension slice of W_A and W_B (the
//      weights do not depend on earlier kernels, so this overlaps them);
//   2. each CTA merges its share of the lm_head kernel's partial top-K lists
//      for positions t and t-1; the cluster folds the CS shares through
//      distributed shared memory (DSMEM), so every CTA knows both candidate
//      sets (rank 0 publishes position t's);
//   3. each CTA gathers the E rows of the 2K tokens for its slice and computes
//      its partial A (W_A x prev rows) and B (W_B x current rows) with bf16
//      mma.sync, fp32 accumulation;
//   4. the partials are summed over the cluster in rank order through DSMEM,
//      each CTA owning 256/CS columns of A and B; A is multiplied by g_t and
//      each CTA forms its partial pair dot products and stores them into rank
//      0's shared memory; rank 0 sums those (rank order) and adds U_t(b): the
//      table S_t;
//   5. the last cluster of a sequence (atomic ticket, no waiting) walks.
// With precomputed tables [A(v) | B(v)] for every token (a handle option),
// steps 1 and 3 are replaced by a gather: each CTA reads its 256/cs columns of
// the 2K candidates' table rows (no weights, no MMA, one cluster barrier less).
// Every summation order is fixed, so results are deterministic.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "walk.cuh"

namespace cg = cooperative_groups;

namespace dfl {

namespace {

constexpr uint32_t kWTileBytes = 256 * 64 * 2;  // 256 rows of W_A (or W_B) x 64 columns, bf16
constexpr int kRedPad = 1;                      // row padding of the reduced slice (bank conflicts)

__host__ __device__ inline uint32_t tail_stage_bytes(int K)
{
    return 2 * kWTileBytes + static_cast<uint32_t>(2 * K) * 128;
}

struct TailLayout {
    uint32_t stage, off_mlist, off_ctalist, off_bar, off_misc, total;
};



__host__ __device__ inline TailLayout tail_layout(int K, int S, int G, int cs)
{
    TailLayout l;
    l.stage = tail_stage_bytes(K);
    const int per = (G + cs - 1) / cs;
    l.off_mlist = S * l.stage;
    l.off_ctalist = l.off_mlist + static_cast<uint32_t>(2 * per * K) * 8;
    l.off_bar = l.off_ctalist + 2 * 32 * 8;
    l.off_misc = l.off_bar + 8 * S;
    l.total = l.off_misc + 16;
    return l;
}

// Loads from another CTA's shared memory (an address from mapa_shared), with
// the cluster state space named explicitly rather than through a generic
// pointer (measured: 0.16 us per batch-1 step on the reduction below).
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_cluster_u64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// grid (1, 1, N * cs), cluster (1, 1, cs), 256 threads.
template <int K, int S>
__global__ void __launch_bounds__(256, 1) select_tail_kernel(const __grid_constant__ TailParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    __shared__ uint64_t wl[8][32];
    __shared__ int32_t cand[2][K];   // [0]: candidates of t, [1]: of t-1 (or the anchor)
    __shared__ float cand_val[K];
    __shared__ int32_t rowtok[2 * K];
    __shared__ float gs[kEmbed];
    __shared__ WalkSmem<K> ws;
    __shared__ int is_last;

    cg::cluster_group cluster = cg::this_cluster();
    const int cs = p.cs;
    const int rank = static_cast<int>(cluster.block_rank());
    const int pos = blockIdx.z / cs;
    const int L = p.L, N = p.N, G = p.G;
    const int b = pos / L, t = pos % L;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kc = p.d / cs, nkb = kc / 64, k0 = rank * kc;
    const TailLayout lay = tail_layout(K, S, G, cs);
    uint64_t *const mlist = reinterpret_cast<uint64_t *>(gbase + lay.off_mlist);
    uint64_t *const cta_list = reinterpret_cast<uint64_t *>(gbase + lay.off_ctalist);
    const uint32_t bar_full = base + lay.off_bar;
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(gbase + lay.off_misc);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bar_full + 8u * s, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool tab = p.tab != nullptr;  // precomputed A|B rows: no projections here
    const int pre = nkb < S ? nkb : S;
    if (tid == 0 && !tab) {
        tma_prefetch_desc(&p.tm_wa);
        tma_prefetch_desc(&p.tm_wb);
        const uint64_t pol = l2_policy_evict_last();  // every cluster reads the same slices
        for (int s = 0; s < pre; ++s) {
            const uint32_t st = base + s * lay.stage;
            mbar_arrive_expect_tx(bar_full + 8u * s, 2 * kWTileBytes);
            tma_load_2d(st, &p.tm_wa, k0 + s * 64, 0, bar_full + 8u * s, pol);
            tma_load_2d(st + kWTileBytes, &p.tm_wb, k0 + s * 64, 0, bar_full + 8u * s, pol);
        }
    }
    // the anchor is an input of the run, not written by the previous kernel
    // (it may sit in mapped host memory): read before the dependency wait
    const int32_t anchor_tok = (t == 0 && tid == 32) ? p.anchor[b] : 0;
    pdl_wait();

    // ---------------- 1. candidates of t and t-1 from the partial lists
    const int nq = (t > 0) ? 2 : 1;
    const int per = (G + cs - 1) / cs;
    const int g0 = rank * per;
    const int gn = max(0, min(G, g0 + per) - g0);
    if (tid < kEmbed) gs[tid] = p.gate[static_cast<size_t>(pos) * kEmbed + tid];
    if (rank == 0 && tid == 0) p.thr_g[pos] = 0;  // ready for the next lm_head pass
    {
        const int total = nq * gn * K;
        constexpr int kBatch = 8;
        for (int i0 = 0; i0 < total; i0 += kBatch * 256) {
            uint64_t v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = i0 + u * 256 + tid;
                if (i < total) {
                    const int q = i / (gn * K), rem = i % (gn * K);
                    const int g = g0 + rem / K, k = rem % K;
                    v[u] = p.part[(static_cast<size_t>(g) * N + (pos - q)) * K + k];
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = i0 + u * 256 + tid;
                if (i < total) mlist[i] = v[u];
            }
        }
    }
    __syncthreads();
    {
        const int q = warp >> 2, wi = warp & 3;
        uint64_t run = 0;
        if (q < nq)
            for (int i = wi; i < gn; i += 4) {
                const uint64_t x = (lane < K) ? mlist[(q * gn + i) * K + lane] : 0ull;
                run = list_merge(run, x, lane, K);
            }
        wl[warp][lane] = run;
        __syncthreads();
        if (wi == 0 && q < nq) {
            run = list_merge(run, wl[warp + 1][lane], lane, K);
            run = list_merge(run, wl[warp + 2][lane], lane, K);
            run = list_merge(run, wl[warp + 3][lane], lane, K);
            cta_list[q * 32 + lane] = run;
        }
    }
    cluster.sync();
    {
        // the cluster's CS lists of position t - q, folded in a tree: warp
        // 4q + w merges the lists of ranks 2w and 2w + 1, then pairs of those
        // results, then the last two (three merges deep instead of eight)
        const int q = warp >> 2, w4 = warp & 3;
        uint64_t r = 0;
        if (q < nq) {
            const uint32_t la = smem_u32(cta_list + q * 32 + lane);
            const uint64_t x0 = (2 * w4 < cs && lane < K) ? ld_cluster_u64(mapa_shared(la, 2 * w4)) : 0ull;
            const uint64_t x1 = (2 * w4 + 1 < cs && lane < K) ? ld_cluster_u64(mapa_shared(la, 2 * w4 + 1)) : 0ull;
            r = list_merge(x0, x1, lane, K);
        }
        wl[warp][lane] = r;
        __syncthreads();
        if (q < nq && (w4 & 1) == 0) {
            r = list_merge(r, wl[warp + 1][lane], lane, K);
            wl[warp][lane] = r;
        }
        __syncthreads();
        if (q < nq && w4 == 0) {
            r = list_merge(r, wl[warp + 2][lane], lane, K);
            if (lane < K) {
                cand[q][lane] = key_id(r);
                if (q == 0) cand_val[lane] = key_val(r);
            }
        }
    }
    if (t == 0 && warp == 1 && lane < K) {
        int32_t a = -1;
        if (lane == 0) {
            a = anchor_tok;
            if (a < 0 || static_cast<int64_t>(a) >= p.V) {
                atomicOr(p.err, DEV_ERR_TOKEN);
                a = 0;
            }
        }
        cand[1][lane] = a;
    }
    __syncthreads();
    if (rank == 0 && tid < K) {
        const size_t o = static_cast<size_t>(pos) * K + tid;
        p.ids[o] = cand[0][tid];
        p.vals[o] = cand_val[tid];
        if (p.ids_out) p.ids_out[o] = cand[0][tid];
        if (p.vals_out) p.vals_out[o] = cand_val[tid];
    }
    if (tid < 2 * K) {
        int32_t tok = (tid < K) ? cand[1][tid] : cand[0][tid - K];
        if (tok >= 0 && static_cast<int64_t>(tok) >= p.V) {  // never for keys the lm_head kernel wrote
            atomicOr(p.err, DEV_ERR_TOKEN);
            tok = 0;
        }
        rowtok[tid] = tok;
    }
    __syncthreads();

    // the 256/cs columns of A (rows 0..K-1, times g_t) and B (rows K..2K-1)
    // that this CTA owns, as Red[row][column]
    const int es = kEmbed / cs, e0 = rank * es;
    const int rs = es + kRedPad;
    float *Red;
    if (tab) {
        // ---------------- 2'. gather the rows from the precomputed table
        Red = reinterpret_cast<float *>(gbase);
        for (int i = tid; i < 2 * K * (es / 4); i += 256) {
            const int r = i / (es / 4), e4 = i % (es / 4);
            const int col = e0 + e4 * 4;
            const int tok = rowtok[r];
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tok >= 0)
                v = __ldg(reinterpret_cast<const float4 *>(p.tab + static_cast<size_t>(tok) * 512 + (r < K ? 0 : kEmbed) +
                                                           col));
            if (r < K) {
                v.x *= gs[col];
                v.y *= gs[col + 1];
                v.z *= gs[col + 2];
                v.w *= gs[col + 3];
            }
            float *dst = Red + r * rs + e4 * 4;
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
    } else {
        // ---------------- 2. partial projections over this CTA's slice of d
        auto load_e = [&](int kb, int s) {
            const uint32_t et = base + s * lay.stage + 2 * kWTileBytes;
            for (int i = tid; i < 2 * K * 8; i += 256) {
                const int r = i >> 3, c = i & 7;
                const int tok = rowtok[r];
                const uint16_t *src = p.E + static_cast<size_t>(tok < 0 ? 0 : tok) * p.d + k0 + kb * 64 + c * 8;
                cp_async16(et + swz(r, c), src, tok < 0 ? 0u : 16u);
            }
        };
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if (s < nkb) load_e(s, s);
            cp_async_commit();
        }
        const int part = warp >> 2;  // 0: A = W_A x previous rows, 1: B = W_B x current rows
        const int wm = warp & 3;     // 64 output columns each
        float acc[4][K / 8][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < K / 8; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % S;
            cp_async_wait<S - 1>();
            if (!mbar_wait(bar_full + 8u * s, static_cast<uint32_t>(kb / S) & 1u, abort_flag, false))
                atomicOr(p.err, DEV_ERR_TIMEOUT);
            __syncthreads();
            const uint32_t wt = base + s * lay.stage + part * kWTileBytes;
            const uint32_t et = base + s * lay.stage + 2 * kWTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t af[4][4], bf[K / 16][4];
#pragma unroll
                for (int mi = 0; mi < 4; ++mi)
                    ldmatrix_x4(wt + swz(wm * 64 + mi * 16 + (lane & 15), kk * 2 + (lane >> 4)), af[mi]);
#pragma unroll
                for (int nj = 0; nj < K / 16; ++nj)
                    ldmatrix_x4(et + swz(part * K + nj * 16 + (lane & 7) + ((lane >> 4) << 3), kk * 2 + ((lane >> 3) & 1)),
                                bf[nj]);
#pragma unroll
                for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                    for (int ni = 0; ni < K / 8; ++ni)
                        mma_16816(acc[mi][ni], af[mi], bf[ni >> 1][(ni & 1) * 2], bf[ni >> 1][(ni & 1) * 2 + 1]);
            }
            __syncthreads();
            const int nxt = kb + S;
            if (nxt < nkb) {
                if (tid == 0) {
                    const uint32_t st = base + s * lay.stage;
                    const uint64_t pol = l2_policy_evict_last();
                    mbar_arrive_expect_tx(bar_full + 8u * s, 2 * kWTileBytes);
                    tma_load_2d(st, &p.tm_wa, k0 + nxt * 64, 0, bar_full + 8u * s, pol);
                    tma_load_2d(st + kWTileBytes, &p.tm_wb, k0 + nxt * 64, 0, bar_full + 8u * s, pol);
                }
                load_e(nxt, s);
            }
            cp_async_commit();
        }
        cp_async_wait<0>();
        __syncthreads();

        // partial results as Pa[row][column]: rows 0..K-1 = A of the previous
        // candidates, K..2K-1 = B of the current ones; 256 columns (+4 padding)
        constexpr int kPaStride = kEmbed + 4;
        float *const Pa = reinterpret_cast<float *>(gbase);
        {
            const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < K / 8; ++ni) {
                    const int o = wm * 64 + mi * 16 + g;
                    const int r = part * K + ni * 8 + 2 * t4;
                    Pa[r * kPaStride + o] = acc[mi][ni][0];
                    Pa[(r + 1) * kPaStride + o] = acc[mi][ni][1];
                    Pa[r * kPaStride + o + 8] = acc[mi][ni][2];
                    Pa[(r + 1) * kPaStride + o + 8] = acc[mi][ni][3];
                }
        }
        cluster.sync();

        // ---------------- 3. sum the partials of this CTA's 256/cs columns;
        // A rows times g_t
        Red = Pa + 2 * K * kPaStride;  // [2K][es + pad], after this CTA's Pa
        for (int i = tid; i < 2 * K * (es / 4); i += 256) {
            const int r = i / (es / 4), e4 = i % (es / 4);
            const int col = e0 + e4 * 4;
            float4 v[8];
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
                if (qq < cs)
                    v[qq] = ld_cluster_f4(mapa_shared(smem_u32(Pa + r * kPaStride + col), static_cast<uint32_t>(qq)));
            float4 sum = v[0];
#pragma unroll
            for (int qq = 1; qq < 8; ++qq)
                if (qq < cs) {
                    sum.x += v[qq].x;
                    sum.y += v[qq].y;
                    sum.z += v[qq].z;
                    sum.w += v[qq].w;
                }
            if (r < K) {
                sum.x *= gs[col];
                sum.y *= gs[col + 1];
                sum.z *= gs[col + 2];
                sum.w *= gs[col + 3];
            }
            float *dst = Red + r * rs + e4 * 4;
            dst[0] = sum.x;
            dst[1] = sum.y;
            dst[2] = sum.z;
            dst[3] = sum.w;
        }
    }
    __syncthreads();
    // each CTA's partial pair dots go straight to its slot in rank 0's receive
    // area [CS][K * K]: in rank 0's stage buffers past its partial projections
    // and its reduced slice (which other CTAs read before they write here; no
    // MMA or copy of a stage is pending anywhere by now)
    const uint32_t rx_off = (tab ? 0u : static_cast<uint32_t>(2 * K * (kEmbed + 4) * 4)) +
                            (static_cast<uint32_t>(2 * K * rs * 4) + 15u) / 16u * 16u;
    float *const rx = reinterpret_cast<float *>(gbase + rx_off);
    float *const rx_slot = cluster.map_shared_rank(rx, 0) + rank * K * K;
    for (int pr = tid; pr < K * K; pr += 256) {
        const int i = pr / K, j = pr % K;
        const float *a = Red + i * rs;
        const float *bb = Red + (K + j) * rs;
        float d0 = 0.f, d1 = 0.f;
        int e = 0;
        for (; e + 1 < es; e += 2) {
            d0 = fmaf(a[e], bb[e], d0);
            d1 = fmaf(a[e + 1], bb[e + 1], d1);
        }
        if (e < es) d0 = fmaf(a[e], bb[e], d0);
        rx_slot[pr] = d0 + d1;
    }
    cluster.sync();  // the partials are in place; no CTA reads another CTA's shared memory after this
    if (rank != 0) return;

    // ---------------- 4. rank 0: the table S_t, its partials summed in rank order
    {
        float *Pt = p.P + static_cast<size_t>(pos) * K * K;
        float *Po = p.P_out ? p.P_out + static_cast<size_t>(pos) * K * K : nullptr;
        for (int pr = tid; pr < K * K; pr += 256) {
            const int i = pr / K, j = pr % K;
            float sum = rx[pr];
            for (int qq = 1; qq < cs; ++qq) sum += rx[qq * K * K + pr];
            const float sc = (t == 0 && i > 0) ? -INFINITY : cand_val[j] + sum;
            Pt[pr] = sc;
            if (Po) Po[pr] = sc;
        }
    }

    // ---------------- 5. the last cluster of the sequence walks
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.ticket[b], 1u);
        is_last = (prev == static_cast<unsigned>(L - 1));
        if (is_last) {
            p.ticket[b] = 0;
            __threadfence();
        }
    }
    __syncthreads();
    // The next kernel on the stream (the next lm_head pass) may be scheduled
    // from here: its early weight loads would compete with this kernel's
    // memory phases (measured: 0.85 us per batch-1 step); the other CTAs
    // count as triggered when they exit.
    pdl_trigger();
    if (!is_last) return;
    walk_sequence<K>(p.P + static_cast<size_t>(b) * L * K * K, p.ids + static_cast<size_t>(b) * L * K, L, p.walk,
                     p.tie_eps, reinterpret_cast<float *>(gbase), ws, p.path + static_cast<size_t>(b) * L,
                     p.path_score ? p.path_score + b : nullptr,
                     p.tie_flags ? p.tie_flags + static_cast<size_t>(b) * L : nullptr,
                     SampleArgs{p.u_walk ? p.u_walk + static_cast<size_t>(b) * L : nullptr,
                                p.q_out ? p.q_out + static_cast<size_t>(b) * L * K : nullptr, p.temperature},
                     VerifyArgs{p.target ? p.target + static_cast<size_t>(b) * (L + 1) : nullptr,
                                p.accept ? p.accept + b : nullptr,
                                p.emitted ? p.emitted + static_cast<size_t>(b) * (L + 1) : nullptr,
                                p.done ? p.done + b : nullptr, p.err_snap ? p.err_snap + b : nullptr, p.err,
                                p.step});
}

template <int K, int S>
cudaError_t launch_tail_impl(const TailParams &p, size_t smem, cudaStream_t s)
{
    return launch_ex(select_tail_kernel<K, S>, dim3(1, 1, p.N * p.cs), dim3(256), smem, s, p.cs, p);
}

}  // namespace

int tail_cluster_size(int d)
{
    int cs = 8;
    while (cs > 1 && d % (64 * cs) != 0) cs >>= 1;
    return cs;
}

// Stages for this shape (3 if shared memory allows, else 2), 0 if even 2 do not fit.
int tail_stages(int K, int G, int cs, int smem_optin)
{
    for (int S = 3; S >= 2; --S) {
        const TailLayout l = tail_layout(K, S, G, cs);
        // the staged partial tile and the reduced slice reuse the stage buffers
        const size_t reuse = static_cast<size_t>(2 * K) * (kEmbed + 4) * 4 +
                             static_cast<size_t>(2 * K) * (kEmbed / cs + kRedPad) * 4;
        const size_t walk = static_cast<size_t>(16) * K * K * 4;
        // rank 0 receives the CS CTAs' partial pair dots after those two
        const size_t rx_end = reuse + 16 + static_cast<size_t>(cs) * K * K * 4;
        if (rx_end > static_cast<size_t>(S) * l.stage || walk > static_cast<size_t>(S) * l.stage) continue;
        if (l.total + 1024 + 10 * 1024 <= static_cast<size_t>(smem_optin)) return S;  // 10 KB: static shared memory
    }
    return 0;
}

size_t tail_smem_bytes(int K, int S, int G, int cs)
{
    return tail_layout(K, S, G, cs).total + 1024;
}

cudaError_t prepare_tail(int smem_optin)
{
    cudaError_t e;
    if ((e = set_max_dynamic_smem(select_tail_kernel<16, 3>, smem_optin)) != cudaSuccess) return e;
    if ((e = set_max_dynamic_smem(select_tail_kernel<16, 2>, smem_optin)) != cudaSuccess) return e;
    if ((e = set_max_dynamic_smem(select_tail_kernel<32, 3>, smem_optin)) != cudaSuccess) return e;
    return set_max_dynamic_smem(select_tail_kernel<32, 2>, smem_optin);
}

cudaError_t launch_select_tail(const TailParams &p, int K, int S, size_t smem, cudaStream_t s)
{
    if (K == 16) return S == 3 ? launch_tail_impl<16, 3>(p, smem, s) : launch_tail_impl<16, 2>(p, smem, s);
    return S == 3 ? launch_tail_impl<32, 3>(p, smem, s) : launch_tail_impl<32, 2>(p, smem, s);
}

}  // namespace dfl
