// Candidate projections, pair tables and the walk of the DFlash 2 path selector.
//
// Blog "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path
// Selector": every adjacent pair (a, b) of candidates at position t is scored
//     S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) >,
// all pairs in one shot, and the only sequential work is the final walk over
// the precomputed scores, starting from the last verified token. Here
// A(a) = W_A E[a], B(b) = W_B E[b] (one shared token table E) and
// H(h_t) = g_t = W_H h_t (computed by the lm_head kernel).
//
// projection_kernel: for every sequence, the rows {x0, c_{0,*}, ..., c_{L-1,*}}
//   of E are gathered and multiplied by [W_A; W_B] (512 x d) with warp-level
//   bf16 mma.sync (a dense dot-product tile), fp32 accumulation. When the
//   batch is small the hidden dimension is split over a thread-block cluster
//   and the partial tiles are summed in a fixed order through distributed
//   shared memory (deterministic, no global scratch).
// pair_walk_kernel: one CTA per (sequence, position) builds the K x K table in
//   fp32 (CUDA cores; exact fp32 inputs, no rounding to bf16); the last CTA of
//   each sequence (atomic ticket, no waiting) runs the walk in one warp.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "walk.cuh"

namespace cg = cooperative_groups;

namespace dfl {

namespace {

constexpr int kPM = 128;      // outputs per CTA (rows of [W_A; W_B])
constexpr int kPN = 64;       // gathered rows per CTA
constexpr int kPK = 64;       // hidden columns per stage
constexpr int kPStages = 4;
constexpr int kPThreads = 256;
constexpr int kPsStride = kPM + 4;  // fp32 row stride of the staged output tile
constexpr uint32_t kPStageBytes = (kPM + kPN) * kPK * 2;
constexpr size_t kProjSmem = kPStages * kPStageBytes + kPN * 4;

static_assert(kPN * kPsStride * 4 <= kPStages * kPStageBytes, "output tile must fit in the stage buffers");

__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    // byte offset of 16-byte chunk `chunk` (0..7) of a 128-byte row, XOR-swizzled
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

// grid (4 output tiles, ceil(R_total / 64) row tiles, ksplit); cluster (1, 1, ksplit)
__global__ void __launch_bounds__(kPThreads) projection_kernel(const ProjParams p)
{
    extern __shared__ __align__(128) uint8_t psm[];
    const uint32_t sbase = smem_u32(psm);
    int32_t *const tok = reinterpret_cast<int32_t *>(psm + kPStages * kPStageBytes);

    const int mt = blockIdx.x;        // 0,1: W_A rows; 2,3: W_B rows
    const int n0 = blockIdx.y * kPN;  // first gathered row
    const int kz = blockIdx.z;        // hidden-dimension slice
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint16_t *W = (mt < 2 ? p.WA : p.WB) + static_cast<size_t>((mt & 1) * kPM) * p.d;

    // The weight slice does not depend on earlier kernels: pull it towards L2
    // while the candidates are still being produced.
    pdl_trigger();
    for (int i = tid; i < kPM * (p.kchunk / 64); i += kPThreads) {
        const int r = i / (p.kchunk / 64), c = i % (p.kchunk / 64);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(W + static_cast<size_t>(r) * p.d + kz * p.kchunk + c * 64));
    }
    pdl_wait();

    for (int r = tid; r < kPN; r += kPThreads) {
        const int gr = n0 + r;
        int32_t t = -1;
        if (gr < p.R_total) {
            const int b = gr / p.R, rr = gr % p.R;
            t = (rr == 0) ? p.anchor[b] : p.ids[static_cast<size_t>(b) * p.L * p.K + (rr - 1)];
            if (t < 0 || static_cast<int64_t>(t) >= p.V) {
                atomicOr(p.err, DEV_ERR_TOKEN);
                t = 0;
            }
        }
        tok[r] = t;
    }
    __syncthreads();

    const int k_begin = kz * p.kchunk;
    const int nkb = p.kchunk / kPK;

    auto load_stage = [&](int kb, int stage) {
        const uint32_t ws = sbase + stage * kPStageBytes;
        const uint32_t es = ws + kPM * kPK * 2;
        const int kcol = k_begin + kb * kPK;
        for (int i = tid; i < kPM * 8; i += kPThreads) {
            const int r = i >> 3, c = i & 7;
            cp_async16(ws + swz(r, c), W + static_cast<size_t>(r) * p.d + kcol + c * 8, 16);
        }
        for (int i = tid; i < kPN * 8; i += kPThreads) {
            const int r = i >> 3, c = i & 7;
            const int t = tok[r];
            const uint16_t *src = p.E + static_cast<size_t>(t < 0 ? 0 : t) * p.d + kcol + c * 8;
            cp_async16(es + swz(r, c), src, t < 0 ? 0u : 16u);
        }
    };

    const int wm = warp & 3;   // 32 output rows each
    const int wn = warp >> 2;  // 32 gathered rows each
    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

#pragma unroll
    for (int s = 0; s < kPStages - 1; ++s) {
        if (s < nkb) load_stage(s, s);
        cp_async_commit();
    }
    for (int kb = 0; kb < nkb; ++kb) {
        cp_async_wait<kPStages - 2>();
        __syncthreads();
        const int nxt = kb + kPStages - 1;
        if (nxt < nkb) load_stage(nxt, nxt % kPStages);
        cp_async_commit();
        const uint32_t ws = sbase + (kb % kPStages) * kPStageBytes;
        const uint32_t es = ws + kPM * kPK * 2;
#pragma unroll
        for (int kk = 0; kk < kPK / 16; ++kk) {
            uint32_t af[2][4], bf[2][4];
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int r = wm * 32 + mi * 16 + (lane & 15);
                ldmatrix_x4(ws + swz(r, kk * 2 + (lane >> 4)), af[mi]);
            }
#pragma unroll
            for (int nj = 0; nj < 2; ++nj) {
                const int r = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldmatrix_x4(es + swz(r, kk * 2 + ((lane >> 3) & 1)), bf[nj]);
            }
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    mma_16816(acc[mi][ni], af[mi], bf[ni >> 1][(ni & 1) * 2], bf[ni >> 1][(ni & 1) * 2 + 1]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // stage this CTA's partial tile as Ps[row][output]
    float *const Ps = reinterpret_cast<float *>(psm);
    {
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int o = wm * 32 + mi * 16 + g;
                const int r = wn * 32 + ni * 8 + 2 * t4;
                Ps[r * kPsStride + o] = acc[mi][ni][0];
                Ps[(r + 1) * kPsStride + o] = acc[mi][ni][1];
                Ps[r * kPsStride + o + 8] = acc[mi][ni][2];
                Ps[(r + 1) * kPsStride + o + 8] = acc[mi][ni][3];
            }
    }

    const int ks = p.ksplit;
    const float4 *const Ps4 = reinterpret_cast<const float4 *>(Ps);
    constexpr int kRow4 = kPsStride / 4;  // float4 per staged row
    if (ks > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = static_cast<int>(cluster.block_rank());
        const int rows = kPN / ks;
        // rows [rank * rows, (rank + 1) * rows) of the tile, 128 outputs each,
        // one float4 per thread per pass; the ks partial tiles are read from the
        // peers' shared memory (all loads first, then the fixed-order sum)
        for (int i = tid; i < rows * (kPM / 4); i += kPThreads) {
            const int r = rank * rows + i / (kPM / 4), o4 = i % (kPM / 4);
            float4 part[8];
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
                if (qq < ks) part[qq] = cluster.map_shared_rank(Ps4, qq)[r * kRow4 + o4];
            float4 sum = part[0];
#pragma unroll
            for (int qq = 1; qq < 8; ++qq)
                if (qq < ks) {
                    sum.x += part[qq].x;
                    sum.y += part[qq].y;
                    sum.z += part[qq].z;
                    sum.w += part[qq].w;
                }
            const int gr = n0 + r;
            if (gr < p.R_total)
                *reinterpret_cast<float4 *>(p.AB + static_cast<size_t>(gr) * 512 + mt * kPM + o4 * 4) = sum;
        }
        cluster.sync();  // keep this CTA's tile alive until every peer has read it
    } else {
        __syncthreads();
        for (int i = tid; i < kPN * (kPM / 4); i += kPThreads) {
            const int r = i / (kPM / 4), o4 = i % (kPM / 4);
            const int gr = n0 + r;
            if (gr < p.R_total)
                *reinterpret_cast<float4 *>(p.AB + static_cast<size_t>(gr) * 512 + mt * kPM + o4 * 4) =
                    Ps4[r * kRow4 + o4];
        }
    }
}

// grid B * L; block 256. Builds S_t for one (sequence, position); the last
// CTA of a sequence to finish walks its tables. Every global load batch is
// issued in full before its values are used (one round trip per batch).
template <int K>
__global__ void __launch_bounds__(256) pair_walk_kernel(const PairParams p)
{
    extern __shared__ float pw_smem[];
    float *const Agt = pw_smem;                // (A(prev_i) (.) g_t)[k] at [k * K + i]
    float *const Bt = pw_smem + kEmbed * K;    // B(c_{t,j})[k] at [k * K + j]
    __shared__ float vals[K];
    __shared__ WalkSmem<K> ws;
    __shared__ int is_last;

    pdl_trigger();
    pdl_wait();
    const int L = p.L, R = p.R;
    const int b = blockIdx.x / L, t = blockIdx.x % L;
    const int tid = threadIdx.x;
    const int n_prev = (t == 0) ? 1 : K;
    const size_t pos = static_cast<size_t>(b) * L + t;

    {
        const int k = tid;  // blockDim.x == kEmbed: thread k owns component k
        const size_t rowA0 = static_cast<size_t>(b) * R + (t == 0 ? 0 : 1 + (t - 1) * K);
        const size_t rowB0 = static_cast<size_t>(b) * R + 1 + t * K;
        float a[K], bb[K];
        const float gk = p.gate[pos * kEmbed + k];
        if (p.tab) {  // precomputed A|B rows, found by token
            const int32_t *cur = p.ids + pos * K;
            int32_t x0 = 0;
            if (t == 0) {
                x0 = p.anchor[b];
                if (x0 < 0 || static_cast<int64_t>(x0) >= p.V) {
                    if (tid == 0) atomicOr(p.err, DEV_ERR_TOKEN);
                    x0 = 0;
                }
            }
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const int32_t tok = (t == 0) ? x0 : cur[i - K];  // candidates of t-1
                a[i] = (i < n_prev) ? __ldg(p.tab + static_cast<size_t>(tok) * 512 + k) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < K; ++j) bb[j] = __ldg(p.tab + static_cast<size_t>(cur[j]) * 512 + kEmbed + k);
        } else {
#pragma unroll
            for (int i = 0; i < K; ++i) a[i] = (i < n_prev) ? p.AB[(rowA0 + i) * 512 + k] : 0.f;
#pragma unroll
            for (int j = 0; j < K; ++j) bb[j] = p.AB[(rowB0 + j) * 512 + kEmbed + k];
        }
        const float v = (tid < K) ? p.vals[pos * K + tid] : 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) Agt[k * K + i] = a[i] * gk;
#pragma unroll
        for (int j = 0; j < K; ++j) Bt[k * K + j] = bb[j];
        if (tid < K) vals[tid] = v;
    }
    __syncthreads();

    float *Pt = p.P + pos * K * K;
    float *Po = p.P_out ? p.P_out + pos * K * K : nullptr;
    for (int e = tid; e < K * K; e += blockDim.x) {
        const int i = e / K, jj = e % K;
        float s;
        if (i < n_prev) {
            // two partial sums halve the dependent FMA chain
            float d0 = 0.f, d1 = 0.f;
#pragma unroll 8
            for (int k = 0; k < kEmbed; k += 2) {
                d0 = fmaf(Agt[k * K + i], Bt[k * K + jj], d0);
                d1 = fmaf(Agt[(k + 1) * K + i], Bt[(k + 1) * K + jj], d1);
            }
            s = vals[jj] + (d0 + d1);
        } else {
            s = -INFINITY;  // only the anchor precedes position 0
        }
        Pt[e] = s;
        if (Po) Po[e] = s;
    }

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.ticket[b], 1u);
        is_last = (prev == static_cast<unsigned>(L - 1));
        if (is_last) {
            p.ticket[b] = 0;  // ready for the next run
            __threadfence();
        }
    }
    __syncthreads();
    if (!is_last) return;

    walk_sequence<K>(p.P + static_cast<size_t>(b) * L * K * K, p.ids + static_cast<size_t>(b) * L * K, L, p.walk,
                     p.tie_eps, pw_smem, ws, p.path + static_cast<size_t>(b) * L,
                     p.path_score ? p.path_score + b : nullptr,
                     p.tie_flags ? p.tie_flags + static_cast<size_t>(b) * L : nullptr,
                     SampleArgs{p.u_walk ? p.u_walk + static_cast<size_t>(b) * L : nullptr,
                                p.q_out ? p.q_out + static_cast<size_t>(b) * L * K : nullptr, p.temperature});
}

}  // namespace

int projection_ksplit(int d, int R_total, int num_sms)
{
    const int ntiles = (R_total + kPN - 1) / kPN;
    int ks = 1;
    while (ks < 8 && 4 * ntiles * ks * 2 <= 2 * num_sms && d % (kPK * ks * 2) == 0) ks *= 2;
    return ks;
}

cudaError_t prepare_pair_walk(int smem_optin)
{
    cudaError_t e = set_max_dynamic_smem(projection_kernel, smem_optin);
    if (e != cudaSuccess) return e;
    e = set_max_dynamic_smem(pair_walk_kernel<16>, smem_optin);
    if (e != cudaSuccess) return e;
    return set_max_dynamic_smem(pair_walk_kernel<32>, smem_optin);
}

cudaError_t launch_projection(const ProjParams &p, cudaStream_t s)
{
    return launch_ex(projection_kernel, dim3(4, (p.R_total + kPN - 1) / kPN, p.ksplit), dim3(kPThreads), kProjSmem, s,
                     p.ksplit, p);
}

cudaError_t launch_pair_walk(const PairParams &p, cudaStream_t s)
{
    const size_t smem = 2u * kEmbed * p.K * sizeof(float);
    if (p.K == 16) return launch_ex(pair_walk_kernel<16>, dim3(p.B * p.L), dim3(256), smem, s, 1, p);
    return launch_ex(pair_walk_kernel<32>, dim3(p.B * p.L), dim3(256), smem, s, 1, p);
}

}  // namespace dfl
