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
// The projections A|B of the gathered candidates come from projection.cu.
// pair_walk_kernel: one CTA per (sequence, position) builds the K x K table in
//   fp32 (CUDA cores, register-tiled; exact fp32 inputs, no rounding to bf16);
//   the last CTA of each sequence (atomic ticket, no waiting) runs the walk.
#include "common.cuh"
#include "kernels.h"
#include "walk.cuh"

namespace dfl {

namespace {

// grid B * L; block 256. Builds S_t for one (sequence, position); the last
// CTA of a sequence to finish walks its tables. Every global load batch is
// issued in full before its values are used (one round trip per batch).
// Agt and Bt hold K values per component k in rows of K / 4 float4 units;
// unit u of row k sits at u ^ pw_swz<K>(k), so that the float4 stores of eight
// consecutive components (one shared-memory phase) hit eight different banks
// groups, and a row's units stay a permutation of the row for the readers.
template <int K>
__device__ __forceinline__ int pw_swz(int k)
{
    static_assert(K == 16 || K == 32, "K is 16 or 32");
    constexpr int U = K / 4;
    return (k / (8 / U)) % U;
}

template <int K>
__global__ void __launch_bounds__(256, (K == 16) ? 4 : 2) pair_walk_kernel(const PairParams p)
{
    extern __shared__ float pw_smem[];
    float *const Agt = pw_smem;                // (A(prev_i) (.) g_t)[k], row k, swizzled units
    float *const Bt = pw_smem + kEmbed * K;    // B(c_{t,j})[k], row k, swizzled units
    __shared__ float vals[K];
    __shared__ WalkSmem<K> ws;
    __shared__ int is_last;
    __shared__ int32_t dd_row[2 * K];  // deduplicated AB rows of the predecessors and the candidates

    pdl_wait();
    const int L = p.L, R = p.R;
    const int b = blockIdx.x / L, t = blockIdx.x % L;
    const int tid = threadIdx.x;
    const int n_prev = (t == 0) ? 1 : K;
    const size_t pos = static_cast<size_t>(b) * L + t;

    if (p.dd_tab) {
        if (tid < 2 * K && (tid < n_prev || tid >= K)) {
            int32_t tok;
            if (tid >= K) {
                tok = p.ids[pos * K + (tid - K)];
            } else if (t == 0) {
                tok = p.anchor[b];
                if (tok < 0 || static_cast<int64_t>(tok) >= p.V) tok = 0;  // reported by the compaction
            } else {
                tok = p.ids[(pos - 1) * K + tid];
            }
            const uint64_t mark = __ldcg(reinterpret_cast<const unsigned long long *>(p.dd_tab + tok));
            dd_row[tid] = __ldcg(p.dd_rep + ~static_cast<uint32_t>(mark));
        }
        __syncthreads();
    }

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
        } else if (p.dd_tab) {
#pragma unroll
            for (int i = 0; i < K; ++i)
                a[i] = (i < n_prev) ? p.AB[static_cast<size_t>(dd_row[i]) * 512 + k] : 0.f;
#pragma unroll
            for (int j = 0; j < K; ++j) bb[j] = p.AB[static_cast<size_t>(dd_row[K + j]) * 512 + kEmbed + k];
        } else {
#pragma unroll
            for (int i = 0; i < K; ++i) a[i] = (i < n_prev) ? p.AB[(rowA0 + i) * 512 + k] : 0.f;
#pragma unroll
            for (int j = 0; j < K; ++j) bb[j] = p.AB[(rowB0 + j) * 512 + kEmbed + k];
        }
        const float v = (tid < K) ? p.vals[pos * K + tid] : 0.f;
        float4 *const a4 = reinterpret_cast<float4 *>(Agt + k * K);
        float4 *const b4 = reinterpret_cast<float4 *>(Bt + k * K);
        const int sw = pw_swz<K>(k);
#pragma unroll
        for (int u = 0; u < K / 4; ++u) {
            a4[u ^ sw] = make_float4(a[4 * u] * gk, a[4 * u + 1] * gk, a[4 * u + 2] * gk, a[4 * u + 3] * gk);
            b4[u ^ sw] = make_float4(bb[4 * u], bb[4 * u + 1], bb[4 * u + 2], bb[4 * u + 3]);
        }
        if (tid < K) vals[tid] = v;
    }
    __syncthreads();
    // the next kernel (the next lm_head pass) is scheduled once every CTA has
    // its operands: its early weight loads no longer compete with these
    pdl_trigger();

    float *Pt = p.P + pos * K * K;
    float *Po = p.P_out ? p.P_out + pos * K * K : nullptr;
    {
        // Register tiles: thread (kg, bi, bj) sums, over its component group
        // kg, the RT x RT pairs (bi RT + r1, bj RT + r2), RT = K / 8, reading RT
        // values of each operand per component (one vector load each), so shared
        // memory serves RT^2 FMAs per two loads instead of one FMA per two.
        // Group kg holds the components k = 8 j + 2 kg + e (j < 32, e < 2): their
        // rows share one swizzle (K = 16: pw_swz = kg) or two (K = 32: 2 kg + e),
        // so the column offsets of the loads do not change along the loop.
        constexpr int RT = K / 8;
        const int kg = tid >> 6, bi = (tid >> 3) & 7, bj = tid & 7;
        float acc[RT][RT];
#pragma unroll
        for (int r1 = 0; r1 < RT; ++r1)
#pragma unroll
            for (int r2 = 0; r2 < RT; ++r2) acc[r1][r2] = 0.f;
        int ca[2], cb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int sw = (K == 16) ? kg : 2 * kg + e;  // pw_swz<K>(8 j + 2 kg + e)
            ca[e] = (bi * RT) ^ (sw << 2);
            cb[e] = (bj * RT) ^ (sw << 2);
        }
        const float *arow = Agt + (2 * kg) * K;
        const float *brow = Bt + (2 * kg) * K;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float a[RT], bb[RT];
                if constexpr (RT == 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(arow + e * K + ca[e]);
                    const float4 bv = *reinterpret_cast<const float4 *>(brow + e * K + cb[e]);
                    a[0] = av.x, a[1] = av.y, a[2] = av.z, a[3] = av.w;
                    bb[0] = bv.x, bb[1] = bv.y, bb[2] = bv.z, bb[3] = bv.w;
                } else {
                    const float2 av = *reinterpret_cast<const float2 *>(arow + e * K + ca[e]);
                    const float2 bv = *reinterpret_cast<const float2 *>(brow + e * K + cb[e]);
                    a[0] = av.x, a[1] = av.y;
                    bb[0] = bv.x, bb[1] = bv.y;
                }
#pragma unroll
                for (int r1 = 0; r1 < RT; ++r1)
#pragma unroll
                    for (int r2 = 0; r2 < RT; ++r2) acc[r1][r2] = fmaf(a[r1], bb[r2], acc[r1][r2]);
            }
            arow += 8 * K;
            brow += 8 * K;
        }
        __syncthreads();  // every thread is done with Agt / Bt
        float *const part = pw_smem;  // [4 component groups][K * K], over Agt
#pragma unroll
        for (int r1 = 0; r1 < RT; ++r1)
#pragma unroll
            for (int r2 = 0; r2 < RT; ++r2) part[kg * K * K + (bi * RT + r1) * K + bj * RT + r2] = acc[r1][r2];
        __syncthreads();
        for (int e = tid; e < K * K; e += blockDim.x) {
            const int i = e / K, jj = e % K;
            // the four component groups in order
            const float dot = ((part[e] + part[K * K + e]) + part[2 * K * K + e]) + part[3 * K * K + e];
            const float sc = (i < n_prev) ? vals[jj] + dot : -INFINITY;  // only the anchor precedes position 0
            Pt[e] = sc;
            if (Po) Po[e] = sc;
        }
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
                                p.q_out ? p.q_out + static_cast<size_t>(b) * L * K : nullptr, p.temperature},
                     VerifyArgs{p.target ? p.target + static_cast<size_t>(b) * (L + 1) : nullptr,
                                p.accept ? p.accept + b : nullptr,
                                p.emitted ? p.emitted + static_cast<size_t>(b) * (L + 1) : nullptr,
                                p.done ? p.done + b : nullptr, p.err_snap ? p.err_snap + b : nullptr, p.err,
                                p.step});
}

}  // namespace

cudaError_t prepare_pair_walk(int smem_optin)
{
    cudaError_t e = set_max_dynamic_smem(pair_walk_kernel<16>, smem_optin);
    if (e != cudaSuccess) return e;
    return set_max_dynamic_smem(pair_walk_kernel<32>, smem_optin);
}

cudaError_t launch_pair_walk(const PairParams &p, cudaStream_t s, size_t min_smem)
{
    const size_t need = 2u * kEmbed * p.K * sizeof(float);
    const size_t smem = need > min_smem ? need : min_smem;
    if (p.K == 16) return launch_ex(pair_walk_kernel<16>, dim3(p.B * p.L), dim3(256), smem, s, 1, p);
    return launch_ex(pair_walk_kernel<32>, dim3(p.B * p.L), dim3(256), smem, s, 1, p);
}

}  // namespace dfl
