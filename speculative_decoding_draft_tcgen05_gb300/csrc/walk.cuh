// The walk over one sequence's precomputed pair tables (blog "DFlash 2: Keep
// Drafting Parallel", section "A Lightweight Path Selector": the only
// sequential work is the final walk, starting from the last verified token).
//
// Walks (walk = 0, 1, 2):
// Max-sum (Viterbi) walk: delta_0(j) = S_0(x0, j);
// delta_t(j) = max_i delta_{t-1}(i) + S_t(i, j), the smallest rank i winning
// ties; the path ends at the best final rank (smallest on ties) and is read
// back through the back-pointers. Greedy walk: from x0, the best successor at
// every step (smallest rank on ties). Sampling walk (the pages draw samples
// from the same pair scores): at every step the next rank is drawn from
// softmax(S_t(prev, .) / T) over the K candidates by inverting its CDF in rank
// order with a given uniform u_t; the distribution is written out for the
// rejection-sampling verifier. One warp, lane j = candidate rank j.
#pragma once

#include "common.cuh"

namespace dfl {

template <int K>
struct WalkSmem {
    uint8_t bp[16 * K];    // back-pointers [t][j]
    float mg[16 * K];      // gap between the best and second incoming value [t][j]
    float delta[2][K];     // max-sum values of the previous and current step
    int32_t ids[16 * K];   // candidate tokens [t][rank]
    int ranks[16];
    uint8_t flags[16];
};

struct SampleArgs {
    const float *u;  // [L] uniforms of the sequence (walk 2)
    float *q_out;    // [L, K] drawn-from distributions (walk 2)
    float temperature;
};

// The greedy accept check of the walked path, done by the walking warp when
// the caller passes the target's argmax tokens (NULL target: not done).
struct VerifyArgs {
    const int32_t *target;  // [L + 1] target argmax tokens after x0, path[0], ...
    int32_t *accept;        // [1] n = leading positions with path[t] == target[t]
    int32_t *emitted;       // [L + 1] path[0..n-1], target[n], then -1 (may be NULL)
    // Results written straight to mapped host memory (may be NULL): once this
    // sequence's outputs are written, the device error word as the walker saw
    // it goes to *err_snap and `step` to *done, each write fenced at system
    // scope, so that a host thread polling *done can read the outputs.
    uint32_t *done = nullptr;
    int *err_snap = nullptr;
    const int *err = nullptr;
    uint32_t step = 0;
};

// Called by every thread of a 256-thread CTA, uniformly. Stages the L tables
// P_seq [L, K, K] and the candidates ids_seq [L, K] (written by other CTAs of
// this or an earlier kernel; read around L1) into shared memory (Pb, ws.ids),
// walks them and writes the path tokens ids_seq[t * K + rank_t], the path
// score and the tie flags (bit 0: the choice at t had a margin below tie_eps
// -- for the sampling walk, the uniform lay within tie_eps of a CDF boundary;
// bit 1 at t = L-1: the final choice of the max-sum walk did).
//
// The max-sum recursion runs on all 256 threads: at each step, thread
// (j, ig) takes the predecessors i = ig, ig + 256/K, ... of candidate j in
// increasing order, and the 256/K threads of candidate j (adjacent lanes)
// combine their (best, first index of best, second best) with shuffles. The
// result equals the sequential scan over i: the same sums, the smallest rank
// among equal bests, and a second best equal to the best on a tie. The
// greedy and sampling walks are sequential over t and run on one warp.

template <int K>
__device__ __forceinline__ void walk_sequence(const float *P_seq, const int32_t *ids_seq, int L, int walk,
                                              float tie_eps, float *Pb, WalkSmem<K> &ws, int32_t *path_out,
                                              float *score_out, uint8_t *flags_out, SampleArgs sa = {},
                                              VerifyArgs va = {})
{
    const int tid = threadIdx.x;
    // the target tokens of the accept check do not depend on the walk: loaded
    // with the tables, not after the path is known
    const int32_t tg = (va.target && tid <= L) ? __ldg(va.target + tid) : 0;
    {
        int32_t idv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + u * 256;
            if (i < L * K) idv[u] = __ldcg(ids_seq + i);
        }
        const float4 *src = reinterpret_cast<const float4 *>(P_seq);
        float4 *dst = reinterpret_cast<float4 *>(Pb);
        const int n4 = L * K * K / 4;
        for (int i0 = 0; i0 < n4; i0 += 4 * 256) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * 256 + tid;
                if (i < n4) v[u] = __ldcg(src + i);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * 256 + tid;
                if (i < n4) dst[i] = v[u];
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + u * 256;
            if (i < L * K) ws.ids[i] = idv[u];
        }
        if (walk == 0 && tid < K) ws.delta[0][tid] = __ldcg(P_seq + tid);  // delta_0(j) = S_0(x0, j)
    }
    __syncthreads();
    if (walk == 0) {
        constexpr int kIG = 256 / K;  // threads per candidate j
        constexpr int kIU = K / kIG;  // predecessors per thread
        const int j = tid / kIG, ig = tid % kIG;
        for (int s = 1; s < L; ++s) {
            const float *Ps = Pb + s * K * K;
            const float *dl = ws.delta[(s - 1) & 1];
            float best = -INFINITY, second = -INFINITY;
            int bi = 0;
#pragma unroll
            for (int u = 0; u < kIU; ++u) {
                const int i = ig + u * kIG;
                const float v = dl[i] + Ps[i * K + j];
                if (v > best) {
                    second = best;
                    best = v;
                    bi = i;
                } else if (v > second) {
                    second = v;
                }
            }
#pragma unroll
            for (int off = kIG / 2; off > 0; off >>= 1) {
                const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
                const float os = __shfl_xor_sync(0xFFFFFFFFu, second, off);
                second = fmaxf(fmaxf(second, os), fminf(best, ob));
                if (ob > best || (ob == best && oi < bi)) bi = oi;
                best = fmaxf(best, ob);
            }
            if (ig == 0) {
                ws.bp[s * K + j] = static_cast<uint8_t>(bi);
                ws.mg[s * K + j] = best - second;
                ws.delta[s & 1][j] = best;
            }
            __syncthreads();
        }
    }
    if (tid >= 32) return;
    const int lane = tid;
    const bool active = lane < K;
    float score;

    if (walk == 0) {
        const float delta = active ? ws.delta[(L - 1) & 1][lane] : -INFINITY;
        float bv = active ? delta : -INFINITY;
        int bj = lane;
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
            const int oj = __shfl_xor_sync(0xFFFFFFFFu, bj, off);
            if (ov > bv || (ov == bv && oj < bj)) {
                bv = ov;
                bj = oj;
            }
        }
        float sv = (active && lane != bj) ? delta : -INFINITY;
        for (int off = 16; off > 0; off >>= 1) sv = fmaxf(sv, __shfl_xor_sync(0xFFFFFFFFu, sv, off));
        __syncwarp();
        score = bv;
        if (lane == 0) {
            int jcur = bj;
            for (int s = L - 1; s >= 0; --s) {
                ws.ranks[s] = jcur;
                uint8_t f = 0;
                if (s > 0) {
                    if (ws.mg[s * K + jcur] < tie_eps) f |= 1;
                    jcur = ws.bp[s * K + jcur];
                }
                if (s == L - 1 && bv - sv < tie_eps) f |= 2;
                ws.flags[s] = f;
            }
        }
    } else if (walk == 2) {
        int prev = 0;
        float total = 0.f;
        for (int s = 0; s < L; ++s) {
            const float v = active ? Pb[(s * K + prev) * K + lane] : -INFINITY;
            float m = v;
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            const float e = active ? expf((v - m) / sa.temperature) : 0.f;
            float c = e;  // inclusive running sum in rank order
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xFFFFFFFFu, c, off);
                if (lane >= off) c += y;
            }
            const float Z = __shfl_sync(0xFFFFFFFFu, c, 31);
            const float target = __ldg(sa.u + s) * Z;
            const unsigned above = __ballot_sync(0xFFFFFFFFu, active && c > target);
            const int chosen = above ? __ffs(above) - 1 : K - 1;
            float dist = (lane < K - 1) ? fabsf(c - target) / Z : INFINITY;
            for (int off = 16; off > 0; off >>= 1) dist = fminf(dist, __shfl_xor_sync(0xFFFFFFFFu, dist, off));
            if (sa.q_out && active) sa.q_out[s * K + lane] = e / Z;
            if (lane == 0) {
                ws.ranks[s] = chosen;
                ws.flags[s] = (dist < tie_eps) ? 1 : 0;
            }
            total += __shfl_sync(0xFFFFFFFFu, v, chosen);
            prev = chosen;
        }
        score = total;
    } else {
        int prev = 0;
        float total = 0.f;
        for (int s = 0; s < L; ++s) {
            const float v = active ? Pb[(s * K + prev) * K + lane] : -INFINITY;
            float bv = v;
            int bj = lane;
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
                const int oj = __shfl_xor_sync(0xFFFFFFFFu, bj, off);
                if (ov > bv || (ov == bv && oj < bj)) {
                    bv = ov;
                    bj = oj;
                }
            }
            float sv = (active && lane != bj) ? v : -INFINITY;
            for (int off = 16; off > 0; off >>= 1) sv = fmaxf(sv, __shfl_xor_sync(0xFFFFFFFFu, sv, off));
            if (lane == 0) {
                ws.ranks[s] = bj;
                ws.flags[s] = (bv - sv < tie_eps) ? 1 : 0;
            }
            total += bv;
            prev = bj;
        }
        score = total;
    }
    __syncwarp();
    const int32_t tok = (lane < L) ? ws.ids[lane * K + ws.ranks[lane]] : 0;
    if (lane < L) {
        path_out[lane] = tok;
        if (flags_out) flags_out[lane] = ws.flags[lane];
    }
    if (lane == 0 && score_out) *score_out = score;
    if (va.target) {
        const unsigned miss = __ballot_sync(0xFFFFFFFFu, lane < L && tok != tg);
        const int n = miss ? __ffs(miss) - 1 : L;
        if (lane == 0) *va.accept = n;
        if (va.emitted && lane <= L) va.emitted[lane] = (lane < n) ? tok : (lane == n ? tg : -1);
    }
    if (va.done) {
        __threadfence_system();  // this lane's outputs before the flag
        __syncwarp();
        if (lane == 0) {
            *va.err_snap = *reinterpret_cast<const volatile int *>(va.err);
            __threadfence_system();
            *reinterpret_cast<volatile uint32_t *>(va.done) = va.step;
        }
    }
}

}  // namespace dfl
