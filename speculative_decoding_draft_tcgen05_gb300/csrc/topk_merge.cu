// Merge of the lm_head kernel's partial top-K lists into the K candidates of
// every position (blog "DFlash 2: Keep Drafting Parallel", section "A
// Lightweight Path Selector": the selector keeps the drafter's 16 best tokens
// per draft position). Every CTA of the lm_head pass (or every vocabulary
// shard) wrote one sorted list of K 64-bit keys per position over its share of
// the vocabulary; the top K of their union is the top K over the vocabulary.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

// Writes the merged list of position col (lanes 0..K-1 of one warp hold it)
// and, with deduplication, marks its candidates' gathered rows (and, at a
// sequence's first position, the anchor's, from the thread with first_thread).
__device__ __forceinline__ void merge_emit(int col, uint64_t run, int lane, int K, int32_t *ids_ws, float *vals_ws,
                                           int32_t *ids_out, float *vals_out, uint64_t *keys_out,
                                           const DedupParams &dd, bool first_thread)
{
    if (lane < K) {
        const int32_t id = key_id(run);
        const float v = key_val(run);
        const size_t o = static_cast<size_t>(col) * K + lane;
        ids_ws[o] = id;
        vals_ws[o] = v;
        if (ids_out) ids_out[o] = id;
        if (vals_out) vals_out[o] = v;
        if (keys_out) keys_out[o] = run;
        if (dd.tab && id >= 0 && static_cast<int64_t>(id) < dd.V) {  // this candidate's gathered row
            const int b = col / dd.L, t = col % dd.L;
            const uint32_t gr = static_cast<uint32_t>(b * dd.R + 1 + t * dd.K + lane);
            atomicMax(reinterpret_cast<unsigned long long *>(dd.tab + id),
                      static_cast<unsigned long long>((static_cast<uint64_t>(dd.epoch) << 32) | ~gr));
        }
    }
    if (dd.tab && first_thread && col % dd.L == 0) {  // the sequence's anchor row
        const int b = col / dd.L;
        int32_t x0 = dd.anchor[b];
        if (x0 < 0 || static_cast<int64_t>(x0) >= dd.V) x0 = 0;  // reported by the compaction
        const uint32_t gr = static_cast<uint32_t>(b * dd.R);
        atomicMax(reinterpret_cast<unsigned long long *>(dd.tab + x0),
                  static_cast<unsigned long long>((static_cast<uint64_t>(dd.epoch) << 32) | ~gr));
    }
}

// One CTA per position. The G partial lists of the position are staged in
// shared memory with coalesced loads; each of the 16 warps folds a share of
// them into a sorted list, then the warps' lists are folded pairwise in a
// tree (4 rounds).
constexpr int kMergeWarps = 16;
constexpr int kMergeSurvivors = 128;  // keys the fast path sorts (four warp-wide batches)

template <int K>
__global__ void __launch_bounds__(kMergeWarps * 32) topk_merge_kernel(const uint64_t *__restrict__ part, int G,
                                                                      int N, int32_t *ids_ws, float *vals_ws,
                                                                      int32_t *ids_out, float *vals_out,
                                                                      uint64_t *thr_g, uint64_t *keys_out,
                                                                      const DedupParams dd)
{
    extern __shared__ uint64_t mlists[];  // [G][K]
    __shared__ uint64_t wl[kMergeWarps][32];
    pdl_wait();
    const int col = blockIdx.x;
    if (threadIdx.x == 0) thr_g[col] = 0;  // ready for the next lm_head pass
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // every load of a batch is issued before any of them is stored, so the
    // batch costs one memory round trip
    constexpr int kBatch = 10;
    for (int i0 = 0; i0 < G * K; i0 += kBatch * kMergeWarps * 32) {
        uint64_t v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kMergeWarps * 32 + threadIdx.x;
            v[u] = (i < G * K) ? part[(static_cast<size_t>(i / K) * N + col) * K + (i % K)] : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kMergeWarps * 32 + threadIdx.x;
            if (i < G * K) mlists[i] = v[u];
        }
    }
    __syncthreads();
    // the next kernel (the projections) is scheduled once the lists are in
    // shared memory: its early weight loads no longer compete with these
    // (measured: 1.3 us per batch-8 step)
    pdl_trigger();
    // Fast path: K lists whose best logits are all >= v hold K keys of logit
    // >= v, so the K-th best key is at least (v, any id) and only keys of logit
    // >= v can be in the result (v: the K-th largest best logit among the
    // lists, compared as ordered 32-bit images). Usually a few dozen keys
    // pass; up to four warps sort a batch of 32 each and one warp merges the
    // batches. With more (or fewer than K lists) the lists are merged whole.
    __shared__ uint64_t bound_s;
    __shared__ unsigned nsurv_s;
    __shared__ uint64_t surv[kMergeSurvivors];
    if (warp == 0) {
        uint32_t best = 0;
        for (int g = lane; g < G; g += 32) {
            const uint32_t h = static_cast<uint32_t>(mlists[g * K] >> 32);
            best = h > best ? h : best;
        }
        best = warp_sort_desc_u32(best, lane);
        const uint32_t v = __shfl_sync(0xFFFFFFFFu, best, K - 1);
        if (lane == 0) {
            bound_s = static_cast<uint64_t>(v) << 32;
            nsurv_s = 0;
        }
    }
    __syncthreads();
    const uint64_t bound = bound_s;
    if (bound != 0) {
        for (int i = threadIdx.x; i < G * K; i += kMergeWarps * 32) {
            const uint64_t x = mlists[i];
            if (x >= bound) {
                const unsigned slot = atomicAdd(&nsurv_s, 1u);
                if (slot < kMergeSurvivors) surv[slot] = x;
            }
        }
    }
    __syncthreads();
    const unsigned ns = nsurv_s;
    uint64_t run = 0;
    if (bound != 0 && ns <= kMergeSurvivors) {
        const unsigned nb = (ns + 31) / 32;  // batches of 32 survivors
        if (static_cast<unsigned>(warp) < nb) {
            const unsigned i = warp * 32 + lane;
            const uint64_t x = warp_sort_desc(i < ns ? surv[i] : 0ull, lane);
            wl[warp][lane] = x;
        }
        __syncthreads();
        if (warp == 0) {
            run = nb > 0 ? wl[0][lane] : 0ull;
            if (lane >= K) run = 0;
            for (unsigned w = 1; w < nb; ++w) run = list_merge(run, wl[w][lane], lane, K);
        }
    } else {
        for (int g = warp; g < G; g += kMergeWarps) {
            const uint64_t x = (lane < K) ? mlists[g * K + lane] : 0ull;
            run = list_merge(run, x, lane, K);
        }
        wl[warp][lane] = run;
        __syncthreads();
        for (int step = 1; step < kMergeWarps; step <<= 1) {
            if ((warp & (2 * step - 1)) == 0) {
                run = list_merge(run, wl[warp + step][lane], lane, K);
                wl[warp][lane] = run;
            }
            __syncthreads();
        }
    }
    if (warp == 0) merge_emit(col, run, lane, K, ids_ws, vals_ws, ids_out, vals_out, keys_out, dd, threadIdx.x == 0);
    if (dd.tab && col == 0 && threadIdx.x == 64) *dd.count = 0;  // the compaction runs after this kernel
}

// Few lists per position (G <= 32, e.g. the 10 CTAs of a 256-wide tile at
// the stress shape, or a few vocabulary shards): one warp per position folds
// the G lists in order, sixteen positions per CTA.
__global__ void __launch_bounds__(kMergeWarps * 32) topk_merge_small_kernel(
    const uint64_t *__restrict__ part, int G, int N, int K, int32_t *ids_ws, float *vals_ws, int32_t *ids_out,
    float *vals_out, uint64_t *thr_g, uint64_t *keys_out, const DedupParams dd)
{
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = blockIdx.x * kMergeWarps + warp;
    if (dd.tab && blockIdx.x == 0 && threadIdx.x == 0) *dd.count = 0;  // the compaction runs after this kernel
    if (col >= N) return;
    if (lane == 0) thr_g[col] = 0;  // ready for the next lm_head pass
    uint64_t x[32];
#pragma unroll
    for (int g = 0; g < 32; ++g)  // every load issued before the first merge
        x[g] = (g < G && lane < K) ? part[(static_cast<size_t>(g) * N + col) * K + lane] : 0ull;
    uint64_t run = 0;
#pragma unroll
    for (int g = 0; g < 32; ++g)
        if (g < G) run = list_merge(run, x[g], lane, K);
    pdl_trigger();  // the lists are read (warps past N count as triggered when they exit)
    merge_emit(col, run, lane, K, ids_ws, vals_ws, ids_out, vals_out, keys_out, dd, lane == 0);
}

}  // namespace

cudaError_t prepare_topk_merge(int smem_optin)
{
    cudaError_t e = set_max_dynamic_smem(topk_merge_kernel<16>, smem_optin);
    if (e != cudaSuccess) return e;
    return set_max_dynamic_smem(topk_merge_kernel<32>, smem_optin);
}

cudaError_t launch_topk_merge(const uint64_t *part, int G, int N, int K, int32_t *ids_ws, float *vals_ws,
                              int32_t *ids_out, float *vals_out, uint64_t *thr_g, cudaStream_t s, uint64_t *keys_out,
                              const DedupParams &dd, size_t min_smem)
{
    if (G <= 32)
        return launch_ex(topk_merge_small_kernel, dim3((N + kMergeWarps - 1) / kMergeWarps), dim3(kMergeWarps * 32), 0,
                         s, 1, part, G, N, K, ids_ws, vals_ws, ids_out, vals_out, thr_g, keys_out, dd);
    const size_t need = static_cast<size_t>(G) * K * sizeof(uint64_t);
    const size_t smem = need > min_smem ? need : min_smem;
    if (K == 16)
        return launch_ex(topk_merge_kernel<16>, dim3(N), dim3(kMergeWarps * 32), smem, s, 1, part, G, N, ids_ws,
                         vals_ws, ids_out, vals_out, thr_g, keys_out, dd);
    return launch_ex(topk_merge_kernel<32>, dim3(N), dim3(kMergeWarps * 32), smem, s, 1, part, G, N, ids_ws, vals_ws,
                     ids_out, vals_out, thr_g, keys_out, dd);
}

}  // namespace dfl
