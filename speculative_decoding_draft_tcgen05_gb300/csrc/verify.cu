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
