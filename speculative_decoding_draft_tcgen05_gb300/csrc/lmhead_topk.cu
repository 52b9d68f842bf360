// Fused lm_head GEMM + streaming top-K for the DFlash 2 path selector.
//
// Blog "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path
// Selector": the selector keeps the drafter's 16 best candidates per draft
// position, ranked by the drafter's own logit U_t(b) = W[b] . h_t, and gates
// the pair score with H(h_t). Both are products of a [rows, d] weight with the
// hidden states, so one kernel computes them from the same weight stream:
//   - vocabulary tiles (128 rows of W) feed a running top-K per position;
//   - two extra tiles (the 256 rows of W_H) write the gate g_t = W_H h_t.
// The full logits never reach global memory.
//
// Swap-AB tcgen05 GEMM: the 128 weight rows of a tile are the MMA's M (TMEM
// lanes), the NT positions of an n-tile are N (TMEM columns), K = d is
// streamed 64 columns per stage by TMA into 128-byte-swizzled shared memory.
// Warp roles per CTA (persistent, one CTA per SM):
//   warp 0      TMA producer (one thread), `stages`-deep ring
//   warp 1      TMEM owner and MMA issuer (one thread), two or four
//               accumulators
//   warps 2..9  epilogue: TMEM -> registers -> per-position threshold filter
//               -> the survivors into per-position sorted lists (warp-sorted
//               merges while the lists fill, one thread per position after)
// Each CTA owns one n-tile and every ctas_per_ntile-th M tile; it writes one
// sorted partial list of K keys per position, merged by topk_merge.cu.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr uint32_t kTileABytes = kLmTileM * kLmTileK * 2;  // 16 KB
constexpr uint32_t kTransposeBytes = 16 * kLmTileM * 4;    // 16 columns x 128 rows fp32
// Up to this many surviving keys per warp are inserted one by one; more are
// sorted and merged (a sort + merge costs about as much as 6 to 8 inserts).
constexpr int kInsertLimit = 6;
// Keys the per-tile path can hold per tile (buckets over the transpose buffer).
constexpr int kBucketKeys = static_cast<int>(kTransposeBytes / 8);
// Survivors beyond a position's bucket go to a small pool shared by all
// positions (over the chunked path's row scratch, which the per-tile path does
// not use); only a full pool sends the tile through the chunked path.
constexpr int kPoolKeys = 64;
// First tile (per CTA) that takes the per-tile path. Nearly every logit of
// the first tile passes (the lists are empty), and many of the second at 100+
// positions (more than the buckets hold): both go through the chunked path.
#ifndef DFL_LM_FAST_FROM
#define DFL_LM_FAST_FROM 2
#endif
// Widest position tile that takes the per-tile path (measured at the 256-wide
// tiles of 3840 positions: lm_head 2834 -> 2568 us at K = 16, 3417 -> 3074 us
// at K = 32, against the chunked path throughout).
#ifndef DFL_LM_FAST_MAXNT
#define DFL_LM_FAST_MAXNT 256
#endif

// Inserts the keys bk[s * bstride] (s < n) that exceed th into the sorted list
// l[i * LS] (i < KK, descending) of one position, in registers; th rises to
// the list's K-th key as it fills. Returns whether the list changed; kth is
// its K-th key afterwards.
template <int KK>
__device__ __forceinline__ bool insert_into_list(uint64_t *l, int LS, const uint64_t *bk, int bstride, int n,
                                                 uint64_t &th, uint64_t &kth)
{
    uint64_t y[KK];
#pragma unroll
    for (int i = 0; i < KK; ++i) y[i] = l[i * LS];
    bool dirty = false;
    for (int s2 = 0; s2 < n; ++s2) {
        const uint64_t x = bk[s2 * bstride];
        if (x <= th) continue;
        // keys are distinct: the ones below x move down one place
#pragma unroll
        for (int i = KK - 1; i > 0; --i) y[i] = y[i - 1] < x ? y[i - 1] : (y[i] < x ? x : y[i]);
        y[0] = y[0] < x ? x : y[0];
        th = y[KK - 1] > th ? y[KK - 1] : th;
        dirty = true;
    }
    if (dirty) {
#pragma unroll
        for (int i = 0; i < KK; ++i) l[i * LS] = y[i];
    }
    kth = y[KK - 1];
    return dirty;
}

// v[jj] for a runtime jj in [0, 16), by a select tree on the bits of jj (an
// indexed read would move the register array to local memory).
__device__ __forceinline__ float pick16(const float (&v)[16], int jj)
{
    float a[8], b[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (jj & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (jj & 2) ? a[2 * i + 1] : a[2 * i];
    const float c0 = (jj & 4) ? b[1] : b[0], c1 = (jj & 4) ? b[3] : b[2];
    return (jj & 8) ? c1 : c0;
}

__device__ __forceinline__ void named_bar_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over the epilogue warps that also ORs a predicate across them, so
// that every epilogue thread takes the same abort decision.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Independent accumulation chains per tile. Consecutive MMAs into the same
// accumulator wait for each other, so with few positions (narrow N) one chain
// leaves the tensor pipe idle between MMAs; k-step k of a tile goes to chain
// k mod C and the epilogue adds the C partial sums. Two tiles' worth (double
// buffering) of C chains must fit the 512 TMEM columns.
__host__ __device__ inline int acc_chains(int NT)
{
#ifdef DFL_LM_CHAINS
    return NT * DFL_LM_CHAINS <= 256 ? DFL_LM_CHAINS : 1;
#else
    (void)NT;
    return 1;  // measured: more chains do not speed up the weight stream at N <= 64
#endif
}

// Accumulator buffers in TMEM: four where they fit in the 512 columns, so that
// the MMAs can run up to three tiles ahead of the epilogue (the first tiles of
// a CTA, whose lists start empty, take the epilogue longer than a tile of the
// weight stream), else two.
__host__ __device__ inline int acc_buffers(int NT)
{
#ifdef DFL_LM_ACC_BUFS
    const int want = DFL_LM_ACC_BUFS;
#else
    const int want = 4;
#endif
    return want * acc_chains(NT) * NT <= 512 ? want : 2;
}

__host__ __device__ inline uint32_t tmem_cols_for(int NT)
{
    uint32_t need = static_cast<uint32_t>(acc_buffers(NT) * acc_chains(NT) * NT), c = 32;
    while (c < need) c <<= 1;
    return c;
}

struct Layout {
    uint32_t stage_bytes, off_T, off_wscr, off_list, off_thr, off_thrf, off_rb, off_flags, off_cmask, off_ccnt, off_bar,
        total;
};

// hrows: hidden rows a stage holds (NT, or NT / 2 in a CTA pair, which splits
// the positions of a tile between its two CTAs)
__host__ __device__ inline Layout make_layout(int NT, int K, int stages, int boxes, int hrows)
{
    Layout l;
    l.stage_bytes = static_cast<uint32_t>(boxes) * (kTileABytes + static_cast<uint32_t>(hrows) * kLmTileK * 2);
    l.off_T = stages * l.stage_bytes;
    l.off_wscr = l.off_T + kTransposeBytes;
    l.off_list = l.off_wscr + 8 * kLmTileM;  // eight epilogue warps x 128 row indices
    // lists: entry i of position c at [i * (NT + 1) + c] (odd row length: a warp
    // reading one list and a thread per position both avoid bank conflicts)
    l.off_thr = l.off_list + static_cast<uint32_t>(NT + 1) * K * 8;
    l.off_thrf = l.off_thr + static_cast<uint32_t>(NT) * 8;
    l.off_rb = l.off_thrf + static_cast<uint32_t>(NT) * 4;
    l.off_flags = l.off_rb + static_cast<uint32_t>(NT) * 8;
    l.off_cmask = l.off_flags + 32;  // flag words 0..2, overflow flags 4..5
    l.off_ccnt = l.off_cmask + 16 * 4 * 4;
    l.off_bar = l.off_ccnt + static_cast<uint32_t>(NT) * 4;
    // full[S], empty[S], tfull[4], tempty[4], drain, then tmem base + abort flag
    l.total = l.off_bar + 8u * (2u * stages + 9u) + 16u;
    return l;
}

// kPair: a cluster of two CTAs computes one 256-row tile (cta_group::2 MMAs
// issued by the even CTA): each CTA holds 128 weight rows and half of the
// tile's positions in its shared memory, and receives its 128 rows x NT
// accumulator in its own tensor memory.
template <bool kPair>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_topk_kernel(const __grid_constant__ LmHeadParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzled tiles need 1024 B alignment
    uint8_t *const gbase = smem_raw + (base - raw);

    const int NT = p.NT, K = p.K, S = p.stages;
    const int BX = p.boxes;  // 64-column boxes per stage
    const int HR = kPair ? NT / 2 : NT;  // hidden rows of a stage in this CTA
    const Layout lay = make_layout(NT, K, S, BX, HR);
    const uint32_t w_bytes = static_cast<uint32_t>(BX) * kTileABytes;  // weight part of a stage
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;               // 0: issues the pair's MMAs
    float *const T = reinterpret_cast<float *>(gbase + lay.off_T);
    uint8_t *const wscr = gbase + lay.off_wscr;
    uint64_t *const lists = reinterpret_cast<uint64_t *>(gbase + lay.off_list);
    uint64_t *const thr = reinterpret_cast<uint64_t *>(gbase + lay.off_thr);
    // per position: the logit of the K-th best key so far (-inf until K are held)
    float *const thr_f = reinterpret_cast<float *>(gbase + lay.off_thrf);
    // per position: a threshold from the other CTAs' best logits (see below)
    uint64_t *const rb = reinterpret_cast<uint64_t *>(gbase + lay.off_rb);
    // per 16-column chunk: which columns have a surviving logit (3 rotating words)
    volatile uint32_t *const chunk_flags = reinterpret_cast<volatile uint32_t *>(gbase + lay.off_flags);
    // per column of the current chunk and TMEM lane quadrant: the tile rows whose
    // logit passes the column's float threshold
    uint32_t *const cmask = reinterpret_cast<uint32_t *>(gbase + lay.off_cmask);
    // per-tile path: survivor keys by position (key s of position c at [s * NT + c],
    // over the transpose buffer), their counts, and an overflow flag per tile parity
    uint64_t *const bucket = reinterpret_cast<uint64_t *>(T);
    uint32_t *const col_cnt = reinterpret_cast<uint32_t *>(gbase + lay.off_ccnt);
    volatile uint32_t *const ovf = chunk_flags + 4;
    uint64_t *const pool_key = reinterpret_cast<uint64_t *>(wscr);                  // [kPoolKeys]
    uint16_t *const pool_col = reinterpret_cast<uint16_t *>(wscr + 8 * kPoolKeys);  // [kPoolKeys]
    volatile uint32_t *const pool_cnt = chunk_flags + 6;                            // per tile parity
    const uint32_t bar_full = base + lay.off_bar;
    const uint32_t bar_empty = bar_full + 8u * S;
    const uint32_t bar_tfull = bar_empty + 8u * S;
    const uint32_t bar_tempty = bar_tfull + 32u;
    const uint32_t bar_drain = bar_tempty + 32u;
    uint32_t *const tmem_holder = reinterpret_cast<uint32_t *>(gbase + lay.off_bar + 8u * (2u * S + 9u));
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a pair (CTAs 2i, 2i + 1) shares its position tile; chunk = the CTA's index
    // among the CTAs of its position tile (its partial lists' slot)
    const int n_tile = kPair ? static_cast<int>(blockIdx.x >> 1) % p.n_tiles_n : blockIdx.x % p.n_tiles_n;
    const int chunk = kPair ? (static_cast<int>(blockIdx.x >> 1) / p.n_tiles_n) * 2 + static_cast<int>(blockIdx.x & 1)
                            : blockIdx.x / p.n_tiles_n;
    const int G = p.ctas_per_ntile;
    const bool pilot = !kPair && p.pilot_stride > 0;
    // this CTA's tiles: chunk, chunk + G, ... (a pilot CTA: chunk * pilot_stride
    // only; a pair: the two halves 2 q + rank of the pair's 256-row tiles q)
    const int m_first = kPair ? chunk / 2 : (pilot ? chunk * p.pilot_stride : chunk);
    const int m_step = kPair ? G / 2 : (pilot ? p.m_tiles_total : G);
    const int n_my_tiles = kPair ? (p.m_tiles_total / 2 - m_first + m_step - 1) / m_step
                                 : (pilot ? 1 : (p.m_tiles_total - chunk + G - 1) / G);
    // the 128-row weight tile of this CTA's i-th tile (a pair's m_tiles_total is even)
    auto tile_at = [&](int i) {
        return kPair ? 2 * (m_first + i * m_step) + static_cast<int>(rank) : m_first + i * m_step;
    };
    const int KB = p.d / (kLmTileK * BX);
    const uint32_t tmem_cols = tmem_cols_for(NT);
    const int C = acc_chains(NT);
    const int NA = acc_buffers(NT);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int a = 0; a < 4; ++a) {
            mbar_init(bar_tfull + 8u * a, 1);
            mbar_init(bar_tempty + 8u * a, kPair ? 256 : 128);  // a pair: both CTAs' TMEM readers
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    const int LS = NT + 1;  // row length of the lists
    for (int i = threadIdx.x; i < LS * K; i += kLmThreads) lists[i] = 0;
    for (int i = threadIdx.x; i < NT; i += kLmThreads) col_cnt[i] = 0;
    for (int i = threadIdx.x; i < NT; i += kLmThreads) {
        thr[i] = 0;
        thr_f[i] = -INFINITY;
    }
    if (threadIdx.x < 8) chunk_flags[threadIdx.x] = 0;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_w);
        tma_prefetch_desc(&p.tm_gate);
        tma_prefetch_desc(&p.tm_h);
    }
    if (warp == 1) {
        __syncwarp();
        if constexpr (kPair) {
            tmem_alloc_pair(smem_u32(tmem_holder), tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // the even CTA's barriers are initialised before any use
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_holder);
    // The set-up above overlaps the previous kernel on the stream. Hidden
    // states, the partial lists and the gate are touched only after it has
    // finished (griddepcontrol.wait); the constant weights may be read before.
    pdl_trigger();
    if (!(warp == 0 && lane == 0)) pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
#ifdef DFL_LM_NOHINT
            const uint64_t pol_w = l2_policy_evict_normal();
#else
            // weights: streamed once; a pilot's rows are read again by the main pass
            const uint64_t pol_w = pilot ? l2_policy_evict_last() : l2_policy_evict_first();
#endif
            const uint64_t pol_h = l2_policy_evict_last();   // hidden: re-read by every CTA
            const int total = n_my_tiles * KB;
            // the first ring's weight tiles go out before the wait (the ring
            // starts empty, so no slot has to be waited for)
            const int pre = total < S ? total : S;
            // a pair counts both CTAs' bytes on the even CTA's barriers
            const uint32_t tx_bytes = kPair ? 2u * lay.stage_bytes : lay.stage_bytes;
            const int hrow0 = n_tile * NT + static_cast<int>(rank) * HR;
            auto load = [&](uint32_t dst, const CUtensorMap *tm, int x, int y, uint32_t bar, uint64_t pol) {
                if constexpr (kPair)
                    tma_load_2d_pair(dst, tm, x, y, mapa_shared(bar, 0), pol);
                else
                    tma_load_2d(dst, tm, x, y, bar, pol);
            };
            for (int it = 0; it < pre; ++it) {
                const int m = tile_at(it / KB), kb = it % KB;
                const bool gate = m >= p.m_tiles_vocab;
                const int row0 = (gate ? m - p.m_tiles_vocab : m) * kLmTileM;
                if (rank == 0) mbar_arrive_expect_tx(bar_full + 8u * it, tx_bytes);
                for (int bx = 0; bx < BX; ++bx)
                    load(base + it * lay.stage_bytes + bx * kTileABytes, gate ? &p.tm_gate : &p.tm_w,
                         (kb * BX + bx) * kLmTileK, row0, bar_full + 8u * it, pol_w);
            }
            pdl_wait();
            for (int it = 0; it < pre; ++it)
                for (int bx = 0; bx < BX; ++bx)
                    load(base + it * lay.stage_bytes + w_bytes + bx * HR * kLmTileK * 2, &p.tm_h,
                         ((it % KB) * BX + bx) * kLmTileK, hrow0, bar_full + 8u * it, pol_h);
            int it = pre;
            bool ok = true;
            for (; ok && it < total; ++it) {
                const int m = tile_at(it / KB), kb = it % KB;
                const bool gate = m >= p.m_tiles_vocab;
                const CUtensorMap *tma = gate ? &p.tm_gate : &p.tm_w;
                const int row0 = (gate ? m - p.m_tiles_vocab : m) * kLmTileM;
                const int s = it % S;
                const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
                if (!mbar_wait(bar_empty + 8u * s, ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = base + s * lay.stage_bytes;
                if (rank == 0) mbar_arrive_expect_tx(bar_full + 8u * s, tx_bytes);
                for (int bx = 0; bx < BX; ++bx)
                    load(sa + bx * kTileABytes, tma, (kb * BX + bx) * kLmTileK, row0, bar_full + 8u * s, pol_w);
                for (int bx = 0; bx < BX; ++bx)
                    load(sa + w_bytes + bx * HR * kLmTileK * 2, &p.tm_h, (kb * BX + bx) * kLmTileK, hrow0,
                         bar_full + 8u * s, pol_h);
            }
            if (!ok) {
                atomicOr(p.err, DEV_ERR_TIMEOUT);
                // let the copies already issued land before the CTA can exit
                if (rank == 0) {
                    for (int j = (it > S ? it - S : 0); j < it; ++j)
                        mbar_wait(bar_full + 8u * (j % S), static_cast<uint32_t>(j / S) & 1u, abort_flag, false);
                } else {
                    // the odd CTA of a pair cannot observe its copies (they are
                    // counted on the even CTA's barriers): a copy lands within
                    // microseconds, so it waits 100 us
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 100000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (a pair: the even CTA's)
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * kLmTileM : kLmTileM, NT);
            int it = 0, j = 0;
            bool ok = true;
            for (; ok && j < n_my_tiles; ++j) {
                const int a = j % NA;
                const uint32_t u = static_cast<uint32_t>(j / NA);
                const bool got = kPair ? mbar_wait_cluster(bar_tempty + 8u * a, (u & 1u) ^ 1u, abort_flag)
                                       : mbar_wait(bar_tempty + 8u * a, (u & 1u) ^ 1u, abort_flag);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * C * NT);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
                    const bool full = kPair ? mbar_wait_cluster(bar_full + 8u * s, ph, abort_flag)
                                            : mbar_wait(bar_full + 8u * s, ph, abort_flag);
                    if (!full) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + s * lay.stage_bytes;
                    const uint32_t sb = sa + w_bytes;
                    for (int bx = 0; bx < BX; ++bx) {
#pragma unroll
                        for (int k = 0; k < kLmTileK / 16; ++k) {
                            const int ks = bx * (kLmTileK / 16) + k;  // k-step within the stage
                            const uint64_t ad = smem_desc_sw128(sa + bx * kTileABytes + 32u * k);
                            const uint64_t bd = smem_desc_sw128(sb + bx * HR * kLmTileK * 2 + 32u * k);
                            const uint32_t acc = (kb > 0 || ks >= C) ? 1u : 0u;
                            if constexpr (kPair)
                                umma_bf16_pair(d_tmem + static_cast<uint32_t>((ks % C) * NT), ad, bd, idesc, acc);
                            else
                                umma_bf16(d_tmem + static_cast<uint32_t>((ks % C) * NT), ad, bd, idesc, acc);
                        }
                    }
                    // frees the stage (both CTAs' halves) once these MMAs have read it
                    if constexpr (kPair)
                        umma_commit_pair(bar_empty + 8u * s, 3);
                    else
                        umma_commit(bar_empty + 8u * s);
                }
                if (ok) {
                    if constexpr (kPair)
                        umma_commit_pair(bar_tfull + 8u * a, 3);
                    else
                        umma_commit(bar_tfull + 8u * a);
                }
            }
            if (!ok) atomicOr(p.err, DEV_ERR_TIMEOUT);
            // every MMA must be finished before TMEM is released
            if constexpr (kPair)
                umma_commit_pair(bar_drain, 1);
            else
                umma_commit(bar_drain);
            mbar_wait(bar_drain, 0, abort_flag, false);
        }
    } else {
        // ------------------------------------------------ epilogue
        // Warps 2..5 read TMEM in the chunked path and release each
        // accumulator (warp w may only touch lane quadrant w % 4); in the
        // per-tile path warps 6..9 read it too, from the same quadrants. All
        // eight share the per-position list work and meet at named barrier 1.
        const bool tmem_warp = warp < 6;
        const int ew = warp - 2;           // 0..7: column share
        const int q = warp & 3;            // TMEM lane quadrant
        const int row = q * 32 + lane;     // tile row owned by this thread when it reads TMEM
        const int et = threadIdx.x - 64;   // 0..255 among the epilogue threads
        const int col_base = n_tile * NT;
        const int nvalid = min(NT, p.N - col_base);
        const int ncols16 = (nvalid + 15) & ~15;
        int j = 0;
        int nchunk = 0;  // top-K chunks processed so far (selects the flag word)
        bool ok = true;
        const int fast_from = p.pmax_n > 0 ? 0 : DFL_LM_FAST_FROM;
        // hands accumulator a back to the MMA warp (a pair: to the even CTA's)
        auto release_acc = [&](int a) {
            if constexpr (kPair)
                mbar_arrive_remote(mapa_shared(bar_tempty + 8u * a, 0));
            else
                mbar_arrive(bar_tempty + 8u * a);
        };
        for (; j < n_my_tiles; ++j) {
            const int m = tile_at(j);
            const int a = j % NA;
            const uint32_t u = static_cast<uint32_t>(j / NA);
            const bool gate = m >= p.m_tiles_vocab;
            // the overflow flag of the next tile: every thread read it (as the
            // flag of tile j - 1) before the barriers that ended that tile
            if (threadIdx.x == 64) {
                ovf[(j + 1) & 1] = 0;
                pool_cnt[(j + 1) & 1] = 0;
            }
            // the cross-CTA thresholds, fetched while the accumulator fills
            uint64_t tg[2] = {0ull, 0ull};
            if (!gate) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (et + h * 256 < nvalid)
                        tg[h] = *reinterpret_cast<volatile const uint64_t *>(p.thr_g + col_base + et + h * 256);
            }
            // Used where the list upkeep is the bottleneck (many positions per
            // CTA, measured: from about 100) and the n-tile has enough CTAs to
            // give K maxima.
            // The pilot's maxima take the same path at the first tile.
            const bool from_pilot = p.pmax_n > 0 && !gate && j == 0;
            const bool refresh = from_pilot || (p.tmax && !gate && j == 2 && G >= 2 * K && nvalid >= 96);
            const uint64_t *const rsrc = from_pilot ? p.pmax : p.tmax;
            const int nsrc = from_pilot ? p.pmax_n : G;
            if (refresh) {
                // Every CTA of this n-tile published its best logit per position
                // after its first tile. If at least K of them are >= v, then K
                // logits are >= v, so v bounds the K-th best from below: far
                // higher than any one CTA's K-th best this early. Each lane takes
                // the best of its share of the CTAs; v = the K-th best lane.
                for (int col = ew; col < nvalid; col += 8) {
                    uint64_t t[5];  // G <= 160 CTAs per n-tile: at most 5 per lane
#pragma unroll
                    for (int u2 = 0; u2 < 5; ++u2) {
                        const int g2 = lane + 32 * u2;
                        t[u2] = g2 < nsrc ? __ldcg(rsrc + static_cast<size_t>(g2) * p.N + col_base + col) : 0ull;
                    }
                    uint32_t best = 0;
#pragma unroll
                    for (int u2 = 0; u2 < 5; ++u2) {
                        const uint32_t o = static_cast<uint32_t>(t[u2]);
                        if (static_cast<uint32_t>(t[u2] >> 32) == p.epoch && o > best) best = o;
                    }
                    const uint32_t srt = warp_sort_desc_u32(best, lane);
                    const uint64_t kth = __shfl_sync(0xFFFFFFFFu, srt, K - 1);
                    if (lane == 0) rb[col] = kth << 32;  // any key of that logit value or above passes
                }
            }
            const bool got = !tmem_warp ? true
                             : kPair    ? mbar_wait_cluster(bar_tfull + 8u * a, u & 1u, abort_flag)
                                        : mbar_wait(bar_tfull + 8u * a, u & 1u, abort_flag);
            if (refresh) named_bar_sync(1, 256);
            if (!gate) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = et + h * 256;
                    if (c < nvalid) {
                        const uint64_t t = refresh && rb[c] > tg[h] ? rb[c] : tg[h];
                        if (t > thr[c]) {
                            thr[c] = t;
                            thr_f[c] = key_val(t);
                        }
                    }
                }
            }
            if (named_bar_or(1, 256, !got)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * C * NT);
            const int row0 = (gate ? m - p.m_tiles_vocab : m) * kLmTileM;
            bool released = false;  // the accumulator is handed back to the MMA warp
            const int capc = kBucketKeys / NT;  // keys per position and tile
            if (pilot) {
                // The pilot: per position, the best logit of this tile (rows past
                // V count as nothing), one warp reduction per column and quadrant.
                uint32_t *const qmax = reinterpret_cast<uint32_t *>(T);  // [4][NT]
                if (tmem_warp) {
                    const bool rowok = static_cast<int64_t>(row0) + row < p.V;
                    for (int c0 = 0; c0 < ncols16; c0 += 16) {
                        float v[16];
                        __syncwarp();
                        tmem_load16(taddr + static_cast<uint32_t>(c0), v);
                        for (int c = 1; c < C; ++c) {
                            float w[16];
                            tmem_load16(taddr + static_cast<uint32_t>(c * NT + c0), w);
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) v[jj] += w[jj];
                        }
                        uint32_t mine = 0;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const uint32_t o = __reduce_max_sync(0xFFFFFFFFu, rowok ? f32_to_ordered(v[jj]) : 0u);
                            if (lane == jj) mine = o;
                        }
                        if (lane < 16 && c0 + lane < nvalid) qmax[q * NT + c0 + lane] = mine;
                    }
                    tc_fence_before_sync();
                    release_acc(a);
                }
                named_bar_sync(1, 256);
                for (int c = et; c < nvalid; c += 256) {
                    uint32_t best = qmax[c];
#pragma unroll
                    for (int qq = 1; qq < 4; ++qq) best = max(best, qmax[qq * NT + c]);
                    p.pmax[static_cast<size_t>(chunk) * p.N + col_base + c] = (static_cast<uint64_t>(p.epoch) << 32) | best;
                }
                continue;
            }
            if (!gate && j >= fast_from && NT >= 32 && NT <= DFL_LM_FAST_MAXNT) {
                // Once the lists are warm few logits pass. All eight warps read
                // the tile (warps w and w + 4 share a lane quadrant, each takes
                // every other 16-column chunk), file the survivors by position,
                // and then one thread per position inserts them into its list:
                // no per-chunk barriers. A tile with more survivors at a position
                // than the buckets hold goes through the chunked path below (its
                // accumulator is still held).
                {
                    const bool rowok = static_cast<int64_t>(row0) + row < p.V;
                    const float4 *const thr4 = reinterpret_cast<const float4 *>(thr_f);
                    for (int ci = ew >> 2; ci * 16 < ncols16; ci += 2) {
                        const int c0 = ci * 16;
                        float v[16];
                        __syncwarp();
                        tmem_load16(taddr + static_cast<uint32_t>(c0), v);
                        for (int c = 1; c < C; ++c) {  // the other chains' partial sums, in chain order
                            float w[16];
                            tmem_load16(taddr + static_cast<uint32_t>(c * NT + c0), w);
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) v[jj] += w[jj];
                        }
                        const int vcols = nvalid - c0;
                        uint32_t pm = 0;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float4 t4 = thr4[(c0 >> 2) + q4];
                            const float tt[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int jj = q4 * 4 + e;
                                if (jj < vcols && v[jj] >= tt[e]) pm |= 1u << jj;
                            }
                        }
                        if (!rowok) pm = 0;
                        while (pm) {  // rare: a few survivors per tile and position
                            const int jj = __ffs(pm) - 1;
                            pm &= pm - 1;
                            const int col = c0 + jj;
                            const uint32_t slot = atomicAdd(col_cnt + col, 1u);
                            const uint64_t key = make_key(pick16(v, jj), p.id_base + static_cast<uint32_t>(row0 + row));
                            if (slot < static_cast<uint32_t>(capc)) {
                                bucket[slot * NT + col] = key;
                            } else {
                                const uint32_t ps = atomicAdd(const_cast<uint32_t *>(&pool_cnt[j & 1]), 1u);
                                if (ps < static_cast<uint32_t>(kPoolKeys)) {
                                    pool_key[ps] = key;
                                    pool_col[ps] = static_cast<uint16_t>(col);
                                } else {
                                    ovf[j & 1] = 1;
                                }
                            }
                        }
                    }
                }
                tc_fence_before_sync();
                named_bar_sync(1, 256);
                int nsurv = 0;
                if (et < nvalid) {
                    nsurv = static_cast<int>(col_cnt[et]);
                    col_cnt[et] = 0;  // only this thread touches it until the next tile's filter
                }
                if (ovf[j & 1] == 0) {  // uniform: all read the same flag
                    released = true;
                    if (tmem_warp) release_acc(a);
                    if (nsurv > 0) {  // thread et owns position et
                        const int c = et;
                        uint64_t th = thr[c], kth = 0;
                        const int nb = nsurv < capc ? nsurv : capc;
                        bool dirty = K == 16 ? insert_into_list<16>(lists + c, LS, bucket + c, NT, nb, th, kth)
                                             : insert_into_list<32>(lists + c, LS, bucket + c, NT, nb, th, kth);
                        if (nsurv > capc) {  // the rest of this position's survivors are in the pool
                            const uint32_t np = pool_cnt[j & 1];
                            for (uint32_t i = 0; i < np; ++i) {
                                if (pool_col[i] != c) continue;
                                dirty |= K == 16 ? insert_into_list<16>(lists + c, LS, pool_key + i, 1, 1, th, kth)
                                                 : insert_into_list<32>(lists + c, LS, pool_key + i, 1, 1, th, kth);
                            }
                        }
                        if (dirty) {
                            thr[c] = th;
                            thr_f[c] = th ? key_val(th) : -INFINITY;
                            if (kth) atomicMax(reinterpret_cast<unsigned long long *>(p.thr_g + col_base + c),
                                               static_cast<unsigned long long>(kth));
                        }
                    }
                    named_bar_sync(1, 256);  // lists and thresholds complete for the next tile
                }
            }
            // the chunked path: the first tile(s), W_H tiles and overflowing tiles
            for (int c0 = 0; !released && c0 < ncols16; c0 += 16) {
                float v[16];
                if (tmem_warp) {
                    __syncwarp();
                    tmem_load16(taddr + static_cast<uint32_t>(c0), v);
                    for (int c = 1; c < C; ++c) {  // the other chains' partial sums, in chain order
                        float w[16];
                        tmem_load16(taddr + static_cast<uint32_t>(c * NT + c0), w);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[jj] += w[jj];
                    }
                }
                if (gate) {
                    if (tmem_warp) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int pos = col_base + c0 + jj;
                            if (c0 + jj < nvalid) p.gate[static_cast<size_t>(pos) * kEmbed + row0 + row] = v[jj];
                        }
                    }
                    continue;
                }
                // Cheap filter first: a logit can only enter a list if it is
                // not below that position's threshold (the larger of this
                // CTA's K-th best and the best K-th published by any CTA: at
                // least K logits reach it). Exact ties are settled by the full
                // key below. Chunks where nothing survives end here.
                const int slot = nchunk % 3;
                ++nchunk;
                uint32_t mask = 0;
                if (tmem_warp) {
                    const bool rowok = static_cast<int64_t>(row0) + row < p.V;
                    const int vcols = nvalid - c0;
                    uint32_t mine_cols = 0;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const unsigned b = __ballot_sync(0xFFFFFFFFu, rowok && jj < vcols && v[jj] >= thr_f[c0 + jj]);
                        if (lane == jj) mine_cols = b;
                        mask |= (b ? 1u : 0u) << jj;  // uniform across the warp
                    }
                    if (lane < 16) cmask[lane * 4 + q] = mine_cols;
                }
                if (lane == 0 && mask) atomicOr(const_cast<uint32_t *>(&chunk_flags[slot]), mask);
                named_bar_sync(1, 256);
                const uint32_t flags = chunk_flags[slot];
                // the word of the previous chunk is free again: every epilogue
                // thread read it before arriving at the barrier above
                if (threadIdx.x == 64) chunk_flags[(slot + 2) % 3] = 0;
                if (flags == 0) continue;  // uniform: all read the same word
                if (tmem_warp) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) T[jj * kLmTileM + row] = v[jj];
                }
                named_bar_sync(1, 256);
                for (int cc = ew; cc < 16; cc += 8) {
                    const int col = c0 + cc;
                    if (col >= nvalid || !((flags >> cc) & 1u)) continue;  // uniform across the warp
                    uint64_t th = thr[col];
                    // the tile rows that passed the float filter (from the TMEM warps)
                    uint32_t surv[4];
                    int total = 0;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        surv[qq] = cmask[cc * 4 + qq];
                        total += __popc(surv[qq]);
                    }
                    const bool loaded = total > 0;
                    uint64_t mine = 0;
                    if (loaded) mine = (lane < K) ? lists[lane * LS + col] : 0ull;
                    if (total > kInsertLimit) {
                        // many survivors (early tiles): pack their tile rows densely
                        // in this warp's scratch, then rebuild, sort 32 at a time
                        // and merge each batch into the list
                        uint8_t *const scr = wscr + (warp - 2) * kLmTileM;
                        const unsigned lt = (1u << lane) - 1u;
                        int base_i = 0;
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            if ((surv[qq] >> lane) & 1u) scr[base_i + __popc(surv[qq] & lt)] = static_cast<uint8_t>(qq * 32 + lane);
                            base_i += __popc(surv[qq]);
                        }
                        __syncwarp();
                        int nsort = total;
                        if (total > 64) {
                            // The K-th largest of the lanes' maxima (lane l takes
                            // entries l, l + 32, ...) bounds the K-th best of these
                            // logits from below: K lanes hold one at least that
                            // large. The rows below it are dropped before sorting.
                            float lm = -INFINITY;
                            for (int e = lane; e < total; e += 32) lm = fmaxf(lm, T[cc * kLmTileM + scr[e]]);
                            const uint32_t srt = warp_sort_desc_u32(f32_to_ordered(lm), lane);
                            const float bound = ordered_to_f32(__shfl_sync(0xFFFFFFFFu, srt, K - 1));
                            int out = 0;  // compacted in place: writes never pass the entries still to be read
                            for (int e0 = 0; e0 < total; e0 += 32) {
                                const int e = e0 + lane;
                                int r = 0;
                                bool keep = false;
                                if (e < total) {
                                    r = scr[e];
                                    keep = T[cc * kLmTileM + r] >= bound;
                                }
                                const unsigned kb = __ballot_sync(0xFFFFFFFFu, keep);
                                __syncwarp();
                                if (keep) scr[out + __popc(kb & lt)] = static_cast<uint8_t>(r);
                                out += __popc(kb);
                                __syncwarp();
                            }
                            nsort = out;
                        }
                        for (int b0 = 0; b0 < nsort; b0 += 32) {
                            uint64_t x = 0ull;
                            if (b0 + lane < nsort) {
                                const int r = scr[b0 + lane];
                                x = make_key(T[cc * kLmTileM + r], p.id_base + static_cast<uint32_t>(row0 + r));
                            }
                            x = warp_sort_desc(x, lane);
                            mine = list_merge(mine, x, lane, K);
                        }
                        __syncwarp();
                        const uint64_t kth = shfl_u64(mine, K - 1);
                        th = kth > th ? kth : th;
                    } else if (loaded) {
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            unsigned sv = surv[qq];
                            while (sv) {
                                const int r = qq * 32 + __ffs(sv) - 1;
                                sv &= sv - 1;
                                const uint64_t x = make_key(T[cc * kLmTileM + r], p.id_base + static_cast<uint32_t>(row0 + r));
                                if (x > th) {
                                    mine = list_insert(mine, x, lane, K);
                                    const uint64_t kth = shfl_u64(mine, K - 1);
                                    th = kth > th ? kth : th;
                                }
                            }
                        }
                    }
                    if (loaded) {
                        if (lane < K) lists[lane * LS + col] = mine;
                        const uint64_t kth = shfl_u64(mine, K - 1);
                        if (lane == 0) {
                            thr[col] = th;
                            thr_f[col] = th ? key_val(th) : -INFINITY;
                            // publish this CTA's K-th best: K logits are at least that large
                            if (kth) atomicMax(reinterpret_cast<unsigned long long *>(p.thr_g + col_base + col),
                                               static_cast<unsigned long long>(kth));
                        }
                    }
                }
                named_bar_sync(1, 256);
            }
            if (tmem_warp && !released) {
                tc_fence_before_sync();
                release_acc(a);
            }
            if (p.tmax && !gate && j == 0) {
                named_bar_sync(1, 256);  // the first tile's lists are complete
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = et + h * 256;
                    if (c < nvalid)
                        p.tmax[static_cast<size_t>(chunk) * p.N + col_base + c] =
                            (static_cast<uint64_t>(p.epoch) << 32) | (lists[c] >> 32);
                }
            }
        }
        if (!ok) atomicOr(p.err, DEV_ERR_TIMEOUT);
        named_bar_sync(1, 256);
        for (int i = et; !pilot && i < nvalid * K; i += 256) {
            const int col = i / K;
            p.part[(static_cast<size_t>(chunk) * p.N + col_base + col) * K + (i % K)] = lists[(i % K) * LS + col];
        }
    }

    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // the pair's MMAs, copies and arrivals are over in both CTAs
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, tmem_cols);
        else
            tmem_dealloc(tmem_base, tmem_cols);
    }
}

}  // namespace

size_t lmhead_smem_bytes(int NT, int K, int stages, int boxes, int hrows)
{
    return static_cast<size_t>(make_layout(NT, K, stages, boxes, hrows < 0 ? NT : hrows).total) +
           1024;  // + alignment slack
}

int lmhead_boxes(int d, int NT)
{
#ifdef DFL_LM_BOXES
    int b = DFL_LM_BOXES;
#else
    // measured on GB300: two boxes per stage (256 contiguous bytes of every
    // weight row per request) stream the weight ~14% faster than one
    int b = NT <= 128 ? 2 : 1;  // wide position tiles keep one box so three stages still fit
#endif
    while (b > 1 && d % (kLmTileK * b) != 0) --b;
    return b;
}

cudaError_t prepare_lmhead(int smem_optin)
{
    cudaError_t e = set_max_dynamic_smem(lmhead_topk_kernel<false>, smem_optin);
    if (e == cudaSuccess) e = set_max_dynamic_smem(lmhead_topk_kernel<true>, smem_optin);
    return e;
}

cudaError_t launch_lmhead_topk(const LmHeadParams &p, int grid, size_t smem, cudaStream_t s)
{
    return launch_ex(lmhead_topk_kernel<false>, dim3(grid), dim3(kLmThreads), smem, s, 1, p);
}

// CTA pairs along x (blockIdx.x 2i and 2i + 1 form pair i), PDL allowed.
static cudaLaunchConfig_t pair_config(int grid, size_t smem, cudaStream_t s, cudaLaunchAttribute (&attr)[2])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kLmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

cudaError_t launch_lmhead_topk_pair(const LmHeadParams &p, int grid, size_t smem, cudaStream_t s)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(grid, smem, s, attr);
    return cudaLaunchKernelEx(&cfg, lmhead_topk_kernel<true>, p);
}

int lmhead_pair_max_clusters(size_t smem)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(2, smem, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lmhead_topk_kernel<true>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace dfl
