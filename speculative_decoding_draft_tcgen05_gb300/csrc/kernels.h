// Launch interfaces of the path-selector kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace dfl {

// Bits of the device error word.
enum : int { DEV_ERR_TOKEN = 1, DEV_ERR_TIMEOUT = 2 };

constexpr int kEmbed = 256;  // width of A, B and the context gate

// Launches `kern` with programmatic dependent launch allowed (the kernel may be
// scheduled while its predecessor on the stream finishes; every kernel here
// waits with griddepcontrol.wait before touching data a predecessor wrote) and,
// if cluster_z > 1, thread-block clusters of (1, 1, cluster_z).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_z,
                      Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_z > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = static_cast<unsigned>(cluster_z);
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Lets `kern` use as much dynamic shared memory as the device allows next to
// its static shared memory.
template <typename... KArgs>
cudaError_t set_max_dynamic_smem(void (*kern)(KArgs...), int smem_optin)
{
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_optin - static_cast<int>(fa.sharedSizeBytes));
}

// Sets the shared-memory opt-ins of every kernel on the current device
// (smem_optin = cudaDevAttrMaxSharedMemoryPerBlockOptin).
cudaError_t prepare_lmhead(int smem_optin);
cudaError_t prepare_topk_merge(int smem_optin);
cudaError_t prepare_pair_walk(int smem_optin);

// ---- lm_head GEMM + streaming top-K (and the context gate g = W_H h) ----
constexpr int kLmTileM = 128;   // vocabulary rows per MMA tile (TMEM lanes)
constexpr int kLmTileK = 64;    // hidden columns per pipeline stage (128 B rows)
constexpr int kLmThreads = 320; // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue (TMEM), 6..9 list helpers
#ifndef DFL_LM_MAX_STAGES
#define DFL_LM_MAX_STAGES 8
#endif
constexpr int kLmMaxStages = DFL_LM_MAX_STAGES;  // TMA ring depth cap (shared memory permitting)

struct LmHeadParams {
    CUtensorMap tm_w;     // lm_head W [V, d] bf16, box 64 x 128, 128B swizzle
    CUtensorMap tm_gate;  // W_H [256, d] bf16, box 64 x 128
    CUtensorMap tm_h;     // hidden [N, d] bf16, box 64 x NT
    int64_t V;            // rows of tm_w (a vocabulary shard's rows when id_base > 0)
    uint32_t id_base = 0; // token id of row 0 of tm_w
    int d, N, NT, n_tiles_n, K;
    int m_tiles_vocab, m_tiles_total, ctas_per_ntile, stages;
    int boxes;        // 64-column TMA boxes per pipeline stage (d % (64 * boxes) == 0)
    uint64_t *part;   // [ctas_per_ntile][N][K] partial top-K keys
    float *gate;      // [N][256] g_t = W_H h_t
    uint64_t *thr_g;  // [N] best K-th key published by any CTA; zero on entry, reset by the consumer
    uint64_t *tmax;   // [ctas_per_ntile][N] each CTA's best logit after its first tile, tagged with
                      // `epoch` in the high word (NULL: not used)
    uint32_t epoch;   // differs between consecutive runs on the same tmax
    int *err;
    // Sampled threshold ("pilot"). A pilot launch (pilot_stride > 0) gives each
    // CTA the single vocabulary tile chunk * pilot_stride and publishes only its
    // best logit per position to pmax[chunk][N] (epoch-tagged), nothing else.
    // A main launch with pmax_n > 0 starts every position's threshold at the
    // K-th largest of those pmax_n maxima (K tiles hold a logit at least that
    // large) and takes the per-tile epilogue from its first tile.
    int pilot_stride = 0;
    uint64_t *pmax = nullptr;
    int pmax_n = 0;
};

// hrows: hidden rows per stage (NT; NT / 2 for the CTA-pair kernel)
size_t lmhead_smem_bytes(int NT, int K, int stages, int boxes, int hrows = -1);
int lmhead_boxes(int d, int NT);
cudaError_t launch_lmhead_topk(const LmHeadParams &p, int grid, size_t smem, cudaStream_t s);
// The CTA-pair kernel: one position tile of NT <= 256 positions (tm_h boxes of
// NT / 2 rows), 256-row weight tiles (m_tiles_vocab even: an odd vocabulary
// tile count gets one tile past V, which reads as zeros), grid = 2 x pairs.
cudaError_t launch_lmhead_topk_pair(const LmHeadParams &p, int grid, size_t smem, cudaStream_t s);
// Pairs of the CTA-pair kernel that fit on the device at once (0 if unknown).
int lmhead_pair_max_clusters(size_t smem);

// ---- candidate deduplication (a variant: each distinct token of a batch is projected once) ----
// Gathered row gr of sequence b = gr / R is the anchor x0 (gr % R == 0) or
// candidate gr % R - 1 of the sequence's [L][K] list. The merge marks, per
// token, the first row that holds it: tab[token] = (epoch << 32) | ~row under
// atomicMax, so a newer run's mark always wins and the table needs no reset.
struct DedupParams {
    uint64_t *tab = nullptr;  // [V] marks (NULL: no deduplication)
    unsigned *count = nullptr;  // distinct tokens of the run (reset by the merge)
    int32_t *uniq = nullptr;  // [B * R] the distinct tokens, in the order they were counted
    int32_t *rep = nullptr;   // [B * R] at a token's first row: its index in uniq
    const int32_t *anchor = nullptr;  // [B]
    int *err = nullptr;
    int64_t V = 0;
    int L = 0, K = 0, R = 0;
    uint32_t epoch = 0;
};
// uniq / rep from the marks, one thread per gathered row (R_total rows).
cudaError_t launch_dedup_compact(const DedupParams &d, const int32_t *ids, int R_total, cudaStream_t s);

// Dynamic shared memory that keeps a kernel to at most n CTAs per SM (more
// than 1 / (n + 1) of an SM's shared memory). A grid of at most n waves that
// is launched early (programmatic dependent launch) would otherwise crowd onto
// the SMs its predecessor leaves free; reserving this spreads it over the
// whole GPU as the predecessor's CTAs exit (measured on the merge and the pair
// tables: 3.1 us per step at batch 8 with n = 1, 2.5 us at batch 32 with n = 2).
inline size_t ctas_per_sm_smem(size_t smem_per_sm, int n) { return smem_per_sm / (n + 1) + 1024; }

// Merges the partial lists of every CTA (or of every vocabulary shard: the
// same [G][N][K] layout) into the sorted top-K of each position; keys_out
// (optional) receives the merged keys [N][K]; with dd.tab the merged
// candidates (and the anchors) are marked for deduplication.
// min_smem: dynamic shared memory to reserve at least (see ctas_per_sm_smem).
cudaError_t launch_topk_merge(const uint64_t *part, int G, int N, int K, int32_t *ids_ws,
                              float *vals_ws, int32_t *ids_out, float *vals_out, uint64_t *thr_g, cudaStream_t s,
                              uint64_t *keys_out = nullptr, const DedupParams &dd = DedupParams(),
                              size_t min_smem = 0);

// ---- candidate projections A|B = [W_A; W_B] E[row] (tcgen05, projection.cu) ----
struct ProjParams {
    CUtensorMap tm_wa, tm_wb;     // W_A, W_B [256, d] bf16, box 64 x 256, 128B swizzle
    const uint16_t *E;            // [V, d] bf16 bits
    const int32_t *ids;           // [B, L, K] merged candidates
    const int32_t *anchor;        // [B]
    float *AB;                    // [B * R][512]: cols 0..255 = A, 256..511 = B
    int *err;
    int64_t V;
    int d, L, K, R, R_total;      // gathered row gr: sequence gr / R, row gr % R (0: x0, else a candidate)
    int ksplit;                   // CTAs per output tile along d (1 or 2)
    float *part;                  // [ksplit][R_total][512] partial sums (ksplit > 1)
    unsigned *ticket;             // [row tiles][512 / NC] zero on entry, left zero (ksplit > 1)
    const int32_t *uniq = nullptr;   // deduplicated rows: row gr < *count is token uniq[gr] (NULL: no
    const unsigned *count = nullptr; // deduplication; R_total then only sizes the grid)
};
cudaError_t prepare_projection(int smem_optin);
// Output columns per CTA (64, 128 or 256) for R_total gathered rows: the
// narrowest whose grid still fits one CTA per SM.
int projection_cols(int R_total, int num_sms);
// CTAs per output tile along d for R_total rows and NC output columns (1 or 2),
// and the most rows for which it can be 2 (the partial-sum workspace's size).
int projection_ksplit(int R_total, int NC, int d, int num_sms);
int projection_split_rows(int num_sms);
// p.tm_wa / p.tm_wb must have boxes of 64 columns x NC rows.
cudaError_t launch_projection(const ProjParams &p, int NC, cudaStream_t s);

// ---- pair tables and the walk ----
struct PairParams {
    const float *AB;      // [B * R][512], or NULL with tab
    const float *tab;     // [V][512] precomputed A|B of every token (NULL: use AB)
    const int32_t *anchor;  // [B] (read with tab)
    int *err;
    int64_t V;
    const float *gate;    // [B * L][256]
    const float *vals;    // [B, L, K]
    const int32_t *ids;   // [B, L, K]
    float *P;             // [B, L, K, K] workspace tables
    float *P_out;         // optional copy for the caller
    unsigned *ticket;     // [B] zero between runs
    int32_t *path;        // [B, L]
    float *path_score;    // optional [B]
    uint8_t *tie_flags;   // optional [B, L]
    int B, L, K, R, walk;
    float tie_eps;
    const float *u_walk;  // [B, L] uniforms (sampling walk)
    float *q_out;         // [B, L, K] draft distributions (sampling walk)
    float temperature;
    const uint64_t *dd_tab = nullptr;  // deduplicated AB rows: the row of token v is
    const int32_t *dd_rep = nullptr;   // dd_rep[~low32(dd_tab[v])] (NULL: AB by gathered row)
    const int32_t *target = nullptr;   // [B, L+1] target tokens: the walker also checks the path (NULL: not)
    int32_t *accept = nullptr;         // [B]
    int32_t *emitted = nullptr;        // [B, L+1] (may be NULL)
    uint32_t *done = nullptr;          // [B] host-mapped completion flags (NULL: none), set to `step`
    int *err_snap = nullptr;           // [B] host-mapped copies of the error word
    uint32_t step = 0;
};
// min_smem: dynamic shared memory to reserve at least (see ctas_per_sm_smem).
cudaError_t launch_pair_walk(const PairParams &p, cudaStream_t s, size_t min_smem = 0);

// ---- fused tail for small batches: merge + projections + pair tables + walk ----
struct TailParams {
    CUtensorMap tm_wa, tm_wb;  // W_A, W_B [256, d] bf16, box 64 x 256, 128B swizzle
    const float *tab;          // [V][512] precomputed A|B of every token (NULL: project in the kernel)
    const uint64_t *part;      // [G][N][K] partial top-K keys
    uint64_t *thr_g;           // [N] lm_head thresholds, reset here for the next pass
    const float *gate;         // [N][256]
    const uint16_t *E;         // [V, d] bf16 bits
    const int32_t *anchor;     // [B]
    int32_t *ids;              // [N][K] merged candidates (workspace)
    float *vals;               // [N][K]
    int32_t *ids_out;          // optional copies for the caller
    float *vals_out;
    float *P;                  // [N][K][K] tables (workspace)
    float *P_out;              // optional
    unsigned *ticket;          // [B]
    int32_t *path;             // [B, L]
    float *path_score;         // optional [B]
    uint8_t *tie_flags;        // optional [B, L]
    int *err;
    int64_t V;
    int d, L, G, N, cs, walk;
    float tie_eps;
    const float *u_walk;  // [B, L] uniforms (sampling walk)
    float *q_out;         // [B, L, K] draft distributions (sampling walk)
    float temperature;
    const int32_t *target = nullptr;  // [B, L+1] target tokens: the walker also checks the path (NULL: not)
    int32_t *accept = nullptr;        // [B]
    int32_t *emitted = nullptr;       // [B, L+1] (may be NULL)
    uint32_t *done = nullptr;         // [B] host-mapped completion flags (NULL: none), set to `step`
    int *err_snap = nullptr;          // [B] host-mapped copies of the error word
    uint32_t step = 0;
};
int tail_cluster_size(int d);
int tail_stages(int K, int G, int cs, int smem_optin);
size_t tail_smem_bytes(int K, int S, int G, int cs);
cudaError_t prepare_tail(int smem_optin);
cudaError_t launch_select_tail(const TailParams &p, int K, int S, size_t smem, cudaStream_t s);

// ---- greedy accept check ----
cudaError_t launch_verify(const int32_t *path, const int32_t *target, int B, int L, int32_t *accept,
                          int32_t *emitted, cudaStream_t s);
cudaError_t launch_verify_rejection(const int32_t *path, const int32_t *ids, const float *q, const float *p,
                                    const float *u_acc, const float *u_res, int B, int L, int K, int64_t V,
                                    int32_t *accept, int32_t *emitted, cudaStream_t s);

}  // namespace dfl
