// Host side of the C ABI declared in include/dflash_select.h: argument
// validation, the device workspace, TMA descriptors, the launch sequence of
// one selector run, and per-kernel event timing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "dflash_select.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

dflash_status fail(dflash_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

dflash_status ok()
{
    return DFLASH_OK;
}

#define CUDA_TRY(call)                                                                                    \
    do {                                                                                                  \
        cudaError_t e_ = (call);                                                                          \
        if (e_ != cudaSuccess)                                                                            \
            return fail(DFLASH_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                        __LINE__);                                                                        \
    } while (0)

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// bf16 [rows, cols] row-major, tiles of 64 columns x box_rows rows, 128B swizzle,
// rows past the end read as zero.
dflash_status make_tmap(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(dfl::kLmTileK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%lld, %lld] tensor", static_cast<int>(r),
                    static_cast<long long>(rows), static_cast<long long>(cols));
    return ok();
}

}  // namespace

namespace dfl {

// Used by the other host translation units of the library.
dflash_status host_fail(dflash_status st, const char *msg)
{
    return fail(st, "%s", msg);
}

dflash_status host_make_tmap(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, int box_rows)
{
    return make_tmap(tm, ptr, rows, cols, box_rows);
}

}  // namespace dfl

namespace {

constexpr int kProfileRuns = 4096;
constexpr int kProfileKernels = 6;  // lm_head+top-K, merge, projection, pair+walk, fused tail, dedup
constexpr int kProfileSlots = 5;    // launches recorded per run

// A pilot lm_head pass over kPilotTiles sampled vocabulary tiles (per
// position tile) seeds the thresholds of position tiles at least
// DFL_LM_PILOT_MIN_NT wide.
constexpr int kPilotTiles = 64;
constexpr int kPilotMaxTiles = 160;  // maxima the main pass reads per position (5 per lane)
#ifndef DFL_LM_PILOT_MIN_NT
#define DFL_LM_PILOT_MIN_NT 96
#endif
#ifndef DFL_LM_PILOT_MAX_NTILES
#define DFL_LM_PILOT_MAX_NTILES 16
#endif

// Position counts in (128, 256] run the CTA-pair lm_head kernel (one
// 256-row weight tile per pair, half of the positions in each CTA's shared
// memory): a single-CTA tile of that width holds less weight in flight per
// SM than the HBM stream needs.
#ifndef DFL_LM_PAIR
#define DFL_LM_PAIR 1
#endif
// Two 64-column boxes per stage (three stages of 60 KB rather than six of
// 30 KB): measured 4b_b32 lm_head 191 -> 178 us.
#ifndef DFL_LM_PAIR_BOXES
#define DFL_LM_PAIR_BOXES 2
#endif

struct Plan {
    int N, NT, n_tiles_n, G, grid, stages, boxes, R_total;
    bool pair;                    // the CTA-pair kernel (one position tile, G = 2 x pairs)
    int mt_vocab, mt_total;       // weight tiles of the pass (a pair: vocabulary tiles rounded up to even)
    int pilot_G, pilot_stride;  // pilot CTAs per position tile and their tile stride (0: no pilot)
    int pilot_NT, pilot_ntiles, pilot_stages, pilot_boxes;  // the pilot's own position tiling
    size_t pilot_smem;
    size_t smem;
    bool fused_tail;  // one clustered kernel for merge + projections + tables + walk
    int tail_cs, tail_S;
    size_t tail_smem;
};

struct ProfRun {
    int kid[kProfileSlots];
    int n;
};

}  // namespace

struct dflash_select_ctx {
    dflash_select_config cfg;
    const void *W, *E, *WA, *WB, *WH;
    int device = 0, num_sms = 0;
    size_t smem_optin = 0;  // opt-in shared memory per block
    size_t smem_per_sm = 0;
    CUtensorMap tm_w, tm_gate, tm_h, tm_wa, tm_wb;
    CUtensorMap tm_pa[3], tm_pb[3];  // W_A, W_B with 64 x {64, 128, 256}-row boxes (projection tiles)
    const void *h_ptr = nullptr, *hp_ptr = nullptr;
    int h_rows = -1, h_box = -1, hp_rows = -1, hp_box = -1;
    CUtensorMap tm_hp;  // hidden with whole-tile boxes, for the pilot of a pair pass
    int m_tiles_vocab = 0, m_tiles_total = 0, R = 0;
    int pair_clusters = 0;  // CTA pairs of the pair lm_head kernel that fit at once (0: not used)
    int64_t shard_v0 = 0, shard_rows = 0;  // the rows of W_lm this handle streams: tokens [v0, v0 + rows)

    void *ws = nullptr;
    uint64_t *part = nullptr;
    uint64_t *thr_g = nullptr;  // per-position lm_head thresholds shared by the CTAs
    uint64_t *tmax = nullptr;   // [num_sms][max_batch * L] best logit of each lm_head CTA, epoch-tagged
    uint64_t *pmax = nullptr;   // [kPilotMaxTiles][max_batch * L] the pilot's tile maxima, epoch-tagged
    uint32_t epoch = 0;
    float *gate = nullptr, *vals = nullptr, *AB = nullptr, *P = nullptr;
    float *tab = nullptr;  // [V][512] precomputed A|B of every token (cfg.tables)
    int32_t *ids = nullptr;
    unsigned *ticket = nullptr;
    float *proj_part = nullptr;     // [2][rows][512] partial sums of the split projection
    unsigned *proj_ticket = nullptr;
    uint64_t *dd_tab = nullptr;  // [V] deduplication marks (cfg.dedup)
    unsigned *dd_count = nullptr;
    int32_t *dd_uniq = nullptr, *dd_rep = nullptr;  // [max_batch * R]
    uint32_t dd_epoch = 0;
    int *err = nullptr;
    // staging of dflash_select_step_host: hidden on the device (the one
    // upload); anchor and target in a mapped pinned image that the kernels
    // read directly; the results in a mapped pinned block that the walking
    // kernel writes directly: path [Nmax], accept [Bm], emitted [Bm, L+1], then
    // per sequence a copy of the error word and a completion flag
    uint16_t *st_hidden = nullptr;
    uint8_t *st_in_host = nullptr;  // [anchor [Bm] | target [Bm, L+1] at st_tgt_off], mapped
    uint8_t *st_in_dev = nullptr;   // its device view
    size_t st_tgt_off = 0;
    int32_t *ho_path = nullptr, *ho_accept = nullptr, *ho_emitted = nullptr, *ho_err = nullptr;  // mapped, host view
    uint32_t *ho_done = nullptr;
    int32_t *hd_path = nullptr, *hd_accept = nullptr, *hd_emitted = nullptr, *hd_err = nullptr;  // device view
    uint32_t *hd_done = nullptr;
    uint32_t host_step = 0;  // the step number the flags of the latest host step carry
    // set by dflash_select_step_host for the duration of its run
    uint32_t *hs_done = nullptr;
    int *hs_err_snap = nullptr;
    uint32_t hs_step = 0;
    int *err_host = nullptr;  // pinned

    bool prof = false;
    int prof_runs = 0;
    std::vector<cudaEvent_t> ev;  // kProfileRuns x kProfileSlots x {begin, end}
    std::vector<ProfRun> prof_rec;

    Plan plan(int B) const
    {
        Plan p;
        p.N = B * cfg.L;
        // position tiles of at most 128 up to 256 positions (the per-CTA top-K
        // upkeep grows with the tile's width), 256 beyond
#ifndef DFL_LM_TILE_POS
#define DFL_LM_TILE_POS 128
#endif
        p.pair = DFL_LM_PAIR && p.N > 128 && pair_clusters > 0;
        if (p.pair) {  // position tiles of up to 256, half of each in either CTA of a pair
            p.n_tiles_n = (p.N + 255) / 256;
            p.NT = ((p.N + p.n_tiles_n - 1) / p.n_tiles_n + 15) / 16 * 16;
            if (pair_clusters < p.n_tiles_n) p.pair = false;
        }
        if (p.pair) {
        } else if (p.N <= 256) {
            p.n_tiles_n = (p.N + DFL_LM_TILE_POS - 1) / DFL_LM_TILE_POS;
            p.NT = (((p.N + p.n_tiles_n - 1) / p.n_tiles_n) + 15) / 16 * 16;
        } else {
            p.NT = 256;
            p.n_tiles_n = (p.N + 255) / 256;
        }
        p.mt_vocab = p.pair ? (m_tiles_vocab + 1) / 2 * 2 : m_tiles_vocab;
        p.mt_total = p.mt_vocab + dfl::kEmbed / dfl::kLmTileM;
        // stages that fit for `boxes` boxes of weights and `hrows` hidden rows each
        auto stages_for = [&](int NT, int boxes, int hrows) {
            const size_t fixed = dfl::lmhead_smem_bytes(NT, cfg.K, 0, boxes, hrows);
            const size_t stage = static_cast<size_t>(boxes) * (static_cast<size_t>(dfl::kLmTileM) * dfl::kLmTileK * 2 +
                                                               static_cast<size_t>(hrows) * dfl::kLmTileK * 2);
            int st = static_cast<int>((smem_optin - fixed) / stage);
            if (st > dfl::kLmMaxStages) st = dfl::kLmMaxStages;
            while (st > 1 && dfl::lmhead_smem_bytes(NT, cfg.K, st, boxes, hrows) > smem_optin) --st;  // barriers
            return st;
        };
        int hrows = p.NT;
        if (p.pair) {
            int g2 = (num_sms / 2) / p.n_tiles_n;  // pairs per position tile
            if (g2 > pair_clusters / p.n_tiles_n) g2 = pair_clusters / p.n_tiles_n;
            if (g2 > p.mt_total / 2) g2 = p.mt_total / 2;
            p.G = 2 * g2;
            p.grid = 2 * g2 * p.n_tiles_n;
            hrows = p.NT / 2;
            // two boxes per stage where three such stages fit, else one
            p.boxes = DFL_LM_PAIR_BOXES;
            while (p.boxes > 1 && (cfg.d % (dfl::kLmTileK * p.boxes) != 0 || stages_for(p.NT, p.boxes, hrows) < 3))
                --p.boxes;
        } else {
            int g = num_sms / p.n_tiles_n;
            if (g < 1) g = 1;
            if (g > m_tiles_total) g = m_tiles_total;
            p.G = g;
            p.grid = g * p.n_tiles_n;
            p.boxes = dfl::lmhead_boxes(cfg.d, p.NT);
        }
        p.stages = stages_for(p.NT, p.boxes, hrows);
        p.smem = dfl::lmhead_smem_bytes(p.NT, cfg.K, p.stages, p.boxes, hrows);
        p.pilot_G = 0;
        p.pilot_stride = 0;
        p.pilot_NT = p.NT;
        p.pilot_ntiles = p.n_tiles_n;
        p.pilot_boxes = p.boxes;
        p.pilot_stages = p.stages;
        p.pilot_smem = p.smem;
        if (p.NT >= DFL_LM_PILOT_MIN_NT && p.n_tiles_n <= DFL_LM_PILOT_MAX_NTILES &&
            m_tiles_vocab >= 4 * kPilotTiles) {
            if (p.pair) {  // the pilot runs the single-CTA kernel (up to 256 positions: tiles of at most 128)
                if (p.N <= 256) {
                    p.pilot_ntiles = (p.N + 127) / 128;
                    p.pilot_NT = ((p.N + p.pilot_ntiles - 1) / p.pilot_ntiles + 15) / 16 * 16;
                }
                p.pilot_boxes = dfl::lmhead_boxes(cfg.d, p.pilot_NT);
                p.pilot_stages = stages_for(p.pilot_NT, p.pilot_boxes, p.pilot_NT);
                p.pilot_smem = dfl::lmhead_smem_bytes(p.pilot_NT, cfg.K, p.pilot_stages, p.pilot_boxes);
            }
            // one wave of CTAs with at least kPilotTiles sampled tiles per position tile; with many
            // position tiles 2K of them (the bound takes the K-th largest of 32 lanes' maxima)
            int g = num_sms / p.pilot_ntiles;
            if (g < kPilotTiles) g = p.pilot_ntiles > 2 ? 2 * cfg.K : kPilotTiles;
            if (g > kPilotMaxTiles) g = kPilotMaxTiles;
            if (g > m_tiles_vocab / 4) g = m_tiles_vocab / 4;
            p.pilot_G = g;
            p.pilot_stride = m_tiles_vocab / g;
        }
        p.R_total = B * R;
        p.tail_cs = dfl::tail_cluster_size(cfg.d);
        p.tail_S = dfl::tail_stages(cfg.K, p.G, p.tail_cs, static_cast<int>(smem_optin));
        p.fused_tail = p.n_tiles_n == 1 && p.N * p.tail_cs <= num_sms && p.tail_S > 0;
        p.tail_smem = p.fused_tail ? dfl::tail_smem_bytes(cfg.K, p.tail_S, p.G, p.tail_cs) : 0;
        return p;
    }
};

extern "C" {

const char *dflash_last_error(void)
{
    return g_last_error.c_str();
}

// [A(v) | B(v)] = [W_A; W_B] E[v] for every token v, by the projection kernel
// over the identity list of rows (R = 1: row v is "anchor" v).
static dflash_status build_tables(dflash_select_ctx *c, cudaStream_t s)
{
    const int64_t V = c->cfg.V;
    CUDA_TRY(cudaMalloc(&c->tab, static_cast<size_t>(V) * 512 * sizeof(float)));
    std::vector<int32_t> ident(static_cast<size_t>(V));
    for (int64_t v = 0; v < V; ++v) ident[static_cast<size_t>(v)] = static_cast<int32_t>(v);
    int32_t *rows = nullptr;
    CUDA_TRY(cudaMalloc(&rows, static_cast<size_t>(V) * sizeof(int32_t)));
    cudaError_t e = cudaMemcpyAsync(rows, ident.data(), static_cast<size_t>(V) * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, s);
    dfl::ProjParams pp;
    const int nc = dfl::projection_cols(static_cast<int>(V), c->num_sms);
    const int ti = nc == 64 ? 0 : (nc == 128 ? 1 : 2);
    pp.tm_wa = c->tm_pa[ti];
    pp.tm_wb = c->tm_pb[ti];
    pp.E = static_cast<const uint16_t *>(c->E);
    pp.ids = rows;  // not read with R = 1
    pp.anchor = rows;
    pp.AB = c->tab;
    pp.err = c->err;
    pp.V = V;
    pp.d = c->cfg.d;
    pp.L = 0;
    pp.K = c->cfg.K;
    pp.R = 1;
    pp.R_total = static_cast<int>(V);
    pp.ksplit = 1;
    pp.part = nullptr;
    pp.ticket = nullptr;
    if (e == cudaSuccess) e = dfl::launch_projection(pp, nc, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(rows);
    if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "building the A|B tables failed: %s", cudaGetErrorString(e));
    return ok();
}

static dflash_status check_config(const dflash_select_config *c)
{
    if (!c) return fail(DFLASH_ERR_INVALID_ARG, "config is NULL");
    if (c->K != 16 && c->K != 32) return fail(DFLASH_ERR_UNSUPPORTED, "K must be 16 or 32 (got %d)", c->K);
    if (c->L < 1 || c->L > 16) return fail(DFLASH_ERR_UNSUPPORTED, "L must be in [1, 16] (got %d)", c->L);
    if (c->V < c->K || c->V >= (int64_t(1) << 31))
        return fail(DFLASH_ERR_UNSUPPORTED, "V must satisfy K <= V < 2^31 (got %lld)", static_cast<long long>(c->V));
    if (c->d < 64 || c->d > 16384 || c->d % 64 != 0)
        return fail(DFLASH_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 16384] (got %d)", c->d);
    if (c->e != dfl::kEmbed) return fail(DFLASH_ERR_UNSUPPORTED, "e must be 256 (got %d)", c->e);
    if (c->max_batch < 1 || static_cast<int64_t>(c->max_batch) * c->L > 8192)
        return fail(DFLASH_ERR_UNSUPPORTED, "max_batch must be >= 1 with max_batch * L <= 8192");
    if (c->walk != DFLASH_WALK_VITERBI && c->walk != DFLASH_WALK_GREEDY && c->walk != DFLASH_WALK_SAMPLE)
        return fail(DFLASH_ERR_INVALID_ARG, "walk must be DFLASH_WALK_VITERBI, _GREEDY or _SAMPLE");
    if (c->walk == DFLASH_WALK_SAMPLE && (!(c->temperature > 0.0f) || !std::isfinite(c->temperature)))
        return fail(DFLASH_ERR_INVALID_ARG, "the sampling walk needs a finite temperature > 0");
    if (!(c->tie_eps >= 0.0f) || !std::isfinite(c->tie_eps))
        return fail(DFLASH_ERR_INVALID_ARG, "tie_eps must be finite and >= 0");
    if (c->tables != 0 && c->tables != 1) return fail(DFLASH_ERR_INVALID_ARG, "tables must be 0 or 1");
    if (c->dedup != 0 && c->dedup != 1) return fail(DFLASH_ERR_INVALID_ARG, "dedup must be 0 or 1");
    if (c->dedup && c->tables)
        return fail(DFLASH_ERR_INVALID_ARG, "dedup applies to the per-run projections, not to tables = 1");
    return ok();
}

static dflash_status init_impl(const dflash_select_config *cfg, const void *W_lm, int64_t v0, int64_t rows,
                               const void *E, const void *W_A, const void *W_B, const void *W_H, void *stream,
                               dflash_select_handle *out)
{
    dflash_status st;
    const void *ptrs[5] = {W_lm, E, W_A, W_B, W_H};
    const char *names[5] = {"W_lm", "E", "W_A", "W_B", "W_H"};
    for (int i = 0; i < 5; ++i) {
        if (!ptrs[i]) return fail(DFLASH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(ptrs[i])) return fail(DFLASH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3)
        return fail(DFLASH_ERR_UNSUPPORTED, "this library is built for sm_103 (GB300); device is sm_%d%d", prop.major,
                    prop.minor);

    CUDA_TRY(dfl::prepare_lmhead(static_cast<int>(prop.sharedMemPerBlockOptin)));
    CUDA_TRY(dfl::prepare_topk_merge(static_cast<int>(prop.sharedMemPerBlockOptin)));
    CUDA_TRY(dfl::prepare_pair_walk(static_cast<int>(prop.sharedMemPerBlockOptin)));
    CUDA_TRY(dfl::prepare_projection(static_cast<int>(prop.sharedMemPerBlockOptin)));
    CUDA_TRY(dfl::prepare_tail(static_cast<int>(prop.sharedMemPerBlockOptin)));

    dflash_select_ctx *c = new (std::nothrow) dflash_select_ctx();
    if (!c) return fail(DFLASH_ERR_CUDA, "out of host memory");
    c->cfg = *cfg;
    c->W = W_lm;
    c->E = E;
    c->WA = W_A;
    c->WB = W_B;
    c->WH = W_H;
    c->device = dev;
    c->num_sms = prop.multiProcessorCount;
    c->smem_optin = prop.sharedMemPerBlockOptin;
    c->smem_per_sm = prop.sharedMemPerMultiprocessor;
    c->shard_v0 = v0;
    c->shard_rows = rows;
    c->m_tiles_vocab = static_cast<int>((rows + dfl::kLmTileM - 1) / dfl::kLmTileM);
    c->m_tiles_total = c->m_tiles_vocab + dfl::kEmbed / dfl::kLmTileM;
    c->R = cfg->L * cfg->K + 1;
    {
        // CTA pairs resident at once, for the widest pair configuration (256
        // positions; every configuration holds one CTA per SM)
        const size_t fixed = dfl::lmhead_smem_bytes(256, cfg->K, 0, 1, 128);
        const size_t stage = static_cast<size_t>(dfl::kLmTileM) * dfl::kLmTileK * 2 + 128u * dfl::kLmTileK * 2;
        const size_t smem_pair = fixed + ((prop.sharedMemPerBlockOptin - fixed) / stage) * stage;
        c->pair_clusters = dfl::lmhead_pair_max_clusters(smem_pair);
    }

    if ((st = make_tmap(&c->tm_w, W_lm, rows, cfg->d, dfl::kLmTileM)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_gate, W_H, dfl::kEmbed, cfg->d, dfl::kLmTileM)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_wa, W_A, dfl::kEmbed, cfg->d, dfl::kEmbed)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_wb, W_B, dfl::kEmbed, cfg->d, dfl::kEmbed)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pa[0], W_A, dfl::kEmbed, cfg->d, 64)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pa[1], W_A, dfl::kEmbed, cfg->d, 128)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pa[2], W_A, dfl::kEmbed, cfg->d, 256)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pb[0], W_B, dfl::kEmbed, cfg->d, 64)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pb[1], W_B, dfl::kEmbed, cfg->d, 128)) != DFLASH_OK ||
        (st = make_tmap(&c->tm_pb[2], W_B, dfl::kEmbed, cfg->d, 256)) != DFLASH_OK) {
        delete c;
        return st;
    }

    // workspace: the largest partial-list buffer over every batch size
    size_t part_elems = 0;
    for (int B = 1; B <= cfg->max_batch; ++B) {
        Plan p = c->plan(B);
        size_t e = static_cast<size_t>(p.G) * p.N * cfg->K;
        if (e > part_elems) part_elems = e;
    }
    const size_t Nmax = static_cast<size_t>(cfg->max_batch) * cfg->L;
    const size_t Bm = static_cast<size_t>(cfg->max_batch);
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    size_t off = 0;
    const size_t o_part = off; off += up(part_elems * 8);
    const size_t o_thrg = off; off += up(Nmax * 8);
    const size_t o_tmax = off; off += up(static_cast<size_t>(prop.multiProcessorCount) * Nmax * 8);
    const size_t o_pmax = off; off += up(static_cast<size_t>(kPilotMaxTiles) * Nmax * 8);
    const size_t o_gate = off; off += up(Nmax * dfl::kEmbed * 4);
    const size_t o_ids = off; off += up(Nmax * cfg->K * 4);
    const size_t o_vals = off; off += up(Nmax * cfg->K * 4);
    const size_t o_AB = off; off += up(Bm * c->R * 512 * 4);
    const size_t o_P = off; off += up(Nmax * cfg->K * cfg->K * 4);
    const size_t o_ticket = off; off += up(Bm * 4);
    // the projection's split along d applies up to projection_split_rows rows
    const size_t split_rows =
        std::min(static_cast<size_t>(dfl::projection_split_rows(prop.multiProcessorCount)), Bm * c->R);
    const size_t o_ppart = off; off += up(2 * split_rows * 512 * 4);
    const size_t o_ptick = off; off += up(static_cast<size_t>(8 * (prop.multiProcessorCount / 16 + 1)) * 4);
    const size_t dd_rows = cfg->dedup ? Bm * c->R : 0;
    const size_t o_ddtab = off; off += up(cfg->dedup ? static_cast<size_t>(cfg->V) * 8 : 0);
    const size_t o_ddcnt = off; off += up(cfg->dedup ? 4 : 0);
    const size_t o_dduniq = off; off += up(dd_rows * 4);
    const size_t o_ddrep = off; off += up(dd_rows * 4);
    const size_t o_hid = off; off += up(Nmax * cfg->d * 2);
    const size_t o_err = off; off += up(4);
    const size_t tgt_off = up(Bm * 4), in_bytes = tgt_off + up(Bm * (cfg->L + 1) * 4);
    cudaError_t e = cudaMalloc(&c->ws, off);
    if (e != cudaSuccess) {
        delete c;
        return fail(DFLASH_ERR_CUDA, "cudaMalloc of a %zu-byte workspace failed: %s", off, cudaGetErrorString(e));
    }
    // one mapped pinned allocation: the error word, the image of [anchor |
    // target], and the results block of the host step
    const size_t h_path = up(sizeof(int)) + up(in_bytes);
    const size_t h_acc = h_path + up(Nmax * 4);
    const size_t h_emit = h_acc + up(Bm * 4);
    const size_t h_err = h_emit + up(Bm * (cfg->L + 1) * 4);
    const size_t h_done = h_err + up(Bm * 4);
    const size_t host_bytes = h_done + up(Bm * 4);
    e = cudaHostAlloc(&c->err_host, host_bytes, cudaHostAllocMapped);
    uint8_t *hdev = nullptr;
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&hdev), c->err_host, 0);
    if (e != cudaSuccess) {
        if (c->err_host) cudaFreeHost(c->err_host);
        cudaFree(c->ws);
        delete c;
        return fail(DFLASH_ERR_CUDA, "mapped host allocation of %zu bytes failed: %s", host_bytes,
                    cudaGetErrorString(e));
    }
    std::memset(c->err_host, 0, host_bytes);
    uint8_t *const hhost = reinterpret_cast<uint8_t *>(c->err_host);
    c->st_in_host = hhost + up(sizeof(int));
    c->st_in_dev = hdev + up(sizeof(int));
    c->st_tgt_off = tgt_off;
    c->ho_path = reinterpret_cast<int32_t *>(hhost + h_path);
    c->ho_accept = reinterpret_cast<int32_t *>(hhost + h_acc);
    c->ho_emitted = reinterpret_cast<int32_t *>(hhost + h_emit);
    c->ho_err = reinterpret_cast<int32_t *>(hhost + h_err);
    c->ho_done = reinterpret_cast<uint32_t *>(hhost + h_done);
    c->hd_path = reinterpret_cast<int32_t *>(hdev + h_path);
    c->hd_accept = reinterpret_cast<int32_t *>(hdev + h_acc);
    c->hd_emitted = reinterpret_cast<int32_t *>(hdev + h_emit);
    c->hd_err = reinterpret_cast<int32_t *>(hdev + h_err);
    c->hd_done = reinterpret_cast<uint32_t *>(hdev + h_done);
    uint8_t *w = static_cast<uint8_t *>(c->ws);
    c->part = reinterpret_cast<uint64_t *>(w + o_part);
    c->thr_g = reinterpret_cast<uint64_t *>(w + o_thrg);
    c->tmax = reinterpret_cast<uint64_t *>(w + o_tmax);
    c->pmax = reinterpret_cast<uint64_t *>(w + o_pmax);
    c->gate = reinterpret_cast<float *>(w + o_gate);
    c->ids = reinterpret_cast<int32_t *>(w + o_ids);
    c->vals = reinterpret_cast<float *>(w + o_vals);
    c->AB = reinterpret_cast<float *>(w + o_AB);
    c->P = reinterpret_cast<float *>(w + o_P);
    c->ticket = reinterpret_cast<unsigned *>(w + o_ticket);
    c->proj_part = reinterpret_cast<float *>(w + o_ppart);
    c->proj_ticket = reinterpret_cast<unsigned *>(w + o_ptick);
    if (cfg->dedup) {
        c->dd_tab = reinterpret_cast<uint64_t *>(w + o_ddtab);
        c->dd_count = reinterpret_cast<unsigned *>(w + o_ddcnt);
        c->dd_uniq = reinterpret_cast<int32_t *>(w + o_dduniq);
        c->dd_rep = reinterpret_cast<int32_t *>(w + o_ddrep);
    }
    c->err = reinterpret_cast<int *>(w + o_err);
    c->st_hidden = reinterpret_cast<uint16_t *>(w + o_hid);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(c->ws, 0, off, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaFreeHost(c->err_host);
        cudaFree(c->ws);
        delete c;
        return fail(DFLASH_ERR_CUDA, "workspace initialisation failed: %s", cudaGetErrorString(e));
    }
    if (cfg->tables) {
        st = build_tables(c, s);
        if (st != DFLASH_OK) {
            cudaFree(c->tab);
            cudaFreeHost(c->err_host);
            cudaFree(c->ws);
            delete c;
            return st;
        }
    }
    *out = c;
    return ok();
}

dflash_status dflash_select_init(const dflash_select_config *cfg, const void *W_lm, const void *E, const void *W_A,
                                 const void *W_B, const void *W_H, void *stream, dflash_select_handle *out)
{
    if (!out) return fail(DFLASH_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    dflash_status st = check_config(cfg);
    if (st != DFLASH_OK) return st;
    return init_impl(cfg, W_lm, 0, cfg->V, E, W_A, W_B, W_H, stream, out);
}

dflash_status dflash_select_init_shard(const dflash_select_config *cfg, const void *W_shard, int64_t v0, int64_t v1,
                                       const void *E, const void *W_A, const void *W_B, const void *W_H, void *stream,
                                       dflash_select_handle *out)
{
    if (!out) return fail(DFLASH_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    dflash_status st = check_config(cfg);
    if (st != DFLASH_OK) return st;
    if (v0 < 0 || v1 <= v0 || v1 > cfg->V)
        return fail(DFLASH_ERR_INVALID_ARG, "the shard [%lld, %lld) must be a non-empty range within [0, V = %lld)",
                    static_cast<long long>(v0), static_cast<long long>(v1), static_cast<long long>(cfg->V));
    return init_impl(cfg, W_shard, v0, v1 - v0, E, W_A, W_B, W_H, stream, out);
}

static void prof_ensure(dflash_select_ctx *c)
{
    if (!c->ev.empty()) return;
    c->ev.resize(static_cast<size_t>(kProfileRuns) * kProfileSlots * 2);
    for (auto &x : c->ev) cudaEventCreate(&x);
    c->prof_rec.resize(kProfileRuns);
}

static bool prof_on(dflash_select_ctx *c)
{
    return c->prof && c->prof_runs < kProfileRuns;
}

static void prof_begin(dflash_select_ctx *c, int slot, cudaStream_t s)
{
    if (prof_on(c)) cudaEventRecord(c->ev[(static_cast<size_t>(c->prof_runs) * kProfileSlots + slot) * 2], s);
}

static void prof_end(dflash_select_ctx *c, int slot, int kid, cudaStream_t s)
{
    if (!prof_on(c)) return;
    cudaEventRecord(c->ev[(static_cast<size_t>(c->prof_runs) * kProfileSlots + slot) * 2 + 1], s);
    c->prof_rec[c->prof_runs].kid[slot] = kid;
    c->prof_rec[c->prof_runs].n = slot + 1;
}

// The lm_head + top-K pass (and the gate) of B sequences: partial lists in
// c->part, g_t in c->gate.
static dflash_status launch_lmhead(dflash_select_ctx *c, const void *hidden, const Plan &pl, cudaStream_t s)
{
    const int box = pl.pair ? pl.NT / 2 : pl.NT;
    if (hidden != c->h_ptr || pl.N != c->h_rows || box != c->h_box) {
        dflash_status st = make_tmap(&c->tm_h, hidden, pl.N, c->cfg.d, box);
        if (st != DFLASH_OK) return st;
        c->h_ptr = hidden;
        c->h_rows = pl.N;
        c->h_box = box;
    }
    if (pl.pair && pl.pilot_G > 0 && (hidden != c->hp_ptr || pl.N != c->hp_rows || pl.pilot_NT != c->hp_box)) {
        dflash_status st = make_tmap(&c->tm_hp, hidden, pl.N, c->cfg.d, pl.pilot_NT);
        if (st != DFLASH_OK) return st;
        c->hp_ptr = hidden;
        c->hp_rows = pl.N;
        c->hp_box = pl.pilot_NT;
    }
    dfl::LmHeadParams lp;
    lp.tm_w = c->tm_w;
    lp.tm_gate = c->tm_gate;
    lp.tm_h = c->tm_h;
    lp.V = c->shard_rows;
    lp.id_base = static_cast<uint32_t>(c->shard_v0);
    lp.d = c->cfg.d;
    lp.N = pl.N;
    lp.NT = pl.NT;
    lp.n_tiles_n = pl.n_tiles_n;
    lp.K = c->cfg.K;
    lp.m_tiles_vocab = pl.mt_vocab;
    lp.m_tiles_total = pl.mt_total;
    lp.ctas_per_ntile = pl.G;
    lp.stages = pl.stages;
    lp.boxes = pl.boxes;
    lp.part = c->part;
    lp.gate = c->gate;
    lp.thr_g = c->thr_g;
    lp.tmax = c->tmax;
    lp.epoch = ++c->epoch;
    if (lp.epoch == 0) {
        // The counter wrapped: clear the tagged maxima (tag 0, never current),
        // so that no entry left from 2^32 runs ago can carry the new epoch.
        const size_t row = static_cast<size_t>(c->cfg.max_batch) * c->cfg.L * 8;
        CUDA_TRY(cudaMemsetAsync(c->tmax, 0, static_cast<size_t>(c->num_sms) * row, s));
        CUDA_TRY(cudaMemsetAsync(c->pmax, 0, static_cast<size_t>(kPilotMaxTiles) * row, s));
        lp.epoch = ++c->epoch;
    }
    lp.err = c->err;

    prof_begin(c, 0, s);
    if (pl.pilot_G > 0) {
        dfl::LmHeadParams pp = lp;
        pp.pilot_stride = pl.pilot_stride;
        pp.ctas_per_ntile = pl.pilot_G;
        pp.m_tiles_vocab = c->m_tiles_vocab;
        pp.m_tiles_total = c->m_tiles_total;
        pp.stages = pl.pilot_stages;
        pp.boxes = pl.pilot_boxes;
        pp.NT = pl.pilot_NT;
        pp.n_tiles_n = pl.pilot_ntiles;
        if (pl.pair) pp.tm_h = c->tm_hp;
        pp.tmax = nullptr;
        pp.pmax = c->pmax;
        CUDA_TRY(dfl::launch_lmhead_topk(pp, pl.pilot_G * pl.pilot_ntiles, pl.pilot_smem, s));
        lp.tmax = nullptr;  // the pilot's maxima replace the CTAs' own
        lp.pmax = c->pmax;
        lp.pmax_n = pl.pilot_G;
    }
    if (pl.pair)
        CUDA_TRY(dfl::launch_lmhead_topk_pair(lp, pl.grid, pl.smem, s));
    else
        CUDA_TRY(dfl::launch_lmhead_topk(lp, pl.grid, pl.smem, s));
    prof_end(c, 0, 0, s);
    return ok();
}

// Everything after the lm_head pass: merge of G sorted lists part [G][N][K]
// (the lm_head CTAs' partial lists, or the vocabulary shards' lists),
// projections, pair tables and the walk; the gate comes from c->gate.
static dflash_status launch_tail(dflash_select_ctx *c, const int32_t *anchor, int32_t B, const Plan &pl,
                                 const uint64_t *part, int G, const float *u_walk, int32_t *topk_ids,
                                 float *topk_vals, float *pair_scores, int32_t *path, float *draft_probs,
                                 float *path_score, uint8_t *tie_flags, cudaStream_t s,
                                 const int32_t *target = nullptr, int32_t *accept = nullptr,
                                 int32_t *emitted = nullptr)
{
    int tail_S = pl.tail_S;
    size_t tail_smem = pl.tail_smem;
    bool fused = pl.fused_tail;
    if (G != pl.G) {
        tail_S = dfl::tail_stages(c->cfg.K, G, pl.tail_cs, static_cast<int>(c->smem_optin));
        fused = pl.n_tiles_n == 1 && pl.N * pl.tail_cs <= c->num_sms && tail_S > 0;
        tail_smem = fused ? dfl::tail_smem_bytes(c->cfg.K, tail_S, G, pl.tail_cs) : 0;
    }
    if (fused) {
        dfl::TailParams tp;
        tp.tm_wa = c->tm_wa;
        tp.tm_wb = c->tm_wb;
        tp.tab = c->tab;
        tp.part = part;
        tp.thr_g = c->thr_g;
        tp.gate = c->gate;
        tp.E = static_cast<const uint16_t *>(c->E);
        tp.anchor = anchor;
        tp.ids = c->ids;
        tp.vals = c->vals;
        tp.ids_out = topk_ids;
        tp.vals_out = topk_vals;
        tp.P = c->P;
        tp.P_out = pair_scores;
        tp.ticket = c->ticket;
        tp.path = path;
        tp.path_score = path_score;
        tp.tie_flags = tie_flags;
        tp.err = c->err;
        tp.V = c->cfg.V;
        tp.d = c->cfg.d;
        tp.L = c->cfg.L;
        tp.G = G;
        tp.N = pl.N;
        tp.cs = pl.tail_cs;
        tp.walk = c->cfg.walk;
        tp.tie_eps = c->cfg.tie_eps;
        tp.u_walk = u_walk;
        tp.q_out = draft_probs;
        tp.temperature = c->cfg.temperature;
        tp.target = target;
        tp.accept = accept;
        tp.emitted = emitted;
        tp.done = c->hs_done;
        tp.err_snap = c->hs_err_snap;
        tp.step = c->hs_step;
        prof_begin(c, 1, s);
        CUDA_TRY(dfl::launch_select_tail(tp, c->cfg.K, tail_S, tail_smem, s));
        prof_end(c, 1, 4, s);
        if (prof_on(c)) ++c->prof_runs;
        return ok();
    }

    dfl::DedupParams dd;
    if (c->dd_tab && !c->tab) {
        dd.tab = c->dd_tab;
        dd.count = c->dd_count;
        dd.uniq = c->dd_uniq;
        dd.rep = c->dd_rep;
        dd.anchor = anchor;
        dd.err = c->err;
        dd.V = c->cfg.V;
        dd.L = c->cfg.L;
        dd.K = c->cfg.K;
        dd.R = c->R;
        dd.epoch = ++c->dd_epoch;
        if (dd.epoch == 0) {
            // The counter wrapped: marks of older epochs would outrank the new
            // ones under atomicMax, so the table is cleared (mark 0) first.
            CUDA_TRY(cudaMemsetAsync(c->dd_tab, 0, static_cast<size_t>(c->cfg.V) * 8, s));
            dd.epoch = ++c->dd_epoch;
        }
    }
    int slot = 1;  // profiling slots are filled in launch order
    prof_begin(c, slot, s);
    // one position per CTA: one or two waves spread over the GPU, at most one
    // or two CTAs per SM
    const size_t spread = pl.N <= c->num_sms       ? dfl::ctas_per_sm_smem(c->smem_per_sm, 1)
                          : pl.N <= 2 * c->num_sms ? dfl::ctas_per_sm_smem(c->smem_per_sm, 2)
                                                   : 0;
    CUDA_TRY(dfl::launch_topk_merge(part, G, pl.N, c->cfg.K, c->ids, c->vals, topk_ids, topk_vals, c->thr_g, s,
                                    nullptr, dd, spread));
    prof_end(c, slot++, 1, s);
    if (dd.tab) {
        prof_begin(c, slot, s);
        CUDA_TRY(dfl::launch_dedup_compact(dd, c->ids, pl.R_total, s));
        prof_end(c, slot++, 5, s);
    }

    dfl::ProjParams pp;
    const int nc = dfl::projection_cols(pl.R_total, c->num_sms);
    const int ti = nc == 64 ? 0 : (nc == 128 ? 1 : 2);
    pp.tm_wa = c->tm_pa[ti];
    pp.tm_wb = c->tm_pb[ti];
    pp.E = static_cast<const uint16_t *>(c->E);
    pp.ids = c->ids;
    pp.anchor = anchor;
    pp.AB = c->AB;
    pp.err = c->err;
    pp.V = c->cfg.V;
    pp.d = c->cfg.d;
    pp.L = c->cfg.L;
    pp.K = c->cfg.K;
    pp.R = c->R;
    pp.R_total = pl.R_total;
    pp.ksplit = dfl::projection_ksplit(pl.R_total, nc, c->cfg.d, c->num_sms);
    pp.part = c->proj_part;
    pp.ticket = c->proj_ticket;
    if (dd.tab) {
        pp.uniq = c->dd_uniq;
        pp.count = c->dd_count;
    }
    if (!c->tab) {
        prof_begin(c, slot, s);
        CUDA_TRY(dfl::launch_projection(pp, nc, s));
        prof_end(c, slot++, 2, s);
    }

    dfl::PairParams q;
    q.AB = c->AB;
    q.tab = c->tab;
    q.anchor = anchor;
    q.err = c->err;
    q.V = c->cfg.V;
    q.gate = c->gate;
    q.vals = c->vals;
    q.ids = c->ids;
    q.P = c->P;
    q.P_out = pair_scores;
    q.ticket = c->ticket;
    q.path = path;
    q.path_score = path_score;
    q.tie_flags = tie_flags;
    q.B = B;
    q.L = c->cfg.L;
    q.K = c->cfg.K;
    q.R = c->R;
    q.walk = c->cfg.walk;
    q.tie_eps = c->cfg.tie_eps;
    q.u_walk = u_walk;
    q.q_out = draft_probs;
    q.temperature = c->cfg.temperature;
    if (dd.tab) {
        q.dd_tab = c->dd_tab;
        q.dd_rep = c->dd_rep;
    }
    q.target = target;
    q.accept = accept;
    q.emitted = emitted;
    q.done = c->hs_done;
    q.err_snap = c->hs_err_snap;
    q.step = c->hs_step;
    prof_begin(c, slot, s);
    CUDA_TRY(dfl::launch_pair_walk(q, s, spread));  // one CTA per (sequence, position), as the merge
    prof_end(c, slot, 3, s);
    if (prof_on(c)) ++c->prof_runs;
    return ok();
}

static dflash_status run_impl(dflash_select_handle h, const void *hidden, const int32_t *anchor, int32_t B,
                              const float *u_walk, int32_t *topk_ids, float *topk_vals, float *pair_scores,
                              int32_t *path, float *draft_probs, float *path_score, uint8_t *tie_flags,
                              void *stream, const int32_t *target = nullptr, int32_t *accept = nullptr,
                              int32_t *emitted = nullptr)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    dflash_select_ctx *c = h;
    if (B < 0 || B > c->cfg.max_batch)
        return fail(DFLASH_ERR_INVALID_ARG, "B must be in [0, max_batch=%d] (got %d)", c->cfg.max_batch, B);
    if (B == 0) return ok();
    if (!hidden || !anchor || !path) return fail(DFLASH_ERR_INVALID_ARG, "hidden, anchor and path must not be NULL");
    if (!aligned16(hidden)) return fail(DFLASH_ERR_INVALID_ARG, "hidden is not 16-byte aligned");
    if (c->shard_rows != c->cfg.V)
        return fail(DFLASH_ERR_INVALID_ARG, "a vocabulary-shard handle runs through dflash_select_topk_shard and "
                                            "dflash_select_run_gathered");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Plan pl = c->plan(B);
    dflash_status st = launch_lmhead(c, hidden, pl, s);
    if (st != DFLASH_OK) return st;
    return launch_tail(c, anchor, B, pl, c->part, pl.G, u_walk, topk_ids, topk_vals, pair_scores, path, draft_probs,
                       path_score, tie_flags, s, target, accept, emitted);
}

dflash_status dflash_select_topk_shard(dflash_select_handle h, const void *hidden, int32_t B, uint64_t *shard_keys,
                                       void *stream)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    dflash_select_ctx *c = h;
    if (B < 0 || B > c->cfg.max_batch)
        return fail(DFLASH_ERR_INVALID_ARG, "B must be in [0, max_batch=%d] (got %d)", c->cfg.max_batch, B);
    if (B == 0) return ok();
    if (!hidden || !shard_keys) return fail(DFLASH_ERR_INVALID_ARG, "hidden and shard_keys must not be NULL");
    if (!aligned16(hidden)) return fail(DFLASH_ERR_INVALID_ARG, "hidden is not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Plan pl = c->plan(B);
    const bool prof = c->prof;  // per-kernel timing covers whole runs only
    c->prof = false;
    dflash_status st = launch_lmhead(c, hidden, pl, s);
    c->prof = prof;
    if (st != DFLASH_OK) return st;
    CUDA_TRY(dfl::launch_topk_merge(c->part, pl.G, pl.N, c->cfg.K, c->ids, c->vals, nullptr, nullptr, c->thr_g, s,
                                    shard_keys));
    return ok();
}

dflash_status dflash_select_run_gathered(dflash_select_handle h, const int32_t *anchor, int32_t B,
                                         const uint64_t *all_keys, int32_t G, int32_t *topk_ids, float *topk_vals,
                                         float *pair_scores, int32_t *path, float *path_score, uint8_t *tie_flags,
                                         void *stream)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    dflash_select_ctx *c = h;
    if (c->cfg.walk == DFLASH_WALK_SAMPLE)
        return fail(DFLASH_ERR_INVALID_ARG, "dflash_select_run_gathered takes the max-sum or the greedy walk");
    if (B < 0 || B > c->cfg.max_batch)
        return fail(DFLASH_ERR_INVALID_ARG, "B must be in [0, max_batch=%d] (got %d)", c->cfg.max_batch, B);
    if (G < 1 || G > 1024) return fail(DFLASH_ERR_INVALID_ARG, "G must be in [1, 1024] (got %d)", G);
    if (B == 0) return ok();
    if (!anchor || !all_keys || !path) return fail(DFLASH_ERR_INVALID_ARG, "anchor, all_keys and path must not be NULL");
    const Plan pl = c->plan(B);
    const bool prof = c->prof;  // per-kernel timing covers whole runs only
    c->prof = false;
    const dflash_status st = launch_tail(c, anchor, B, pl, all_keys, G, nullptr, topk_ids, topk_vals, pair_scores,
                                         path, nullptr, path_score, tie_flags, static_cast<cudaStream_t>(stream));
    c->prof = prof;
    return st;
}

dflash_status dflash_select_run(dflash_select_handle h, const void *hidden, const int32_t *anchor, int32_t B,
                                int32_t *topk_ids, float *topk_vals, float *pair_scores, int32_t *path,
                                float *path_score, uint8_t *tie_flags, void *stream)
{
    if (h && h->cfg.walk == DFLASH_WALK_SAMPLE)
        return fail(DFLASH_ERR_INVALID_ARG, "a sampling handle runs through dflash_select_run_sampled");
    return run_impl(h, hidden, anchor, B, nullptr, topk_ids, topk_vals, pair_scores, path, nullptr, path_score,
                    tie_flags, stream);
}

dflash_status dflash_select_run_verify(dflash_select_handle h, const void *hidden, const int32_t *anchor, int32_t B,
                                       const int32_t *target, int32_t *path, int32_t *accept_len, int32_t *emitted,
                                       int32_t *topk_ids, float *topk_vals, float *pair_scores, float *path_score,
                                       uint8_t *tie_flags, void *stream)
{
    if (h && h->cfg.walk == DFLASH_WALK_SAMPLE)
        return fail(DFLASH_ERR_INVALID_ARG, "a sampling handle runs through dflash_select_run_sampled");
    if (B > 0 && (!target || !accept_len)) return fail(DFLASH_ERR_INVALID_ARG, "target and accept_len must not be NULL");
    return run_impl(h, hidden, anchor, B, nullptr, topk_ids, topk_vals, pair_scores, path, nullptr, path_score,
                    tie_flags, stream, target, accept_len, emitted);
}

dflash_status dflash_select_run_sampled(dflash_select_handle h, const void *hidden, const int32_t *anchor,
                                        int32_t B, const float *u_walk, int32_t *topk_ids, float *topk_vals,
                                        float *pair_scores, int32_t *path, float *draft_probs,
                                        float *path_score, uint8_t *tie_flags, void *stream)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    if (h->cfg.walk != DFLASH_WALK_SAMPLE)
        return fail(DFLASH_ERR_INVALID_ARG, "dflash_select_run_sampled needs a handle created with DFLASH_WALK_SAMPLE");
    if (B > 0 && (!u_walk || !draft_probs))
        return fail(DFLASH_ERR_INVALID_ARG, "u_walk and draft_probs must not be NULL");
    return run_impl(h, hidden, anchor, B, u_walk, topk_ids, topk_vals, pair_scores, path, draft_probs, path_score,
                    tie_flags, stream);
}

dflash_status dflash_verify_rejection(const int32_t *path, const int32_t *topk_ids, const float *draft_probs,
                                      const float *target_probs, const float *u_acc, const float *u_res, int32_t B,
                                      int32_t L, int32_t K, int64_t V, int32_t *accept_len, int32_t *emitted,
                                      void *stream)
{
    if (B < 0) return fail(DFLASH_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
    if (L < 1 || L > 16) return fail(DFLASH_ERR_INVALID_ARG, "L must be in [1, 16] (got %d)", L);
    if (K != 16 && K != 32) return fail(DFLASH_ERR_INVALID_ARG, "K must be 16 or 32 (got %d)", K);
    if (V < K || V >= (int64_t(1) << 31)) return fail(DFLASH_ERR_INVALID_ARG, "V must satisfy K <= V < 2^31");
    if (B == 0) return ok();
    if (!path || !topk_ids || !draft_probs || !target_probs || !u_acc || !u_res || !accept_len || !emitted)
        return fail(DFLASH_ERR_INVALID_ARG, "NULL argument");
    CUDA_TRY(dfl::launch_verify_rejection(path, topk_ids, draft_probs, target_probs, u_acc, u_res, B, L, K, V,
                                          accept_len, emitted, static_cast<cudaStream_t>(stream)));
    return ok();
}

dflash_status dflash_verify_prefix(const int32_t *path, const int32_t *target, int32_t B, int32_t L,
                                   int32_t *accept_len, int32_t *emitted, void *stream)
{
    if (B < 0) return fail(DFLASH_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
    if (L < 1 || L > 16) return fail(DFLASH_ERR_INVALID_ARG, "L must be in [1, 16] (got %d)", L);
    if (B == 0) return ok();
    if (!path || !target || !accept_len)
        return fail(DFLASH_ERR_INVALID_ARG, "path, target and accept_len must not be NULL");
    CUDA_TRY(dfl::launch_verify(path, target, B, L, accept_len, emitted, static_cast<cudaStream_t>(stream)));
    return ok();
}

// How long dflash_select_step_host polls its completion flags before it
// synchronises the stream instead (the kernels' own waits give up after 1 s).
constexpr int kHostWaitMs = 3000;

static dflash_status read_device_error(dflash_select_ctx *c, cudaStream_t s)
{
    CUDA_TRY(cudaMemcpyAsync(c->err_host, c->err, sizeof(int), cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    const int e = *c->err_host;
    if (e == 0) return ok();
    CUDA_TRY(cudaMemsetAsync(c->err, 0, sizeof(int), s));
    CUDA_TRY(cudaStreamSynchronize(s));
    if (e & dfl::DEV_ERR_TIMEOUT)
        return fail(DFLASH_ERR_TIMEOUT, "a kernel pipeline wait exceeded its time bound (device error word %d)", e);
    return fail(DFLASH_ERR_DEVICE_CHECK, "a token id outside [0, V) reached the selector (device error word %d)", e);
}

dflash_status dflash_select_step_host(dflash_select_handle h, const void *hidden_host, const int32_t *anchor_host,
                                      const int32_t *target_host, int32_t B, int32_t *path_host, int32_t *accept_host,
                                      int32_t *emitted_host, void *stream)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    dflash_select_ctx *c = h;
    if (B < 0 || B > c->cfg.max_batch)
        return fail(DFLASH_ERR_INVALID_ARG, "B must be in [0, max_batch=%d] (got %d)", c->cfg.max_batch, B);
    if (B == 0) return ok();
    if (!hidden_host || !anchor_host || !target_host || !path_host || !accept_host || !emitted_host)
        return fail(DFLASH_ERR_INVALID_ARG, "host buffers must not be NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int L = c->cfg.L;
    const size_t nb = static_cast<size_t>(B);
    // anchor and target are read by the kernels from the handle's mapped
    // pinned image; the previous call returned once its walkers, the last
    // readers of that image, had finished, so it is free
    uint8_t *const in_host = c->st_in_host;
    const size_t tgt_off = c->st_tgt_off;
    std::memcpy(in_host, anchor_host, nb * 4);
    std::memcpy(in_host + tgt_off, target_host, nb * (L + 1) * 4);
    const int32_t *anchor_dev = reinterpret_cast<const int32_t *>(c->st_in_dev);
    const int32_t *target_dev = reinterpret_cast<const int32_t *>(c->st_in_dev + tgt_off);
    CUDA_TRY(cudaMemcpyAsync(c->st_hidden, hidden_host, nb * L * c->cfg.d * 2, cudaMemcpyHostToDevice, s));
    // the walkers write the results, a copy of the error word and a flag per
    // sequence straight into the mapped block
    // never 0, the value the flags start with: after the counter wraps, a
    // sequence slot not used before must not read as finished
    if (++c->host_step == 0) c->host_step = 1;
    const uint32_t step = c->host_step;
    c->hs_done = c->hd_done;
    c->hs_err_snap = c->hd_err;
    c->hs_step = step;
    dflash_status st = dflash_select_run_verify(h, c->st_hidden, anchor_dev, B, target_dev, c->hd_path,
                                                c->hd_accept, c->hd_emitted, nullptr, nullptr, nullptr, nullptr,
                                                nullptr, stream);
    c->hs_done = nullptr;
    c->hs_err_snap = nullptr;
    if (st != DFLASH_OK) return st;
    // Wait for every sequence's flag (bounded; past the bound the stream is
    // synchronised and the device error word decides), then read the results.
    const auto t0 = std::chrono::steady_clock::now();
    bool all = false;
    for (uint32_t it = 0; !all; ++it) {
        all = true;
        for (int32_t b = 0; b < B && all; ++b)
            all = __atomic_load_n(c->ho_done + b, __ATOMIC_ACQUIRE) == step;
        if (!all && (it & 1023u) == 1023u &&
            std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(kHostWaitMs))
            break;
    }
    if (!all) {
        CUDA_TRY(cudaStreamSynchronize(s));
        st = read_device_error(c, s);
        if (st != DFLASH_OK) return st;
        for (int32_t b = 0; b < B; ++b)
            if (__atomic_load_n(c->ho_done + b, __ATOMIC_ACQUIRE) != step)
                return fail(DFLASH_ERR_CUDA, "sequence %d of the host step produced no results", b);
    }
    int e = 0;
    for (int32_t b = 0; b < B; ++b) e |= c->ho_err[b];
    if (e != 0) {
        CUDA_TRY(cudaStreamSynchronize(s));
        return read_device_error(c, s);  // reports and clears the latched word
    }
    std::memcpy(path_host, c->ho_path, nb * L * 4);
    std::memcpy(accept_host, c->ho_accept, nb * 4);
    std::memcpy(emitted_host, c->ho_emitted, nb * (L + 1) * 4);
    return ok();
}

dflash_status dflash_select_sync_status(dflash_select_handle h, void *stream)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    return read_device_error(h, static_cast<cudaStream_t>(stream));
}

dflash_status dflash_select_profile(dflash_select_handle h, int32_t enable)
{
    if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
    if (enable) prof_ensure(h);
    h->prof = enable != 0;
    if (enable) h->prof_runs = 0;
    return ok();
}

dflash_status dflash_select_profile_read(dflash_select_handle h, double *ms_total, int64_t *launches,
                                         int32_t max_kernels, int32_t *n_kernels)
{
    if (!h || !ms_total || !launches || !n_kernels) return fail(DFLASH_ERR_INVALID_ARG, "NULL argument");
    const int nk = max_kernels < kProfileKernels ? max_kernels : kProfileKernels;
    for (int k = 0; k < nk; ++k) {
        ms_total[k] = 0.0;
        launches[k] = 0;
    }
    for (int r = 0; r < h->prof_runs; ++r) {
        const ProfRun &pr = h->prof_rec[r];
        for (int slot = 0; slot < pr.n; ++slot) {
            cudaEvent_t *e = &h->ev[(static_cast<size_t>(r) * kProfileSlots + slot) * 2];
            CUDA_TRY(cudaEventSynchronize(e[1]));
            float ms = 0.f;
            CUDA_TRY(cudaEventElapsedTime(&ms, e[0], e[1]));
            if (pr.kid[slot] < nk) {
                ms_total[pr.kid[slot]] += ms;
                launches[pr.kid[slot]] += 1;
            }
        }
    }
    *n_kernels = nk;
    return ok();
}

int32_t dflash_select_launches_per_run(dflash_select_handle h, int32_t B)
{
    if (!h || B <= 0 || B > h->cfg.max_batch) return 0;
    const Plan pl = h->plan(B);
    return (pl.pilot_G > 0 ? 1 : 0) + (pl.fused_tail ? 2 : (h->tab ? 3 : (h->dd_tab ? 5 : 4)));
}

dflash_status dflash_select_destroy(dflash_select_handle h)
{
    if (!h) return ok();
    dflash_status st = DFLASH_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        st = fail(DFLASH_ERR_CUDA, "device synchronisation failed before destroy");
    } else {
        int e = 0;
        if (cudaMemcpy(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess && e != 0)
            st = (e & dfl::DEV_ERR_TIMEOUT) ? fail(DFLASH_ERR_TIMEOUT, "pending device timeout at destroy")
                                            : fail(DFLASH_ERR_DEVICE_CHECK, "pending out-of-range token at destroy");
    }
    for (auto &x : h->ev) cudaEventDestroy(x);
    cudaFreeHost(h->err_host);
    cudaFree(h->ws);
    cudaFree(h->tab);
    delete h;
    return st;
}

}  // extern "C"
