// dflash_lmhead_topk_noalloc: the lm_head + top-K stage of the selector for
// callers that may not allocate device memory.
//
// Some hosts embed this library where device memory is owned by someone else:
// an inference engine that hands out one preallocated arena, a process under a
// strict memory budget, or code running where a cudaMalloc would synchronise
// the device and is therefore forbidden. Such a caller cannot create a
// selector handle (dflash_select_init allocates the workspace). This entry
// point needs nothing but the caller's inputs and outputs. The scratch the
// lm_head kernel uses (per-CTA partial top-K lists, per-position thresholds,
// an error word, and the logit values when the caller does not want them)
// lives in one file-scope device array of fixed size, created when the
// library's kernels are loaded on a GPU and kept by that GPU until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "dflash_select.h"
#include "kernels.h"

namespace dfl {
dflash_status host_fail(dflash_status st, const char *msg);
dflash_status host_make_tmap(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols, int box_rows);
}  // namespace dfl

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;       // 4 MiB per GPU
constexpr size_t kErrOffset = 0;                        // device error word
constexpr size_t kThrOffset = 256;                      // u64 thresholds [N <= 256]
constexpr size_t kZeroBytes = kThrOffset + 256 * 8;     // what each call clears
constexpr size_t kValsOffset = kZeroBytes;              // fp32 [N <= 256][K <= 32]
constexpr size_t kPartOffset = kValsOffset + 256 * 32 * 4;
constexpr size_t kPartBytes = kScratchBytes - kPartOffset;
constexpr int kMaxPositions = 256;
constexpr int kMaxDevices = 64;

// The scratch. Host code must never pass `g_noalloc_scratch` itself to a
// kernel: on the host the name is only a stand-in for the symbol. Its device
// address comes from cudaGetSymbolAddress (per device, below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch
    int num_sms = 0;
    int smem_optin = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

dflash_status fail(dflash_status st, const char *fmt, long long a = 0, long long b = 0)
{
    char buf[256];
    snprintf(buf, sizeof buf, fmt, a, b);
    return dfl::host_fail(st, buf);
}

// Once per device, with that device current: find the scratch's device
// address and set the kernels' shared-memory opt-ins.
dflash_status setup_current_device(DeviceSetup *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(DFLASH_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device index %lld out of range", dev);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.scratch) {
        int major = 0, minor = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return fail(DFLASH_ERR_CUDA, "cudaDeviceGetAttribute failed on device %lld", dev);
        if (major != 10 || minor != 3)
            return fail(DFLASH_ERR_UNSUPPORTED, "built for sm_103 (GB300); device is sm_%lld%lld", major, minor);
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(DFLASH_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed (error %lld)", e);
        if (dfl::prepare_lmhead(optin) != cudaSuccess || dfl::prepare_topk_merge(optin) != cudaSuccess)
            return fail(DFLASH_ERR_CUDA, "setting the kernels' shared-memory limit failed");
        s.num_sms = sms;
        s.smem_optin = optin;
        s.scratch = static_cast<unsigned char *>(ptr);
    }
    *out = s;
    return DFLASH_OK;
}

}  // namespace

extern "C" dflash_status dflash_lmhead_topk_noalloc(const void *W_lm, int64_t V, int32_t d, const void *hidden,
                                                    int32_t N, int32_t K, int32_t *topk_ids, float *topk_vals,
                                                    int32_t *device_status, void *stream)
{
    if (N < 0) return fail(DFLASH_ERR_INVALID_ARG, "N must be >= 0 (got %lld)", N);
    if (N == 0) return DFLASH_OK;
    if (!W_lm || !hidden || !topk_ids) return fail(DFLASH_ERR_INVALID_ARG, "W_lm, hidden and topk_ids must not be NULL");
    if ((reinterpret_cast<uintptr_t>(W_lm) | reinterpret_cast<uintptr_t>(hidden)) & 15u)
        return fail(DFLASH_ERR_INVALID_ARG, "W_lm and hidden must be 16-byte aligned");
    if (K != 16 && K != 32) return fail(DFLASH_ERR_UNSUPPORTED, "K must be 16 or 32 (got %lld)", K);
    if (V < K || V >= (int64_t(1) << 31))
        return fail(DFLASH_ERR_UNSUPPORTED, "V must satisfy K <= V < 2^31 (got %lld)", V);
    if (d < 64 || d > 16384 || d % 64 != 0)
        return fail(DFLASH_ERR_UNSUPPORTED, "d must be a multiple of 64 in [64, 16384] (got %lld)", d);
    if (N > kMaxPositions)
        return fail(DFLASH_ERR_UNSUPPORTED, "N = %lld positions exceeds the %lld this entry point can hold", N,
                    kMaxPositions);

    DeviceSetup dev;
    dflash_status st = setup_current_device(&dev);
    if (st != DFLASH_OK) return st;

    // The selector's own tiling for up to 256 positions: position tiles of at
    // most 128 (the per-tile epilogue's range), each with its own share of the
    // SMs.
    const int n_tiles_n = (N + 127) / 128;
    const int NT = ((N + n_tiles_n - 1) / n_tiles_n + 15) / 16 * 16;
    const int m_tiles = static_cast<int>((V + dfl::kLmTileM - 1) / dfl::kLmTileM);
    int G = dev.num_sms / n_tiles_n;
    if (G < 1) G = 1;
    if (G > m_tiles) G = m_tiles;
    const size_t part_bytes = static_cast<size_t>(G) * N * K * sizeof(uint64_t);
    if (part_bytes > kPartBytes)
        return fail(DFLASH_ERR_UNSUPPORTED,
                    "N * K too large: the partial lists need %lld bytes, the fixed scratch holds %lld",
                    static_cast<long long>(part_bytes), static_cast<long long>(kPartBytes));

    dfl::LmHeadParams p;
    if ((st = dfl::host_make_tmap(&p.tm_w, W_lm, V, d, dfl::kLmTileM)) != DFLASH_OK) return st;
    p.tm_gate = p.tm_w;  // no gate tiles are scheduled (m_tiles_total == m_tiles_vocab)
    if ((st = dfl::host_make_tmap(&p.tm_h, hidden, N, d, NT)) != DFLASH_OK) return st;
    p.V = V;
    p.d = d;
    p.N = N;
    p.NT = NT;
    p.n_tiles_n = n_tiles_n;
    p.K = K;
    p.m_tiles_vocab = m_tiles;
    p.m_tiles_total = m_tiles;
    p.ctas_per_ntile = G;
    p.boxes = dfl::lmhead_boxes(d, NT);
    const size_t fixed = dfl::lmhead_smem_bytes(NT, K, 0, p.boxes);
    const size_t stage = static_cast<size_t>(p.boxes) *
                         (static_cast<size_t>(dfl::kLmTileM) * dfl::kLmTileK * 2 + static_cast<size_t>(NT) * dfl::kLmTileK * 2);
    int stages = static_cast<int>((static_cast<size_t>(dev.smem_optin) - fixed) / stage);
    if (stages > dfl::kLmMaxStages) stages = dfl::kLmMaxStages;
    p.stages = stages;
    p.part = reinterpret_cast<uint64_t *>(dev.scratch + kPartOffset);
    p.gate = nullptr;
    p.thr_g = reinterpret_cast<uint64_t *>(dev.scratch + kThrOffset);
    p.tmax = nullptr;  // no cross-CTA maxima (they would need per-call scratch)
    p.epoch = 0;
    p.err = reinterpret_cast<int *>(dev.scratch + kErrOffset);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word and the per-position thresholds must start at zero
    if (cudaMemsetAsync(dev.scratch, 0, kZeroBytes, s) != cudaSuccess)
        return fail(DFLASH_ERR_CUDA, "clearing the scratch failed");
    cudaError_t e = dfl::launch_lmhead_topk(p, G * n_tiles_n, dfl::lmhead_smem_bytes(NT, K, stages, p.boxes), s);
    if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "lm_head kernel launch failed (error %lld)", e);
    float *vals = topk_vals ? topk_vals : reinterpret_cast<float *>(dev.scratch + kValsOffset);
    e = dfl::launch_topk_merge(p.part, G, N, K, topk_ids, vals, nullptr, nullptr, p.thr_g, s);
    if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "merge kernel launch failed (error %lld)", e);
    if (device_status &&
        cudaMemcpyAsync(device_status, p.err, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return fail(DFLASH_ERR_CUDA, "copying the device status failed");
    return DFLASH_OK;
}
