// static_scratch.cu -- smc_step_static: the fused SMC-SD step with its scratch in a fixed area of
// device memory owned by this library, for callers that cannot hand in a workspace.
//
// Some callers have no way to allocate device memory for a workspace, or must not: a plain C host
// program without a device allocator, a plugin that may not touch its host's allocator or memory
// pools, a serving step whose device memory was planned once up front. This entry point gives
// them the same step as smc_step with nothing allocated by the call: the scratch lives in a
// file-scope device array of kStaticScratchBytes (32 MiB), set aside when the library's device
// code is loaded.
//
// Per call: the part of the scratch that must start at zero (error flag, completion and claim
// counters) is cleared on the stream first; when the problem's shape differs from the previous
// call on this device, the tag of the cached exp table is cleared too, since the table then sits
// at another offset. The call then runs smc_step on that scratch and, if `status` is given,
// copies the call's device-side status (0 or a negative SMCSD_* code) there.
//
// Every call on one device uses the same scratch: calls whose device work may overlap (on
// different streams, or from several host threads without ordering) race on it and give wrong
// results. The first call on each device looks the scratch's address up (cudaGetSymbolAddress,
// with that device current); make that first call before any stream capture begins.
#include <atomic>
#include <mutex>

#include "smcsd.h"
#include "smcsd_internal.cuh"

namespace smcsd {

constexpr size_t kStaticScratchBytes = SMCSD_STATIC_SCRATCH_BYTES;
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

struct StaticShape {
    int S, K, V;
};

static std::atomic<void*> g_scratch_addr[kStaticMaxDevices];
static std::mutex g_shape_mu;
static StaticShape g_last_shape[kStaticMaxDevices];
static bool g_have_shape[kStaticMaxDevices];

// Device address of the scratch on the current device, looked up once per device.
static int scratch_address(int dev, void** out) {
    void* a = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_step_scratch) != cudaSuccess || !a) return SMCSD_ERR_CUDA;
        g_scratch_addr[dev].store(a, std::memory_order_release);
    }
    *out = a;
    return SMCSD_OK;
}

// True if (S, K, V) differs from the previous call's on this device (and records it).
static bool shape_changed(int dev, int S, int K, int V) {
    std::lock_guard<std::mutex> lock(g_shape_mu);
    const StaticShape& last = g_last_shape[dev];
    const bool changed = !g_have_shape[dev] || last.S != S || last.K != K || last.V != V;
    g_last_shape[dev] = StaticShape{S, K, V};
    g_have_shape[dev] = true;
    return changed;
}

}  // namespace smcsd

using namespace smcsd;

extern "C" int smc_step_static(const void* tgt_logits, const void* drf_logits, int dtype,
                               const int32_t* draft_tokens, int G, int N, int K, int V,
                               float temperature, float alpha, const float* bonus_uniforms,
                               float* logw, int32_t* bonus_token, float ess_threshold,
                               const float* resample_uniforms, int32_t* ancestors, float* ess,
                               int32_t* resampled, const int32_t* table_in, int32_t* table_out,
                               int pages_per_seq, int32_t* refcount, int num_pages,
                               int32_t* status, void* stream) {
    if (G <= 0 || N <= 0 || K < 0 || V <= 0 || (long long)G * N > 0x7fffffffLL)
        return SMCSD_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(G * N, K, V);
    if (L.total > kStaticScratchBytes) return SMCSD_ERR_WORKSPACE;  // problem too large for it
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMCSD_ERR_CUDA;
    if (dev < 0 || dev >= kStaticMaxDevices) return SMCSD_ERR_CUDA;
    void* ws = nullptr;
    int rc = scratch_address(dev, &ws);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, L.fast, st) != cudaSuccess) return SMCSD_ERR_CUDA;
    if (shape_changed(dev, G * N, K, V) &&
        cudaMemsetAsync(static_cast<char*>(ws) + L.tab, 0, 16, st) != cudaSuccess)
        return SMCSD_ERR_CUDA;
    rc = smc_step(tgt_logits, drf_logits, dtype, draft_tokens, G, N, K, V, temperature, alpha,
                  bonus_uniforms, logw, bonus_token, ess_threshold, resample_uniforms, ancestors,
                  ess, resampled, table_in, table_out, pages_per_seq, refcount, num_pages, ws,
                  L.total, stream);
    if (rc) return rc;
    if (status && cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return SMCSD_ERR_CUDA;
    return SMCSD_OK;
}
