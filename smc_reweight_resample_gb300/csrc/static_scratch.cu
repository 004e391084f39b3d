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
// Placement. The workspace of a call is the last ws_layout(G*N, K, V).total bytes of the area.
// The cached exp table is the last section of every layout and has the same size for every
// shape, so it sits at one address for all shapes, and no section of any other shape ever
// overlaps it: a table published by one call stays intact whatever shapes run in between, and
// its tag (the scale it was built for) decides alone whether a later call may copy it.
//
// Per call: the part of the workspace that must start at zero (error flag, completion and claim
// counters) is cleared on the stream first. The call then runs smc_step on that workspace and,
// if `status` is given, copies the call's device-side status (0 or a negative SMCSD_* code)
// there. No host-side state depends on the shape.
//
// Every call on one device uses the same scratch: calls whose device work may overlap (on
// different streams, or from several host threads without ordering) race on it and give wrong
// results. The first call on each device looks the scratch's address up (cudaGetSymbolAddress,
// with that device current); make that first call before any stream capture begins.
#include <atomic>

#include "smcsd.h"
#include "smcsd_internal.cuh"

namespace smcsd {

constexpr size_t kStaticScratchBytes = SMCSD_STATIC_SCRATCH_BYTES;
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

static std::atomic<void*> g_scratch_addr[kStaticMaxDevices];

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
    // the workspace ends where the area ends (L.total is a multiple of 256, so it stays aligned)
    ws = static_cast<char*>(ws) + (kStaticScratchBytes - L.total);
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, L.fast, st) != cudaSuccess) return SMCSD_ERR_CUDA;
    rc = smc_step(tgt_logits, drf_logits, dtype, draft_tokens, G, N, K, V, temperature, alpha,
                  bonus_uniforms, logw, bonus_token, ess_threshold, resample_uniforms, ancestors,
                  ess, resampled, table_in, table_out, pages_per_seq, refcount, num_pages, ws,
                  L.total, stream);
    if (rc) return rc;
    if (status && cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return SMCSD_ERR_CUDA;
    return SMCSD_OK;
}
