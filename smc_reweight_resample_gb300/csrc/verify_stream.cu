// verify_stream.cu -- the streaming pass over all target and draft logits rows with direct
// global loads, used when the rows are not 16-byte aligned (the aligned case runs the TMA
// pipeline in stream_tma.cu). Same chunk partials and epilogues (smcsd_epilogue.cuh).
//
// One 640-thread block per SM, 20 warps claiming chunks from the grid-wide dealing as they become
// free; every logit is read from HBM exactly once. Rows that are drawn from (the (K+1)-th target row of each particle) take
// the precise path with the block's shared-memory exp table.
#include "smcsd_epilogue.cuh"

namespace smcsd {

constexpr int kStreamThreads = 640;

template <int DT, int MODE>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(const __grid_constant__ StreamParams p) {
    constexpr bool kPrecise = MODE != kModeSD;
    __shared__ Exp2Table sT;
    extern __shared__ __align__(16) float2 sTab[];  // kTabSize entries when the table is used
    if (MODE == kModeSMCStep) zero_refcount(p);
    load_exp2_table(p.T, sT);
    PreciseCtx P{p.sc_t, &sT, nullptr, p.ws, p.direct};
    if (kPrecise && DT == 1 && p.use_table) {
        setup_exp_table(sTab, p.sc_t, &sT, p.ws, ws_ptr<uint32_t>(p.ws, p.L.tab),
                        ws_ptr<float2>(p.ws, p.L.tab + 16), p.direct, threadIdx.x, blockDim.x, 0);
        P.tab = sTab;
    }
    // Items (chunks, sequence-major) are dealt dynamically: warp w of every block claims the next
    // chunk of stripe w (chunks w, w + W, w + 2W, ... for W warps per block) from a grid-wide
    // counter, and claims its following chunk before it works on the current one.
    if (threadIdx.x == 0) griddep_launch_dependents();
    constexpr int W = kStreamThreads / kWarp;
    unsigned* claim = ws_ptr<unsigned>(p.ws, p.L.claim);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t pol = l2_evict_first();
    long long nxt = 0;
    if (lane == 0) nxt = claim_item(claim, warp, W, p.items);
    nxt = __shfl_sync(0xffffffffu, nxt, 0);
    for (;;) {
        const long long it = nxt;
        if (it < 0) break;
        if (lane == 0) nxt = claim_item(claim, warp, W, p.items);
        nxt = __shfl_sync(0xffffffffu, nxt, 0);
        const ChunkRef c = chunk_ref(p, (uint32_t)it);
        if (!c.valid) continue;
        const int s = c.s, slot = c.slot, chunk = c.chunk, ks = c.ks;
        const bool is_draft = c.is_draft;
        const void* rp = row_ptr<DT>(is_draft ? p.R.drf : p.R.tgt, c.row, p.R.V);
        if (!kPrecise || slot != 2 * ks) {
            uint4 raw[kLoads];
            load_chunk_interleaved<DT>(rp, p.R.V, p.vec, chunk, lane, raw, pol);
            const float2 fp = fast_partial<DT>(raw, is_draft ? p.sc_d.c2 : p.sc_t.c2, p.ws);
            if (lane == 0)
                ws_ptr<float2>(p.ws, p.L.fast)[((size_t)s * p.slots + slot) * p.cpr + chunk] = fp;
        } else {
            float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * p.cpr + chunk;
            float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + ((size_t)(s * 2) * p.cpr + chunk) * kSubs;
            precise_partials<DT>(rp, p.R.V, p.vec, chunk, lane, P, tot, sub);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) reset_claims(claim, W);
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

template <int DT, int MODE>
static cudaError_t launch_stream_t(const StreamParams& p, cudaStream_t st) {
    auto kern = stream_kernel<DT, MODE>;
    const int wpb = kStreamThreads / kWarp;
    const long long want = (p.items + wpb - 1) / wpb;
    const long long cap = device_sm_count();
    int grid = (int)(want < cap ? want : cap);
    if (grid < 1) grid = 1;
    const size_t smem = (MODE != kModeSD && DT == 1 && p.use_table) ? (size_t)kTabSize * sizeof(float2) : 0;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kStreamThreads, smem, st>>>(p);
    return cudaGetLastError();
}

static cudaError_t launch_stream_pass(const StreamParams& p, cudaStream_t st) {
    if (p.vec) return launch_stream_tma(p, st);
    if (p.dtype == 0) {
        if (p.mode == kModeSD) return launch_stream_t<0, kModeSD>(p, st);
        if (p.mode == kModeSMC) return launch_stream_t<0, kModeSMC>(p, st);
        return launch_stream_t<0, kModeSMCStep>(p, st);
    }
    if (p.mode == kModeSD) return launch_stream_t<1, kModeSD>(p, st);
    if (p.mode == kModeSMC) return launch_stream_t<1, kModeSMC>(p, st);
    return launch_stream_t<1, kModeSMCStep>(p, st);
}

cudaError_t launch_stream(const StreamParams& p, cudaStream_t st) {
    cudaError_t e = launch_stream_pass(p, st);
    if (e == cudaSuccess) e = launch_finish(p, st);
    if (e != cudaSuccess || p.mode != kModeSMCStep || p.N <= kWarp) return e;
    // groups too large for the finishing pass's one-warp group part
    const ResampleParams rp{p.logw, p.G, p.N, p.ess_threshold, p.resample_uniforms, p.ancestors,
                            p.ess, p.resampled, p.ws, p.T};
    e = launch_resample(rp, st);
    if (e != cudaSuccess || !p.table_in) return e;
    const RemapParams mp{p.ancestors, p.resampled, p.G, p.N, p.table_in, p.table_out,
                         p.pages_per_seq, p.refcount, p.num_pages, p.ws};
    return launch_remap(mp, st);
}

}  // namespace smcsd
