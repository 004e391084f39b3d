// finish.cu -- the finishing pass after the streaming pass (smcsd_epilogue.cuh), one block per
// sequence, one warp per row: the row's normaliser from its chunk partials, or, for the bonus
// row of a particle, the drawn (K+1)-th token; then warp 0 runs the sequence epilogue (SD ratio
// tests and hand-off, or the SMC log-weight update). In the fused step the block of each group's
// last particle (a counter per group, release on arrival, acquire by the last) then computes the
// group's ESS and resampling on warp 0 and remaps its page-table rows with all threads.
//
// Running this after the stream instead of inside it keeps the stream free of per-chunk
// completion counts (each a device-scope release), and a block's barrier orders its rows before
// its sequence epilogue. The pass is launched as a programmatic dependent of the stream, so that
// its launch overlaps the stream's tail; it waits for the stream to complete before it reads
// anything the stream wrote.
//
// The bonus row's rescan evaluates the 64 weights of one lane block without the shared-memory
// exp table: the general path gives the same weights as the table (the table holds exactly its
// values), so the walk reproduces the streamed partials.
#include "smcsd_epilogue.cuh"

namespace smcsd {

constexpr int kFinishMaxWarps = 16;

// The fused step's group part for groups of at most kWarp particles, run by the block of the
// group's last particle: warp 0 computes the ESS and resamples into shared memory (one particle
// per lane), then all threads remap the group's page-table rows. Larger groups go to the
// stand-alone resampling and page-table kernels after this pass: their code kept out of this
// kernel, whose every SM runs it cold, keeps its instruction footprint small.
__device__ __forceinline__ void group_part(const StreamParams& p, int g, int32_t* sAnc, int* sRes,
                                           int bar, int nthr, const Exp2Table& T) {
    const int N = p.N;
    const int lane = threadIdx.x & 31;
    int32_t* anc = p.ancestors + (size_t)g * N;
    if (threadIdx.x < kWarp) {
        float* lw = p.logw + (size_t)g * N;
        float* ess = p.ess ? p.ess + g : nullptr;
        int32_t* rs = p.resampled ? p.resampled + g : nullptr;
        const float U = __ldg(p.resample_uniforms + g);
        int a0;
        bool res;
        if (!group_resample_fast(lw, N, p.ess_threshold, U, anc, ess, rs, lane, a0, res)) {
            int a[1];
            res = group_resample_small<1>(lw, N, p.ess_threshold, U, anc, ess, rs, p.ws, lane, T, a);
            a0 = a[0];
        }
        if (lane < N) sAnc[lane] = a0;
        if (lane == 0) *sRes = res ? 1 : 0;
    }
    bar_sync(bar, nthr);
    if (!p.table_in) return;
    const int P = p.pages_per_seq;
    const int32_t* tin = p.table_in + (size_t)g * N * P;
    int32_t* tout = p.table_out + (size_t)g * N * P;
    const bool res = *sRes != 0;
    if ((P & 3) == 0 && ((reinterpret_cast<uintptr_t>(tin) | reinterpret_cast<uintptr_t>(tout)) & 15u) == 0)
        remap_rows_block<4>(p, tin, tout, sAnc, res, N, P, nthr);
    else
        remap_rows_block<1>(p, tin, tout, sAnc, res, N, P, nthr);
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kFinishMaxWarps * kWarp)
    finish_kernel(const __grid_constant__ StreamParams p) {
    // dynamic shared memory: row normalisers, draft tokens and the logits there per row slot,
    // then (fused step) the group's ancestors
    extern __shared__ __align__(16) unsigned char dsm[];
    float2* sL = reinterpret_cast<float2*>(dsm);
    int* sX = reinterpret_cast<int*>(sL + p.slots);
    float* sZ = reinterpret_cast<float*>(sX + p.slots);
    int32_t* sAnc = reinterpret_cast<int32_t*>(sZ + p.slots);
    __shared__ Exp2Table sT;
    __shared__ int sLast, sRes;
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        sT.hi[i] = p.T.hi[i];
        sT.lo[i] = p.T.lo[i];
    }
    const int s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    // the next kernel on the stream may launch now; a programmatic dependent waits for this
    // kernel's completion before it touches memory
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int ks = seq_len(p.R, s, p.ws);
    // what does not depend on the streaming pass is read while it finishes
    float lw_old = 0.0f;
    if (ks >= 0) {
        for (int slot = warp; slot < 2 * ks; slot += nw)
            if (lane == 0) prefetch_token_logit<DT>(p, s, slot, sX, sZ);
        if (MODE != kModeSD && threadIdx.x == 0 && p.logw) lw_old = __ldcg(p.logw + s);
        if (MODE == kModeSMCStep && p.table_in && (int)threadIdx.x * 32 < p.pages_per_seq)
            l2_prefetch(p.table_in + (size_t)s * p.pages_per_seq + threadIdx.x * 32);
    }
    __syncthreads();
    griddep_wait();
    if (ks < 0) return;  // (the same on every thread of the block)
    const PreciseCtx P{p.sc_t, &sT, nullptr, p.ws, p.direct};
    for (int slot = warp; slot <= 2 * ks; slot += nw)
        if (!(p.drf_logq && slot < 2 * ks && (slot & 1)))  // (draft rows with a given log q)
            row_epilogue<DT, MODE>(p, P, s, slot, ks, lane, sL);
    // The sequence (and group) epilogue needs only the rows with a draft token. When the block has
    // a warp per row, the bonus row's warp (warp 2ks) keeps drawing while the others go on, meeting
    // at a named barrier without it; otherwise the whole block meets.
    // (The whole-sequence power target needs the bonus row's weight factor: no split then.)
    const bool split = MODE != kModeSD && nw == 2 * ks + 1 && ks > 0 && !p.target_seq;
    if (split && warp == 2 * ks) return;
    const int bar = split ? 1 : 0, nthr = split ? 2 * ks * kWarp : (int)blockDim.x;
    bar_sync(bar, nthr);
    if (warp == 0) {
        if (MODE == kModeSD) {
            sd_seq_epilogue(p, s, ks, lane, sL, sX, sZ, sT);
        } else {
            smc_particle_epilogue(p, s, lane, __shfl_sync(0xffffffffu, lw_old, 0), sL, sX, sZ);
            if (MODE == kModeSMCStep && p.N <= kWarp) {
                const bool last = arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_group) + s / p.N, (unsigned)p.N, lane);
                if (lane == 0) sLast = last ? 1 : 0;
            }
        }
    }
    if (MODE != kModeSMCStep || p.N > kWarp) return;
    bar_sync(bar, nthr);
    if (sLast) group_part(p, s / p.N, sAnc, &sRes, bar, nthr, sT);  // (the block's shared copy)
}

static cudaError_t launch_dependent(const void* kern, dim3 grid, dim3 block, size_t smem,
                                    const StreamParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<StreamParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int DT, int MODE>
static cudaError_t launch_finish_t(const StreamParams& p, cudaStream_t st) {
    const int nw = p.slots < kFinishMaxWarps ? p.slots : kFinishMaxWarps;
    const size_t smem = (size_t)p.slots * (sizeof(float2) + sizeof(int) + sizeof(float)) +
                        (MODE == kModeSMCStep ? (size_t)kWarp * sizeof(int32_t) : 0);
    auto kern = finish_kernel<DT, MODE>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(reinterpret_cast<const void*>(kern), dim3((unsigned)p.R.S),
                            dim3((unsigned)(nw * kWarp)), smem, p, st);
}

cudaError_t launch_finish(const StreamParams& p, cudaStream_t st) {
    if (p.dtype == 0) {
        if (p.mode == kModeSD) return launch_finish_t<0, kModeSD>(p, st);
        if (p.mode == kModeSMC) return launch_finish_t<0, kModeSMC>(p, st);
        return launch_finish_t<0, kModeSMCStep>(p, st);
    }
    if (p.mode == kModeSD) return launch_finish_t<1, kModeSD>(p, st);
    if (p.mode == kModeSMC) return launch_finish_t<1, kModeSMC>(p, st);
    return launch_finish_t<1, kModeSMCStep>(p, st);
}

}  // namespace smcsd
