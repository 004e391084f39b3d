// finish.cu -- the finishing passes after the streaming pass (smcsd_epilogue.cuh):
//   finish_kernel  one block per sequence, one warp per row: the row's normaliser from its
//                  chunk partials, or, for the bonus row of a particle, the drawn (K+1)-th
//                  token; then warp 0 runs the sequence epilogue (SD ratio tests and hand-off, or
//                  the SMC log-weight update);
//   group_kernel   (fused step) one block per group: warp 0 computes the ESS and resamples, then
//                  all warps remap the group's page-table rows.
//
// Running these after the stream instead of inside it keeps the stream free of per-chunk
// completion counts (each a device-scope release), and a block's barrier orders its rows before
// its sequence epilogue, so no counter or fence is needed here either. Each pass is launched as a
// programmatic dependent of the one before, so that its launch overlaps that pass's tail; it
// waits for the earlier pass to complete before it reads anything the earlier pass wrote.
//
// The bonus row's rescan evaluates the 64 weights of one lane block without the shared-memory
// exp table: the general path gives the same weights as the table (the table holds exactly its
// values), so the walk reproduces the streamed partials.
#include "smcsd_epilogue.cuh"

namespace smcsd {

constexpr int kFinishMaxWarps = 32;
constexpr int kGroupThreads = 256;

template <int DT, int MODE>
__global__ void __launch_bounds__(kFinishMaxWarps * kWarp)
    finish_kernel(const __grid_constant__ StreamParams p) {
    __shared__ Exp2Table sT;
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        sT.hi[i] = p.T.hi[i];
        sT.lo[i] = p.T.lo[i];
    }
    __syncthreads();
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
    const PreciseCtx P{p.sc_t, &sT, nullptr, p.ws, p.direct};
    const int s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int ks = seq_len(p.R, s, p.ws);
    if (ks < 0) return;  // (the same on every thread of the block)
    for (int slot = warp; slot <= 2 * ks; slot += nw) row_epilogue<DT, MODE>(p, P, s, slot, ks, lane);
    __syncthreads();
    if (warp != 0) return;
    if (MODE == kModeSD)
        sd_seq_epilogue(p, s, ks, lane);
    else
        smc_particle_epilogue(p, s, lane);
}

__global__ void __launch_bounds__(kGroupThreads) group_kernel(const __grid_constant__ StreamParams p) {
    extern __shared__ int32_t sAnc[];  // [N]
    __shared__ int sRes;
    griddep_wait();
    const int g = blockIdx.x, N = p.N;
    const int lane = threadIdx.x & 31;
    int32_t* anc = p.ancestors + (size_t)g * N;
    if (threadIdx.x < kWarp) {
        float* lw = p.logw + (size_t)g * N;
        float* ess = p.ess ? p.ess + g : nullptr;
        int32_t* rs = p.resampled ? p.resampled + g : nullptr;
        const float U = __ldg(p.resample_uniforms + g);
        bool res;
        if (N <= kWarp * kResamplePer) {
            int anc_reg[kResamplePer];
            res = group_resample_small(lw, N, p.ess_threshold, U, anc, ess, rs, p.ws, lane, p.T, anc_reg);
            const int per = (N + kWarp - 1) / kWarp;
#pragma unroll
            for (int q = 0; q < kResamplePer; ++q)
                if (q < per && lane * per + q < N) sAnc[lane * per + q] = anc_reg[q];
        } else {
            res = group_resample_general(lw, N, p.ess_threshold, U, anc, ess, rs, p.ws, lane);
            __syncwarp();
            for (int j = lane; j < N; j += kWarp) sAnc[j] = __ldcg(anc + j);
        }
        if (lane == 0) sRes = res ? 1 : 0;
    }
    __syncthreads();
    if (!p.table_in) return;
    const int P = p.pages_per_seq;
    const int32_t* tin = p.table_in + (size_t)g * N * P;
    int32_t* tout = p.table_out + (size_t)g * N * P;
    const bool res = sRes != 0;
    if ((P & 3) == 0 && ((reinterpret_cast<uintptr_t>(tin) | reinterpret_cast<uintptr_t>(tout)) & 15u) == 0)
        remap_rows_block<4>(p, tin, tout, sAnc, res, N, P);
    else
        remap_rows_block<1>(p, tin, tout, sAnc, res, N, P);
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
    cudaError_t e = launch_dependent(reinterpret_cast<const void*>(finish_kernel<DT, MODE>),
                                     dim3((unsigned)p.R.S), dim3((unsigned)(nw * kWarp)), 0, p, st);
    if (e != cudaSuccess || MODE != kModeSMCStep) return e;
    const size_t smem = (size_t)p.N * sizeof(int32_t);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(reinterpret_cast<const void*>(group_kernel), dim3((unsigned)p.G),
                            dim3(kGroupThreads), smem, p, st);
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
