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

// Cluster primitives for the group exchange (one thread-block cluster per group, rank j = the
// group's particle j): distributed shared memory stores and mbarrier arrivals in the leader
// (rank 0), whose waits acquire at cluster scope.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* q) { return (uint32_t)__cvta_generic_to_shared(q); }
// The address of the same shared variable in the block of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_store(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// An arrival on an mbarrier of another block of the cluster, ordered after this thread's earlier
// stores (release at cluster scope).
__device__ __forceinline__ void cluster_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Wait (at most kClusterWaitNs) for phase `parity` of the block's own mbarrier, acquiring what
// the arriving blocks wrote before their arrivals.
constexpr unsigned long long kClusterWaitNs = 2000000000ull;
__device__ __forceinline__ bool cluster_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool cluster_wait(uint32_t bar, uint32_t parity) {
    if (cluster_try_wait(bar, parity)) return true;
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (cluster_try_wait(bar, parity)) return true;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > kClusterWaitNs) return false;
    }
}

// The fused step's group part for groups of at most kWarp particles, run by one block of the
// group: warp 0 computes the ESS and resamples into shared memory (one particle per lane), then
// all threads remap the group's page-table rows. The log-weights come from global memory, or from
// lw_in (shared memory) when given; the input page-table rows likewise from `stage` when given.
// Larger groups go to the stand-alone resampling and page-table kernels after this pass: their
// code kept out of this kernel, whose every SM runs it cold, keeps its instruction footprint
// small.
__device__ __forceinline__ void group_part(const StreamParams& p, int g, int32_t* sAnc, int* sRes,
                                           int bar, int nthr, const Exp2Table& T,
                                           const float* lw_in = nullptr, const int32_t* stage = nullptr) {
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
        if (!group_resample_fast(lw, N, p.ess_threshold, U, anc, ess, rs, lane, a0, res, lw_in)) {
            int a[1];
            res = group_resample_small<1>(lw, N, p.ess_threshold, U, anc, ess, rs, p.ws, lane, T, a, lw_in);
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
        remap_rows_block<4>(p, tin, tout, sAnc, res, N, P, nthr, stage);
    else
        remap_rows_block<1>(p, tin, tout, sAnc, res, N, P, nthr, stage);
}

// Bytes of the finishing kernel's dynamic shared memory before the staged page-table rows, and
// whether a group's rows are staged (cluster mode, at most kStageMaxBytes).
constexpr size_t kStageMaxBytes = 32 * 1024;
__host__ __device__ inline size_t finish_smem_base(const StreamParams& p, int mode) {
    const size_t b = (size_t)p.slots * (sizeof(float2) + sizeof(int) + sizeof(float)) +
                     (mode == kModeSMCStep ? (size_t)kWarp * sizeof(int32_t) : 0);
    return (b + 15) & ~(size_t)15;
}
__host__ __device__ inline bool finish_stages_table(const StreamParams& p) {
    return p.table_in != nullptr && (size_t)p.N * p.pages_per_seq * sizeof(int32_t) <= kStageMaxBytes;
}

// kCL (fused step, groups of 2..16 particles): the grid runs as one thread-block cluster per
// group. Each block hands its particle's new log-weight to the group's leader (cluster rank 0)
// by a distributed shared-memory store and an mbarrier arrival; the leader, which staged the
// group's page-table rows in its shared memory while the stream finished, then resamples and
// remaps. No global counter, fence or reload of the log-weights sits on the group's chain.
template <int DT, int MODE, bool kCL>
__global__ void __launch_bounds__(kFinishMaxWarps * kWarp)
    finish_kernel(const __grid_constant__ StreamParams p) {
    // dynamic shared memory: row normalisers, draft tokens and the logits there per row slot,
    // then (fused step) the group's ancestors, then (cluster leader) the group's page-table rows
    extern __shared__ __align__(16) unsigned char dsm[];
    float2* sL = reinterpret_cast<float2*>(dsm);
    int* sX = reinterpret_cast<int*>(sL + p.slots);
    float* sZ = reinterpret_cast<float*>(sX + p.slots);
    int32_t* sAnc = reinterpret_cast<int32_t*>(sZ + p.slots);
    __shared__ Exp2Table sT;
    __shared__ int sLast, sRes;
    __shared__ __align__(8) uint64_t sBar;  // (cluster leader) the group's log-weight arrivals
    __shared__ float sLwG[kWarp];           // (cluster leader) the group's new log-weights
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        sT.hi[i] = p.T.hi[i];
        sT.lo[i] = p.T.lo[i];
    }
    const int s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const bool leader = kCL && cluster_rank() == 0;
    int32_t* stage = nullptr;
    if (kCL) {
        if (leader && threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sBar)), "r"((unsigned)p.N)
                         : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        cluster_sync_all();  // the leader's barrier is initialised before any block arrives on it
    }
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
        if (leader && finish_stages_table(p)) {
            // the group's input page-table rows, into shared memory
            stage = reinterpret_cast<int32_t*>(dsm + finish_smem_base(p, MODE));
            const int n = p.N * p.pages_per_seq;
            const int32_t* tin = p.table_in + (size_t)s * p.pages_per_seq;
            if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(tin) & 15u) == 0) {
                for (int i = threadIdx.x; i < n / 4; i += blockDim.x)
                    reinterpret_cast<int4*>(stage)[i] = __ldg(reinterpret_cast<const int4*>(tin) + i);
            } else {
                for (int i = threadIdx.x; i < n; i += blockDim.x) stage[i] = __ldg(tin + i);
            }
        } else if (!kCL && MODE == kModeSMCStep && p.table_in && (int)threadIdx.x * 32 < p.pages_per_seq) {
            l2_prefetch(p.table_in + (size_t)s * p.pages_per_seq + threadIdx.x * 32);
        }
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
            const float lw = smc_particle_epilogue(p, s, lane, __shfl_sync(0xffffffffu, lw_old, 0), sL, sX, sZ);
            if (kCL) {
                if (lane == 0) {
                    // the leader's copy of this particle's log-weight, then the arrival
                    const uint32_t j = (uint32_t)(s % p.N);
                    cluster_store(cluster_map(smem_addr(&sLwG[j]), 0), lw);
                    cluster_arrive(cluster_map(smem_addr(&sBar), 0));
                }
            } else if (MODE == kModeSMCStep && p.N <= kWarp) {
                const bool last = arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_group) + s / p.N, (unsigned)p.N, lane);
                if (lane == 0) sLast = last ? 1 : 0;
            }
        }
    }
    if (MODE != kModeSMCStep || p.N > kWarp) return;
    if (kCL) {
        if (!leader) return;
        if (warp == 0) {
            const bool ok = __all_sync(0xffffffffu, cluster_wait(smem_addr(&sBar), 0u));
            if (lane == 0) {
                sLast = ok ? 1 : 0;
                if (!ok) raise_error(p.ws, kErrTimeout);
            }
        }
    }
    bar_sync(bar, nthr);
    if (sLast)  // (the block's shared copy of the exp table)
        group_part(p, s / p.N, sAnc, &sRes, bar, nthr, sT, kCL ? sLwG : nullptr, stage);
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
    const size_t smem = finish_smem_base(p, MODE);
    auto kern = finish_kernel<DT, MODE, false>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(reinterpret_cast<const void*>(kern), dim3((unsigned)p.R.S),
                            dim3((unsigned)(nw * kWarp)), smem, p, st);
}

// The fused step with one cluster per group (finish_kernel<DT, kModeSMCStep, true>), for groups
// of 2..16 particles of fixed-length sequences. Returns cudaErrorNotSupported, before launching
// anything, when this device cannot run such clusters (the caller then takes the counter path).
template <int DT>
static cudaError_t launch_finish_cluster_t(const StreamParams& p, cudaStream_t st) {
    const int nw = p.slots < kFinishMaxWarps ? p.slots : kFinishMaxWarps;
    const size_t smem = finish_smem_base(p, kModeSMCStep) +
                        (finish_stages_table(p) ? (size_t)p.N * p.pages_per_seq * sizeof(int32_t) : 0);
    auto kern = finish_kernel<DT, kModeSMCStep, true>;
    const void* fn = reinterpret_cast<const void*>(kern);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && p.N > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // (so that no later launch check reports this refusal)
        return cudaErrorNotSupported;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.R.S);
    cfg.blockDim = dim3((unsigned)(nw * kWarp));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.N;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // (the occupancy query takes the cluster shape alone)
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        return cudaErrorNotSupported;
    }
    cfg.numAttrs = 2;
    void* args[] = {const_cast<StreamParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Whether the fused step finishes with one cluster per group.
static bool finish_by_cluster(const StreamParams& p) {
    return p.mode == kModeSMCStep && p.N >= 2 && p.N <= 16 && !p.R.toff && p.R.S % p.N == 0;
}

cudaError_t launch_finish(const StreamParams& p, cudaStream_t st) {
    if (finish_by_cluster(p)) {
        const cudaError_t e = p.dtype == 0 ? launch_finish_cluster_t<0>(p, st) : launch_finish_cluster_t<1>(p, st);
        if (e != cudaErrorNotSupported) return e;
    }
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
