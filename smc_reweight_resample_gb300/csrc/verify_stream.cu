// verify_stream.cu -- the streaming pass over all target and draft logits rows, with the
// per-sequence epilogues run by the last warp to finish a sequence:
//   SD    ("Faster LLM Inference via Sequential Monte Carlo", sec. 1): row normalisers, the
//         ratio tests min(1, p/q) in position order, the acceptance length, and the hand-off of
//         the row (pair) to draw the final token from;
//   SMC   (same page, sec. 2 steps 3-4 and sec. 3): row normalisers, the log-weight update
//         sum_k log pi_k(x_k) - log q_k(x_k), the (K+1)-th token drawn from pi at row K;
//   step  additionally, per group of N particles (last particle of the group): effective
//         sample size, systematic resampling and the page-table remap with refcounts.
//
// Bandwidth: every logit is read from HBM exactly once, by one warp, with 16-byte loads of
// 512 contiguous bytes per instruction. The kernel is persistent (a grid of resident blocks
// striding over all chunks); sequences are laid out consecutively in the chunk order so that
// they complete, and run their epilogues, while other warps are still streaming.
#include "smcsd_launch.cuh"
#include "smcsd_sampling.cuh"

namespace smcsd {

constexpr int kStreamThreads = 256;

__device__ __forceinline__ void load_table_smem(const Exp2Table& src, Exp2Table& dst) {
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        dst.hi[i] = src.hi[i];
        dst.lo[i] = src.lo[i];
    }
    __syncthreads();
}

// log p(x) - log q(x) at position k of sequence s, given the two row normalisers.
template <int DT>
__device__ __forceinline__ double log_ratio(const StreamParams& p, int s, int k, double Lt,
                                            double Ld, bool& ok) {
    const Rows& R = p.R;
    const long long dr = drow_of(R, s, k);
    const int x = __ldg(R.toks + dr);
    if (x < 0 || x >= R.V) {
        raise_error(p.ws, kErrRange);
        ok = false;
        return 0.0;
    }
    const float zt = logit_at<DT>(row_ptr<DT>(R.tgt, trow_of(R, s, k), R.V), x);
    const float zd = logit_at<DT>(row_ptr<DT>(R.drf, dr, R.V), x);
    ok = true;
    return (p.sc_t.c * (double)zt - Lt) - (p.sc_d.c * (double)zd - Ld);
}

// SD: normalisers of all 2*ks+1 rows, acceptance length, hand-off to the drawing passes.
template <int DT>
__device__ void sd_seq_epilogue(const StreamParams& p, int s, int ks, int lane) {
    const Rows& R = p.R;
    const int cpr = p.cpr;
    const float2* fast = ws_ptr<float2>(p.ws, p.L.fast) + (size_t)s * p.slots * cpr;
    const float* u = p.uniforms + (size_t)s * (R.K + 1);
    int acc = ks;
    for (int k0 = 0; k0 < ks; k0 += 4) {
        const int nk = min(4, ks - k0);
        double Lt[4], Ld[4];
        rows_lse_fast4(fast + (size_t)(2 * k0) * cpr, 2 * cpr, nk, cpr, p.sc_t, lane, Lt);
        rows_lse_fast4(fast + (size_t)(2 * k0 + 1) * cpr, 2 * cpr, nk, cpr, p.sc_d, lane, Ld);
        bool rej = false;
        if (lane < nk) {
            const int k = k0 + lane;
            const double lt = pick4(Lt, lane), ld = pick4(Ld, lane);
            bool ok;
            const double ell = log_ratio<DT>(p, s, k, lt, ld, ok);
            const double a = exp(ell < 0.0 ? ell : 0.0);  // min(1, p/q)
            rej = !ok || !((double)__ldg(u + k) < a);
            if (p.lse_tgt) p.lse_tgt[trow_of(R, s, k)] = (float)lt;
            if (p.lse_drf) p.lse_drf[drow_of(R, s, k)] = (float)ld;
        }
        const unsigned b = __ballot_sync(0xffffffffu, rej);
        if (b && acc == ks) acc = k0 + __ffs(b) - 1;
    }
    double Lb[4];
    rows_lse_fast4(fast + (size_t)(2 * ks) * cpr, cpr, 1, cpr, p.sc_t, lane, Lb);
    if (lane == 0) {
        if (p.lse_tgt) p.lse_tgt[trow_of(R, s, ks)] = (float)Lb[0];
        p.accept_len[s] = acc;
        SeqState* st = ws_ptr<SeqState>(p.ws, p.L.seq) + s;
        st->mode = acc < ks ? 1 : 0;
        st->acc = acc;
        st->trow = trow_of(R, s, acc);
        st->drow = acc < ks ? drow_of(R, s, acc) : -1;
    }
}

// SMC: log-weight update and the (K+1)-th token of particle s.
template <int DT>
__device__ void smc_particle_epilogue(const StreamParams& p, const Exp2Table& T, int s,
                                      int lane) {
    const Rows& R = p.R;
    const int K = R.K, cpr = p.cpr;
    const float2* fast = ws_ptr<float2>(p.ws, p.L.fast) + (size_t)s * p.slots * cpr;
    double inc = 0.0;
    for (int k0 = 0; k0 < K; k0 += 4) {
        const int nk = min(4, K - k0);
        double Lt[4], Ld[4];
        rows_lse_fast4(fast + (size_t)(2 * k0) * cpr, 2 * cpr, nk, cpr, p.sc_t, lane, Lt);
        rows_lse_fast4(fast + (size_t)(2 * k0 + 1) * cpr, 2 * cpr, nk, cpr, p.sc_d, lane, Ld);
        double ell = 0.0;
        if (lane < nk) {
            const int k = k0 + lane;
            const double lt = pick4(Lt, lane), ld = pick4(Ld, lane);
            bool ok;
            ell = log_ratio<DT>(p, s, k, lt, ld, ok);
            if (p.lse_tgt) p.lse_tgt[trow_of(R, s, k)] = (float)lt;
            if (p.lse_drf) p.lse_drf[drow_of(R, s, k)] = (float)ld;
        }
        inc += warp_sum_d(ell);
    }
    // bonus token from pi at target row K
    const float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
    const float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kLoads;
    const long long rowK = trow_of(R, s, K);
    double lseK = 0.0;
    const int tok = draw_precise_row<DT>(tot, sub, cpr, row_ptr<DT>(R.tgt, rowK, R.V), R.V, p.vec,
                                         p.sc_t, T, __ldg(p.uniforms + s), p.ws, lane, &lseK);
    if (lane == 0) {
        p.logw[s] = (float)((double)__ldcg(p.logw + s) + inc);
        if (tok < 0) raise_error(p.ws, kErrNonfinite);
        p.bonus_token[s] = tok < 0 ? 0 : tok;
        if (p.lse_tgt) p.lse_tgt[rowK] = (float)lseK;
    }
}

// SMC step: ESS, systematic resampling and page-table remap of group g.
__device__ void smc_group_epilogue(const StreamParams& p, int g, int lane) {
    const int N = p.N;
    int32_t* anc = p.ancestors + (size_t)g * N;
    const bool res = group_resample(p.logw + (size_t)g * N, N, p.ess_threshold,
                                    __ldg(p.resample_uniforms + g), anc, p.ess ? p.ess + g : nullptr,
                                    p.resampled ? p.resampled + g : nullptr, p.ws, lane);
    __syncwarp();
    if (!p.table_in) return;
    const int P = p.pages_per_seq;
    const long long n = (long long)N * P;
    for (long long idx = lane; idx < n; idx += kWarp) {
        const int j = (int)(idx / P), col = (int)(idx - (long long)j * P);
        const int a = res ? anc[j] : j;
        const int32_t id = __ldg(p.table_in + ((size_t)g * N + a) * P + col);
        p.table_out[((size_t)g * N + j) * P + col] = id;
        if (p.refcount && id != -1) {
            if (id < 0 || id >= p.num_pages)
                raise_error(p.ws, kErrRange);
            else
                atomicAdd(p.refcount + id, 1);
        }
    }
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kStreamThreads)
    stream_kernel(const __grid_constant__ StreamParams p) {
    __shared__ Exp2Table sT;
    load_table_smem(p.T, sT);
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const long long nwarps = (long long)gridDim.x * wpb;
    const int per_seq = p.slots * p.cpr;
    unsigned* cnt_seq = ws_ptr<unsigned>(p.ws, p.L.cnt_seq1);
    for (long long it = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); it < p.items;
         it += nwarps) {
        const int s = (int)(it / per_seq);
        const int rem = (int)(it - (long long)s * per_seq);
        const int slot = rem / p.cpr, chunk = rem - slot * p.cpr;
        const int ks = seq_len(p.R, s, p.ws);
        if (ks < 0 || slot > 2 * ks) continue;
        const bool is_draft = slot < 2 * ks && (slot & 1);
        const int k = slot >> 1;
        const long long row = is_draft ? drow_of(p.R, s, k) : trow_of(p.R, s, k);
        const void* rp = row_ptr<DT>(is_draft ? p.R.drf : p.R.tgt, row, p.R.V);
        ChunkRegs<DT> r;
        if (p.vec)
            load_chunk<DT, true>(rp, p.R.V, chunk, lane, r);
        else
            load_chunk<DT, false>(rp, p.R.V, chunk, lane, r);
        const bool precise = MODE != kModeSD && slot == 2 * ks;
        if (!precise) {
            const float2 fp = fast_partial<DT>(r, is_draft ? p.sc_d.c2 : p.sc_t.c2, p.ws);
            if (lane == 0)
                ws_ptr<float2>(p.ws, p.L.fast)[((size_t)s * p.slots + slot) * p.cpr + chunk] = fp;
        } else {
            float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * p.cpr + chunk;
            float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + ((size_t)(s * 2) * p.cpr + chunk) * kLoads;
            precise_partials<DT>(r, p.sc_t, sT, p.ws, lane, tot, sub);
        }
        const unsigned expected = (unsigned)(2 * ks + 1) * (unsigned)p.cpr;
        if (arrive_last(cnt_seq + s, expected, lane)) {
            if (MODE == kModeSD) {
                sd_seq_epilogue<DT>(p, s, ks, lane);
            } else {
                smc_particle_epilogue<DT>(p, sT, s, lane);
                if (MODE == kModeSMCStep) {
                    const int g = s / p.N;
                    if (arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_group) + g, (unsigned)p.N, lane))
                        smc_group_epilogue(p, g, lane);
                }
            }
        }
    }
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
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kStreamThreads, 0);
    if (e != cudaSuccess) return e;
    const int wpb = kStreamThreads / kWarp;
    long long want = (p.items + wpb - 1) / wpb;
    long long cap = (long long)device_sm_count() * (occ > 0 ? occ : 1);
    int grid = (int)(want < cap ? want : cap);
    if (grid < 1) grid = 1;
    kern<<<grid, kStreamThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_stream(const StreamParams& p, cudaStream_t st) {
    if (p.dtype == 0) {
        if (p.mode == kModeSD) return launch_stream_t<0, kModeSD>(p, st);
        if (p.mode == kModeSMC) return launch_stream_t<0, kModeSMC>(p, st);
        return launch_stream_t<0, kModeSMCStep>(p, st);
    }
    if (p.mode == kModeSD) return launch_stream_t<1, kModeSD>(p, st);
    if (p.mode == kModeSMC) return launch_stream_t<1, kModeSMC>(p, st);
    return launch_stream_t<1, kModeSMCStep>(p, st);
}

}  // namespace smcsd
