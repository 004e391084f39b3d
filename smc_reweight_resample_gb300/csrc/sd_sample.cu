// sd_sample.cu -- the final token of speculative-decoding verify ("Faster LLM Inference via
// Sequential Monte Carlo", sec. 1, with the textbook rule): after the first pass has fixed the
// acceptance length, draw either the bonus token from p at the last target row, or the
// correction token from normalise(max(0, p - q)) at the rejected position, by inverse CDF.
//
// Pass 2 (sd_rows_kernel): double-float chunk sums of exp(z/T) over the row(s) to draw from.
//   Its per-sequence epilogue draws the bonus token directly, or turns the sums into the
//   reciprocal normalisers 1/Z_t, 1/Z_d that the residual needs.
// Pass 3 (sd_residual_kernel): double-float chunk sums of max(0, p_i - q_i); its epilogue draws
//   the correction token (or falls back to p at the same row if the residual has no mass).
// Both passes re-read one or two rows per sequence, which the first pass has just streamed.
#include "smcsd_launch.cuh"
#include "smcsd_sampling.cuh"

namespace smcsd {

constexpr int kSampleThreads = 256;

__device__ __forceinline__ void load_table_smem2(const Exp2Table& src, Exp2Table& dst) {
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        dst.hi[i] = src.hi[i];
        dst.lo[i] = src.lo[i];
    }
    __syncthreads();
}

// residual weight max(0, p_i - q_i) of one logit pair, p_i = exp(c zt) / Z_t etc.
struct ResidualCtx {
    Scale sc;
    int n_t, n_d;
    dd inv_t, inv_d;
};
__device__ __forceinline__ dd residual_weight(float zt, float zd, const ResidualCtx& c,
                                              const Exp2Table& T, void* ws) {
    ddx et, ed;
    dd pt{0.0f, 0.0f}, qd{0.0f, 0.0f};
    if (precise_exp(zt, c.sc, T, ws, et)) pt = dd_mul(scaled(et, c.n_t), c.inv_t);
    if (precise_exp(zd, c.sc, T, ws, ed)) qd = dd_mul(scaled(ed, c.n_d), c.inv_d);
    dd d = two_sum(pt.hi, -qd.hi);
    d.lo = f_add(d.lo, f_sub(pt.lo, qd.lo));
    d = two_sum(d.hi, d.lo);
    return d.hi > 0.0f ? d : dd{0.0f, 0.0f};
}

template <int DT>
struct ResidualSlice {
    const void* trow;
    const void* drow;
    int V;
    bool vec;
    ResidualCtx c;
    const Exp2Table* T;
    void* ws;
    __device__ __forceinline__ void operator()(int chunk, int sub, int lane,
                                               dd (&w)[Geo<DT>::kPerVec]) const {
        float xt[Geo<DT>::kPerVec], xd[Geo<DT>::kPerVec];
        if (vec) {
            load_slice<DT, true>(trow, V, chunk, sub, lane, xt);
            load_slice<DT, true>(drow, V, chunk, sub, lane, xd);
        } else {
            load_slice<DT, false>(trow, V, chunk, sub, lane, xt);
            load_slice<DT, false>(drow, V, chunk, sub, lane, xd);
        }
#pragma unroll
        for (int q = 0; q < Geo<DT>::kPerVec; ++q) w[q] = residual_weight(xt[q], xd[q], c, *T, ws);
    }
};

__device__ __forceinline__ ResidualCtx residual_ctx(const SeqState* st, const Scale& sc) {
    ResidualCtx c;
    c.sc = sc;
    c.n_t = __ldcg(&st->n_t);
    c.n_d = __ldcg(&st->n_d);
    c.inv_t = dd{__ldcg(&st->inv_t_hi), __ldcg(&st->inv_t_lo)};
    c.inv_d = dd{__ldcg(&st->inv_d_hi), __ldcg(&st->inv_d_lo)};
    return c;
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads) sd_rows_kernel(const __grid_constant__ SampleParams p) {
    __shared__ Exp2Table sT;
    load_table_smem2(p.T, sT);
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int cpr = p.cpr;
    const long long items = (long long)p.R.S * 2 * cpr;
    const long long nwarps = (long long)gridDim.x * wpb;
    SeqState* seq = ws_ptr<SeqState>(p.ws, p.L.seq);
    for (long long it = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); it < items; it += nwarps) {
        const int s = (int)(it / (2 * cpr));
        const int rem = (int)(it - (long long)s * 2 * cpr);
        const int which = rem / cpr, chunk = rem - which * cpr;
        if (seq_len(p.R, s, p.ws) < 0) continue;
        const int mode = __ldcg(&seq[s].mode);
        if (which == 1 && mode == 0) continue;
        const long long row = which == 0 ? __ldcg(&seq[s].trow) : __ldcg(&seq[s].drow);
        const void* rp = row_ptr<DT>(which == 0 ? p.R.tgt : p.R.drf, row, p.R.V);
        ChunkRegs<DT> r;
        if (p.vec)
            load_chunk<DT, true>(rp, p.R.V, chunk, lane, r);
        else
            load_chunk<DT, false>(rp, p.R.V, chunk, lane, r);
        float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2 + which) * cpr + chunk;
        float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + ((size_t)(s * 2 + which) * cpr + chunk) * kLoads;
        precise_partials<DT>(r, p.sc, sT, p.ws, lane, tot, sub);
        const unsigned expected = (unsigned)((mode == 1 ? 2 : 1) * cpr);
        if (!arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_seq2) + s, expected, lane)) continue;

        // epilogue of sequence s
        const float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
        const float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kLoads;
        if (mode == 0) {
            const float u = __ldg(p.uniforms + (size_t)s * (p.R.K + 1) + p.R.K);
            const int tok = draw_precise_row<DT>(tot_t, sub_t, cpr,
                                                 row_ptr<DT>(p.R.tgt, __ldcg(&seq[s].trow), p.R.V),
                                                 p.R.V, p.vec, p.sc, sT, u, p.ws, lane, nullptr);
            if (lane == 0) {
                if (tok < 0) raise_error(p.ws, kErrNonfinite);
                p.out_token[s] = tok < 0 ? 0 : tok;
            }
        } else {
            const float4* tot_d = tot_t + cpr;
            const int nt = row_exponent(tot_t, cpr, lane), nd = row_exponent(tot_d, cpr, lane);
            const dd Rt = row_total(tot_t, cpr, nt, lane), Rd = row_total(tot_d, cpr, nd, lane);
            if (lane == 0) {
                if (!(Rt.hi > 0.0f) || !(Rd.hi > 0.0f)) raise_error(p.ws, kErrNonfinite);
                const dd it_ = dd_recip(Rt), id_ = dd_recip(Rd);
                seq[s].n_t = nt;
                seq[s].n_d = nd;
                seq[s].inv_t_hi = it_.hi;
                seq[s].inv_t_lo = it_.lo;
                seq[s].inv_d_hi = id_.hi;
                seq[s].inv_d_lo = id_.lo;
            }
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads)
    sd_residual_kernel(const __grid_constant__ SampleParams p) {
    __shared__ Exp2Table sT;
    load_table_smem2(p.T, sT);
    constexpr int PV = Geo<DT>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int cpr = p.cpr;
    const long long items = (long long)p.R.S * cpr;
    const long long nwarps = (long long)gridDim.x * wpb;
    SeqState* seq = ws_ptr<SeqState>(p.ws, p.L.seq);
    for (long long it = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); it < items; it += nwarps) {
        const int s = (int)(it / cpr);
        const int chunk = (int)(it - (long long)s * cpr);
        if (seq_len(p.R, s, p.ws) < 0) continue;
        if (__ldcg(&seq[s].mode) != 1) continue;
        const long long tr = __ldcg(&seq[s].trow), dr = __ldcg(&seq[s].drow);
        const void* trp = row_ptr<DT>(p.R.tgt, tr, p.R.V);
        const void* drp = row_ptr<DT>(p.R.drf, dr, p.R.V);
        const ResidualCtx c = residual_ctx(seq + s, p.sc);
        dd total{0.0f, 0.0f};
        float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int v = 0; v < kLoads; ++v) {
            float xt[PV], xd[PV];
            if (p.vec) {
                load_slice<DT, true>(trp, p.R.V, chunk, v, lane, xt);
                load_slice<DT, true>(drp, p.R.V, chunk, v, lane, xd);
            } else {
                load_slice<DT, false>(trp, p.R.V, chunk, v, lane, xt);
                load_slice<DT, false>(drp, p.R.V, chunk, v, lane, xd);
            }
            dd acc{kBias, 0.0f};
#pragma unroll
            for (int q = 0; q < PV; ++q) acc_biased(acc, residual_weight(xt[q], xd[q], c, sT, p.ws));
            const dd sv = warp_sum_dd(unbias(acc));
            total = dd_add(total, sv);
            if (lane == v) mine = pack_part(sv, 0);
        }
        float4* tot = ws_ptr<float4>(p.ws, p.L.rtot) + (size_t)s * cpr;
        float4* sub = ws_ptr<float4>(p.ws, p.L.rsub) + (size_t)s * cpr * kLoads;
        if (lane < kLoads) sub[(size_t)chunk * kLoads + lane] = mine;
        if (lane == 0) tot[chunk] = pack_part(total, 0);
        if (!arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_seq3) + s, (unsigned)cpr, lane)) continue;

        // epilogue: draw from the residual, or from p at the same row if it has no mass
        const float u = __ldg(p.uniforms + (size_t)s * (p.R.K + 1) + p.R.K);
        const dd R = row_total(tot, cpr, 0, lane);
        int tok;
        if (R.hi > 0.0f) {
            ResidualSlice<DT> fn{trp, drp, p.R.V, p.vec, c, &sT, p.ws};
            tok = draw_inverse_cdf<PV>(tot, sub, cpr, Geo<DT>::kChunk, Geo<DT>::kSub, u, lane, fn,
                                       nullptr);
        } else {
            const float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
            const float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kLoads;
            tok = draw_precise_row<DT>(tot_t, sub_t, cpr, trp, p.R.V, p.vec, p.sc, sT, u, p.ws, lane,
                                       nullptr);
        }
        if (lane == 0) {
            if (tok < 0) raise_error(p.ws, kErrNonfinite);
            p.out_token[s] = tok < 0 ? 0 : tok;
        }
    }
}

template <typename Kern>
static int grid_for(Kern kern, long long warps_needed) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSampleThreads, 0) != cudaSuccess)
        occ = 1;
    const int wpb = kSampleThreads / kWarp;
    long long want = (warps_needed + wpb - 1) / wpb;
    long long cap = (long long)device_sm_count() * (occ > 0 ? occ : 1);
    long long g = want < cap ? want : cap;
    return (int)(g < 1 ? 1 : g);
}

template <int DT>
static cudaError_t launch_sd_sample_t(const SampleParams& p, cudaStream_t st) {
    auto k2 = sd_rows_kernel<DT>;
    k2<<<grid_for(k2, (long long)p.R.S * 2 * p.cpr), kSampleThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto k3 = sd_residual_kernel<DT>;
    k3<<<grid_for(k3, (long long)p.R.S * p.cpr), kSampleThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sd_sample(const SampleParams& p, cudaStream_t st) {
    return p.dtype == 0 ? launch_sd_sample_t<0>(p, st) : launch_sd_sample_t<1>(p, st);
}

}  // namespace smcsd
