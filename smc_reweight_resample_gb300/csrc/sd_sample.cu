// sd_sample.cu -- the final token of speculative-decoding verify ("Faster LLM Inference via
// Sequential Monte Carlo", sec. 1, with the textbook rule): after the first pass has fixed the
// acceptance length, draw either the bonus token from p at the last target row, or the
// correction token from normalise(max(0, p - q)) at the rejected position, by inverse CDF.
//
// Rows 16-byte aligned (the common case): one more pipelined pass (stream_tma.cu, kModeSDFinal)
// over the (target, draft) row pair each sequence draws from gives the precise partials of a
// bonus row, or, for a rejected position, per lane block the double-float sums of exp(c z_t) and
// exp(c z_d) over all positions (the two normalisers) and over the positions with
// z_t - z_d > theta = (L_t - L_d) / c, which are exactly those with p_i > q_i up to the float
// accuracy of theta (a position that close to the boundary has a residual of at most ~1e-6 of its
// p_i). sd_final_finish_kernel then draws: the residual's chunk and lane-block masses are
// A / Z_t - B / Z_d, and the one lane block it rescans takes max(0, p_i - q_i) position by
// position.
// Rows not aligned: the direct-load passes below. Pass 2 (sd_rows_kernel): double-float chunk
// sums of exp(z/T) over the row(s) to draw from; its per-sequence epilogue draws the bonus token
// directly, or turns the sums into the reciprocal normalisers 1/Z_t, 1/Z_d that the residual
// needs. Pass 3 (sd_residual_kernel): double-float sums of max(0, p_i - q_i) per lane block; its
// epilogue draws the correction token (or falls back to p at the same row if the residual has no
// mass).
// The final-token passes re-read one or two rows per sequence, which the first pass has just
// streamed.
#include "smcsd_epilogue.cuh"

namespace smcsd {

constexpr int kSampleThreads = 256;  // three blocks per SM beside the 62 KB exp table

template <int DT>
struct ResidualBlock {
    const void* trow;
    const void* drow;
    int V;
    ResidualCtx c;
    PreciseCtx P;
    static constexpr int PL = Geo<DT>::kSub / kWarp;
    __device__ __forceinline__ void operator()(int chunk, int sub, int lane, int, dd (&w)[PL]) const {
        const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)sub * Geo<DT>::kSub + lane * PL;
#pragma unroll
        for (int q = 0; q < PL; ++q) {
            const long long e = e0 + q;
            w[q] = e < V ? residual_weight<DT>(logit_bits<DT>(trow, e), logit_bits<DT>(drow, e), c, P)
                         : dd{0.0f, 0.0f};
        }
    }
    __device__ __forceinline__ void prefetch(int chunk, int lane) const {
        const long long e = (long long)chunk * Geo<DT>::kChunk + (long long)lane * (128 / Geo<DT>::kBytes);
        if (chunk >= 0 && e < V) {
            l2_prefetch(static_cast<const char*>(trow) + e * Geo<DT>::kBytes);
            l2_prefetch(static_cast<const char*>(drow) + e * Geo<DT>::kBytes);
        }
    }
};


__device__ __forceinline__ void load_exp2_table_s(const Exp2Table& src, Exp2Table& dst) {
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        dst.hi[i] = src.hi[i];
        dst.lo[i] = src.lo[i];
    }
    __syncthreads();
}

template <int DT>
__device__ __noinline__ void sd_rows_epilogue(const SampleParams& p, const PreciseCtx& P, int s,
                                              int mode, int lane) {
    const int cpr = p.cpr;
    SeqState* seq = ws_ptr<SeqState>(p.ws, p.L.seq);
    const float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
    const float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kSubs;
    if (mode == 0) {
        const float u = __ldg(p.uniforms + (size_t)s * (p.R.K + 1) + p.R.K);
        const int tok = draw_precise_row<DT>(tot_t, sub_t, cpr,
                                             row_ptr<DT>(p.R.tgt, __ldcg(&seq[s].trow), p.R.V),
                                             p.R.V, P, u, lane, nullptr);
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

template <int DT>
__global__ void __launch_bounds__(kSampleThreads, 3) sd_rows_kernel(const __grid_constant__ SampleParams p) {
    __shared__ Exp2Table sT;
    extern __shared__ __align__(16) float2 sTab[];  // kTabSize entries when the table is used
    load_exp2_table_s(p.T, sT);
    PreciseCtx P{p.sc, &sT, nullptr, p.ws, p.direct};
    if (DT == 1 && p.use_table) {
        setup_exp_table(sTab, p.sc, &sT, p.ws, ws_ptr<uint32_t>(p.ws, p.L.tab),
                        ws_ptr<float2>(p.ws, p.L.tab + 16), p.direct, threadIdx.x, blockDim.x, 0);
        P.tab = sTab;
    }
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
        float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2 + which) * cpr + chunk;
        float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + ((size_t)(s * 2 + which) * cpr + chunk) * kSubs;
        precise_partials<DT, true>(rp, p.R.V, p.vec, chunk, lane, P, tot, sub);
        const unsigned expected = (unsigned)((mode == 1 ? 2 : 1) * cpr);
        if (arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_seq2) + s, expected, lane))
            sd_rows_epilogue<DT>(p, P, s, mode, lane);
    }
}

template <int DT>
__device__ __noinline__ void sd_residual_epilogue(const SampleParams& p, const PreciseCtx& P,
                                                  const ResidualCtx& c, int s, const void* trp,
                                                  const void* drp, int lane) {
    const int cpr = p.cpr;
    const float4* tot = ws_ptr<float4>(p.ws, p.L.rtot) + (size_t)s * cpr;
    const float4* sub = ws_ptr<float4>(p.ws, p.L.rsub) + (size_t)s * cpr * kSubs;
    const float u = __ldg(p.uniforms + (size_t)s * (p.R.K + 1) + p.R.K);
    const dd R = row_total(tot, cpr, 0, lane);
    int tok;
    if (R.hi > 0.0f) {
        ResidualBlock<DT> fn{trp, drp, p.R.V, c, P};
        tok = draw_inverse_cdf<ResidualBlock<DT>::PL>(tot, sub, cpr, Geo<DT>::kChunk, Geo<DT>::kSub, u,
                                                      lane, fn, nullptr);
    } else {
        const float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
        const float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kSubs;
        tok = draw_precise_row<DT>(tot_t, sub_t, cpr, trp, p.R.V, P, u, lane, nullptr);
    }
    if (lane == 0) {
        if (tok < 0) raise_error(p.ws, kErrNonfinite);
        p.out_token[s] = tok < 0 ? 0 : tok;
    }
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads, 3)
    sd_residual_kernel(const __grid_constant__ SampleParams p) {
    __shared__ Exp2Table sT;
    extern __shared__ __align__(16) float2 sTab[];  // kTabSize entries when the table is used
    load_exp2_table_s(p.T, sT);
    PreciseCtx P{p.sc, &sT, nullptr, p.ws, p.direct};
    if (DT == 1 && p.use_table) {
        setup_exp_table(sTab, p.sc, &sT, p.ws, ws_ptr<uint32_t>(p.ws, p.L.tab),
                        ws_ptr<float2>(p.ws, p.L.tab + 16), p.direct, threadIdx.x, blockDim.x, 0);
        P.tab = sTab;
    }
    constexpr int SUB = Geo<DT>::kSub;
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
        const void* trp = row_ptr<DT>(p.R.tgt, __ldcg(&seq[s].trow), p.R.V);
        const void* drp = row_ptr<DT>(p.R.drf, __ldcg(&seq[s].drow), p.R.V);
        const ResidualCtx c = residual_ctx(seq + s, P);
        // this lane's block of SUB logits: with 16-byte loads when both rows allow them (the
        // next piece of each row in flight while the current one is weighed), else logit by logit
        const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)lane * SUB;
        dd acc{kBias, 0.0f};
        if (p.vec && __all_sync(0xffffffffu, e0 + SUB <= p.R.V)) {
            constexpr int PERP = 16 / Geo<DT>::kBytes;
            const uint4* bt = reinterpret_cast<const uint4*>(static_cast<const char*>(trp) + e0 * Geo<DT>::kBytes);
            const uint4* bd = reinterpret_cast<const uint4*>(static_cast<const char*>(drp) + e0 * Geo<DT>::kBytes);
            uint4 ct = __ldg(bt), cd = __ldg(bd);
#pragma unroll 1
            for (int i = 0; i < kLoads; ++i) {
                uint4 nt = ct, nd = cd;
                if (i + 1 < kLoads) {
                    nt = __ldg(bt + i + 1);
                    nd = __ldg(bd + i + 1);
                }
                const uint32_t wt[4] = {ct.x, ct.y, ct.z, ct.w}, wd[4] = {cd.x, cd.y, cd.z, cd.w};
#pragma unroll
                for (int q = 0; q < PERP; ++q) {
                    const uint32_t xt = DT == 1 ? ((q & 1) ? (wt[q >> 1] >> 16) : (wt[q >> 1] & 0xffffu)) : wt[q];
                    const uint32_t xd = DT == 1 ? ((q & 1) ? (wd[q >> 1] >> 16) : (wd[q >> 1] & 0xffffu)) : wd[q];
                    acc_biased(acc, residual_weight<DT>(xt, xd, c, P));
                }
                acc = fast_two_sum(acc.hi, acc.lo);
                ct = nt;
                cd = nd;
            }
        } else {
#pragma unroll 1
            for (int q0 = 0; q0 < SUB; q0 += 16) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const long long e = e0 + q0 + q;
                    if (e < p.R.V)
                        acc_biased(acc, residual_weight<DT>(logit_bits<DT>(trp, e), logit_bits<DT>(drp, e), c, P));
                }
                acc = fast_two_sum(acc.hi, acc.lo);
            }
        }
        const dd sv = unbias(acc);
        float4* tot = ws_ptr<float4>(p.ws, p.L.rtot) + (size_t)s * cpr;
        float4* sub = ws_ptr<float4>(p.ws, p.L.rsub) + (size_t)s * cpr * kSubs;
        sub[(size_t)chunk * kSubs + lane] = pack_part(sv, 0);
        const dd total = warp_sum_dd(sv);
        if (lane == 0) tot[chunk] = pack_part(total, 0);
        if (arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_seq3) + s, (unsigned)cpr, lane))
            sd_residual_epilogue<DT>(p, P, c, s, trp, drp, lane);
    }
}

// Chunk and lane-block records of the residual max(0, p - q) of a sequence from the final-token
// pass's sums (see final_consumer): for a chunk, (A 2^n_t a - B 2^n_d b) with a = 1/Z_t in units
// of 2^-N_t and b = 1/Z_d in units of 2^-N_d, clamped at 0 (a position whose difference lies
// within rounding of theta can leave a tiny negative amount), as absolute values (exponent 0).
struct ResidualParts {
    const float4* tot_t;  // S_t chunk totals (with n_t), then S_d's at + cpr
    const float4* sub_t;  // {S_t, A} lane blocks; {S_d, B} at + cpr * kSubs
    const float4* ab;     // {A, B} chunk totals
    int cpr, Nt, Nd;
    dd a, b;
    __device__ __forceinline__ dd value(float ahi, float alo, float bhi, float blo, int c) const {
        const int nt = __float_as_int(ld_cg4(tot_t + c).z), nd = __float_as_int(ld_cg4(tot_t + cpr + c).z);
        dd x{0.0f, 0.0f}, y{0.0f, 0.0f};
        if (nt != kNoMass && ahi > 0.0f) {
            const float sc = pow2i(nt - Nt);
            x = dd_mul(dd{f_mul(ahi, sc), f_mul(alo, sc)}, a);
        }
        if (nd != kNoMass && bhi > 0.0f) {
            const float sc = pow2i(nd - Nd);
            y = dd_mul(dd{f_mul(bhi, sc), f_mul(blo, sc)}, b);
        }
        const dd r = dd_sub(x, y);
        return r.hi > 0.0f ? r : dd{0.0f, 0.0f};
    }
    __device__ __forceinline__ float4 chunk(int c) const {
        const float4 v = ld_cg4(ab + c);
        return pack_part(value(v.x, v.y, v.z, v.w, c), 0);
    }
    __device__ __forceinline__ float4 block(int c, int l) const {
        const float4 t = ld_cg4(sub_t + (size_t)c * kSubs + l);
        const float4 d = ld_cg4(sub_t + (size_t)(cpr + c) * kSubs + l);
        return pack_part(value(t.z, t.w, d.z, d.w, c), 0);
    }
};

// The target row's own partials from the same records (the zero-mass fallback: a draw from p).
struct TargetParts {
    const float4* tot_t;
    const float4* sub_t;
    __device__ __forceinline__ float4 chunk(int c) const { return ld_cg4(tot_t + c); }
    __device__ __forceinline__ float4 block(int c, int l) const {
        const float4 v = ld_cg4(sub_t + (size_t)c * kSubs + l);
        return make_float4(v.x, v.y, ld_cg4(tot_t + c).z, 0.0f);
    }
};

// The final token of each sequence after the merged final-token pass, one warp per sequence (a
// programmatic dependent of the pass): the bonus draw from p at the last target row, or the
// correction draw from normalise(max(0, p - q)) at the rejected position, whose normalisers and
// residual masses come from the pass's sums; a residual without mass falls back to p.
template <int DT>
__global__ void __launch_bounds__(kWarp) sd_final_finish_kernel(const __grid_constant__ SampleParams p) {
    __shared__ Exp2Table sT;
    load_exp2_table_s(p.T, sT);
    const PreciseCtx P{p.sc, &sT, nullptr, p.ws, p.direct};
    const int lane = threadIdx.x & 31;
    const int s = (int)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    griddep_wait();
    if (s >= p.R.S || seq_len(p.R, s, p.ws) < 0) return;
    const int cpr = p.cpr;
    const SeqState* st = ws_ptr<SeqState>(p.ws, p.L.seq) + s;
    const int mode = __ldcg(&st->mode);
    const float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
    const float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kSubs;
    const void* trp = row_ptr<DT>(p.R.tgt, __ldcg(&st->trow), p.R.V);
    const float u = __ldg(p.uniforms + (size_t)s * (p.R.K + 1) + p.R.K);
    int tok;
    if (mode == 0) {
        tok = draw_precise_row<DT>(tot_t, sub_t, cpr, trp, p.R.V, P, u, lane, nullptr);
    } else {
        const void* drp = row_ptr<DT>(p.R.drf, __ldcg(&st->drow), p.R.V);
        // both rows' common exponents and totals from one read of their chunk totals
        int Nt = kNoMass, Nd = kNoMass;
        dd Zt{0.0f, 0.0f}, Zd{0.0f, 0.0f};
        if (cpr <= kDrawCache * kWarp) {
            float4 vt[kDrawCache], vd[kDrawCache];
#pragma unroll
            for (int q = 0; q < kDrawCache; ++q) {
                const int ch = lane + q * kWarp;
                vt[q] = ch < cpr ? ld_cg4(tot_t + ch) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                vd[q] = ch < cpr ? ld_cg4(tot_t + cpr + ch) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (vt[q].x > 0.0f) Nt = max(Nt, __float_as_int(vt[q].z));
                if (vd[q].x > 0.0f) Nd = max(Nd, __float_as_int(vd[q].z));
            }
            Nt = warp_max_i(Nt);
            Nd = warp_max_i(Nd);
#pragma unroll
            for (int q = 0; q < kDrawCache; ++q) {
                Zt = dd_add(Zt, part_value(vt[q], Nt));
                Zd = dd_add(Zd, part_value(vd[q], Nd));
            }
            Zt = warp_sum_dd(Zt);
            Zd = warp_sum_dd(Zd);
        } else {
            Nt = row_exponent(tot_t, cpr, lane);
            Nd = row_exponent(tot_t + cpr, cpr, lane);
            Zt = row_total(tot_t, cpr, Nt, lane);
            Zd = row_total(tot_t + cpr, cpr, Nd, lane);
        }
        if (Nt == kNoMass || Nd == kNoMass || !(Zt.hi > 0.0f) || !(Zd.hi > 0.0f)) {
            if (lane == 0) raise_error(p.ws, kErrNonfinite);
            if (lane == 0) p.out_token[s] = 0;
            return;
        }
        ResidualCtx c;
        c.n_t = Nt;
        c.n_d = Nd;
        c.inv_t = dd_recip(Zt);
        c.inv_d = dd_recip(Zd);
        c.direct = false;  // (no shared-memory table here: the general weights)
        c.a_t = c.a_d = dd{0.0f, 0.0f};
        const ResidualParts rp{tot_t, sub_t, ws_ptr<float4>(p.ws, p.L.rtot) + (size_t)s * cpr, cpr,
                               Nt, Nd, c.inv_t, c.inv_d};
        ResidualBlock<DT> fn{trp, drp, p.R.V, c, P};
        tok = draw_inverse_cdf_parts<ResidualBlock<DT>::PL>(rp, cpr, Geo<DT>::kChunk, Geo<DT>::kSub,
                                                            u, lane, fn, nullptr);
        if (tok < 0) {  // the residual has no mass (only through rounding): a draw from p
            PreciseBlock<DT> fn{trp, p.R.V, P};
            tok = draw_inverse_cdf_parts<PreciseBlock<DT>::PL>(TargetParts{tot_t, sub_t}, cpr,
                                                               Geo<DT>::kChunk, Geo<DT>::kSub, u,
                                                               lane, fn, nullptr);
        }
    }
    if (lane == 0) {
        if (tok < 0) raise_error(p.ws, kErrNonfinite);
        p.out_token[s] = tok < 0 ? 0 : tok;
    }
}

template <typename Kern>
static int grid_for(Kern kern, long long warps_needed, size_t smem) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSampleThreads, smem) != cudaSuccess)
        occ = 1;
    const int wpb = kSampleThreads / kWarp;
    const long long want = (warps_needed + wpb - 1) / wpb;
    const long long cap = (long long)device_sm_count() * (occ > 0 ? occ : 1);
    const long long g = want < cap ? want : cap;
    return (int)(g < 1 ? 1 : g);
}

// One warp per sequence, one sequence per block (the draws are long dependent chains: each gets
// an SM's issue slots to itself), launched as a programmatic dependent of the stream before.
static cudaError_t launch_warp_per_block(const void* kern, const SampleParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.R.S);
    cfg.blockDim = dim3(kWarp);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    SampleParams q = p;
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int DT>
static cudaError_t launch_sd_sample_t(const SampleParams& p, cudaStream_t st) {
    const size_t smem = (DT == 1 && p.use_table) ? (size_t)kTabSize * sizeof(float2) : 0;
    auto k2 = sd_rows_kernel<DT>;
    auto k3 = sd_residual_kernel<DT>;
    cudaError_t e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (p.vec) {
        // aligned rows: one final-token pass over the (target, draft) row pairs as the pipelined
        // stream, then the per-sequence draws as a programmatic dependent
        StreamParams sp{};
        sp.R = p.R;
        sp.dtype = DT;
        sp.vec = true;
        sp.sc_t = sp.sc_d = p.sc;
        sp.use_table = p.use_table;
        sp.direct = p.direct;
        sp.T = p.T;
        sp.ws = p.ws;
        sp.L = p.L;
        sp.cpr = p.cpr;
        sp.slots = 2 * p.R.K + 1;
        sp.div_cpr = make_fastdiv((uint32_t)p.cpr);
        sp.mode = kModeSDFinal;
        e = launch_stream_tma(sp, st);
        if (e == cudaSuccess) e = launch_warp_per_block(reinterpret_cast<const void*>(sd_final_finish_kernel<DT>), p, st);
        return e;
    }
    k2<<<grid_for(k2, (long long)p.R.S * 2 * p.cpr, smem), kSampleThreads, smem, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k3<<<grid_for(k3, (long long)p.R.S * p.cpr, smem), kSampleThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sd_sample(const SampleParams& p, cudaStream_t st) {
    return p.dtype == 0 ? launch_sd_sample_t<0>(p, st) : launch_sd_sample_t<1>(p, st);
}

}  // namespace smcsd
