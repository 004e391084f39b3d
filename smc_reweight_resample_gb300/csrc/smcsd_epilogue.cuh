// smcsd_epilogue.cuh -- per-sequence and per-group epilogues of the streaming pass, run by the
// last warp to finish a sequence's chunks (or a group's particles):
//   SD    ("Faster LLM Inference via Sequential Monte Carlo", sec. 1): row normalisers, the
//         ratio tests min(1, p/q) in position order, the acceptance length, and the hand-off of
//         the row (pair) to draw the final token from;
//   SMC   (same page, sec. 2 steps 3-4 and sec. 3): row normalisers, the log-weight update
//         sum_k log pi_k(x_k) - log q_k(x_k), the (K+1)-th token drawn from pi at row K;
//   step  additionally, per group of N particles (last particle of the group): effective
//         sample size, systematic resampling and the page-table remap with refcounts.
#pragma once

#include "smcsd_launch.cuh"

namespace smcsd {

__device__ __forceinline__ void load_exp2_table(const Exp2Table& src, Exp2Table& dst) {
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
__device__ __noinline__ void sd_seq_epilogue(const StreamParams& p, int s, int ks, int lane) {
    const Rows& R = p.R;
    const int cpr = p.cpr;
    const float2* fast = ws_ptr<float2>(p.ws, p.L.fast) + (size_t)s * p.slots * cpr;
    const float* u = p.uniforms + (size_t)s * (R.K + 1);
    int acc = ks;
    for (int k0 = 0; k0 < ks; k0 += 4) {
        const int nk = min(4, ks - k0);
        const double lt = rows_lse_fast4(fast + (size_t)(2 * k0) * cpr, 2 * cpr, nk, cpr, p.sc_t, lane);
        const double ld = rows_lse_fast4(fast + (size_t)(2 * k0 + 1) * cpr, 2 * cpr, nk, cpr, p.sc_d, lane);
        bool rej = false;
        if (lane < nk) {
            const int k = k0 + lane;
            if (!(lt == lt) || !(ld == ld)) raise_error(p.ws, kErrNonfinite);  // a row without mass
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
    const double Lb = rows_lse_fast4(fast + (size_t)(2 * ks) * cpr, cpr, 1, cpr, p.sc_t, lane);
    if (lane == 0) {
        if (!(Lb == Lb)) raise_error(p.ws, kErrNonfinite);
        if (p.lse_tgt) p.lse_tgt[trow_of(R, s, ks)] = (float)Lb;
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
__device__ __noinline__ void smc_particle_epilogue(const StreamParams& p, const PreciseCtx& P,
                                                   int s, int lane) {
    const Rows& R = p.R;
    const int K = R.K, cpr = p.cpr;
    const float2* fast = ws_ptr<float2>(p.ws, p.L.fast) + (size_t)s * p.slots * cpr;
    double inc = 0.0;
    for (int k0 = 0; k0 < K; k0 += 4) {
        const int nk = min(4, K - k0);
        const double lt = rows_lse_fast4(fast + (size_t)(2 * k0) * cpr, 2 * cpr, nk, cpr, p.sc_t, lane);
        const double ld = rows_lse_fast4(fast + (size_t)(2 * k0 + 1) * cpr, 2 * cpr, nk, cpr, p.sc_d, lane);
        double ell = 0.0;
        if (lane < nk) {
            const int k = k0 + lane;
            if (!(lt == lt) || !(ld == ld)) raise_error(p.ws, kErrNonfinite);  // a row without mass
            bool ok;
            ell = log_ratio<DT>(p, s, k, lt, ld, ok);
            if (p.lse_tgt) p.lse_tgt[trow_of(R, s, k)] = (float)lt;
            if (p.lse_drf) p.lse_drf[drow_of(R, s, k)] = (float)ld;
        }
        inc += warp_sum_d(ell);
    }
    // the (K+1)-th token from pi at target row K
    const float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * cpr;
    const float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * cpr * kSubs;
    const long long rowK = trow_of(R, s, K);
    double lseK = 0.0;
    const int tok = draw_precise_row<DT>(tot, sub, cpr, row_ptr<DT>(R.tgt, rowK, R.V), R.V, P,
                                         __ldg(p.uniforms + s), lane, &lseK);
    if (lane == 0) {
        p.logw[s] = (float)((double)__ldcg(p.logw + s) + inc);
        if (tok < 0) raise_error(p.ws, kErrNonfinite);
        p.bonus_token[s] = tok < 0 ? 0 : tok;
        if (p.lse_tgt) p.lse_tgt[rowK] = (float)lseK;
    }
}

// SMC step: ESS, systematic resampling and page-table remap of group g.
static __device__ __noinline__ void smc_group_epilogue(const StreamParams& p, int g, int lane) {
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

// What chunk `it` of the sequence-major order is.
struct ChunkRef {
    int s, slot, chunk, ks;
    bool valid, is_draft;
    long long row;
};
__device__ __forceinline__ ChunkRef chunk_ref(const StreamParams& p, uint32_t it) {
    ChunkRef c;
    c.s = (int)fast_div(it, p.div_seq);
    const uint32_t rem = it - (uint32_t)c.s * p.div_seq.d;
    c.slot = (int)fast_div(rem, p.div_cpr);
    c.chunk = (int)(rem - (uint32_t)c.slot * p.div_cpr.d);
    c.ks = seq_len(p.R, c.s, p.ws);
    c.valid = c.ks >= 0 && c.slot <= 2 * c.ks;
    c.is_draft = c.slot < 2 * c.ks && (c.slot & 1);
    const int k = c.slot >> 1;
    c.row = c.valid ? (c.is_draft ? drow_of(p.R, c.s, k) : trow_of(p.R, c.s, k)) : 0;
    return c;
}

// The end of one chunk: count it for its sequence; the last chunk's warp runs the sequence
// epilogue and, in the fused step, the group's.
template <int DT, int MODE>
__device__ __forceinline__ void finish_chunk(const StreamParams& p, const PreciseCtx& P, int s,
                                             int ks, int lane) {
    const unsigned expected = (unsigned)(2 * ks + 1) * (unsigned)p.cpr;
    if (!arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_seq1) + s, expected, lane)) return;
    if (MODE == kModeSD) {
        sd_seq_epilogue<DT>(p, s, ks, lane);
    } else {
        smc_particle_epilogue<DT>(p, P, s, lane);
        if (MODE == kModeSMCStep) {
            const int g = s / p.N;
            if (arrive_last(ws_ptr<unsigned>(p.ws, p.L.cnt_group) + g, (unsigned)p.N, lane))
                smc_group_epilogue(p, g, lane);
        }
    }
}

}  // namespace smcsd
