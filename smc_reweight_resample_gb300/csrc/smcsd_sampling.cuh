// smcsd_sampling.cuh -- per-chunk partials, row normalisers, the inverse-CDF draw over a row,
// and per-group effective sample size with systematic resampling. Warp-level device code
// shared by the kernels.
#pragma once

#include "smcsd_internal.cuh"

namespace smcsd {

__device__ __forceinline__ float hw_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------------------------------
// chunk partials
// ------------------------------------------------------------------------------------------

// Fast partial of one chunk: {m, sum exp(c (z - m))} with m the chunk's largest logit (raw,
// before scaling; c > 0 keeps the order). An all-masked chunk gives {-inf, 0}.
template <int DT>
__device__ __forceinline__ float2 fast_partial(const ChunkRegs<DT>& r, float c2, void* ws) {
    constexpr int PV = Geo<DT>::kPerVec;
    float m = kNegInf;
#pragma unroll
    for (int v = 0; v < kLoads; ++v)
#pragma unroll
        for (int q = 0; q < PV; ++q) m = fmaxf(m, r.x[v][q]);
    m = warp_max(m);
    if (m == kNegInf) {
        bool nan = false;
#pragma unroll
        for (int v = 0; v < kLoads; ++v)
#pragma unroll
            for (int q = 0; q < PV; ++q) nan |= (r.x[v][q] != r.x[v][q]);
        if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0) raise_error(ws, kErrNonfinite);
        return make_float2(kNegInf, 0.0f);
    }
    float acc[kLoads];
#pragma unroll
    for (int v = 0; v < kLoads; ++v) {
        float a = 0.0f;
#pragma unroll
        for (int q = 0; q < PV; ++q) a += hw_exp2((r.x[v][q] - m) * c2);
        acc[v] = a;
    }
    float s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    s = warp_sum(s);
    if (!(s == s) || m == -kNegInf) {  // NaN or +inf in the chunk
        if ((threadIdx.x & 31) == 0) raise_error(ws, kErrNonfinite);
    }
    return make_float2(m, s);
}

// Precise partials of one chunk of a row that will be sampled: eight double-float sums
// sum_i exp(c z_i) / 2^nref over the 512-byte slices, and their total. Lane v < 8 stores slice
// v, lane 0 the total.
template <int DT>
__device__ __forceinline__ void precise_partials(const ChunkRegs<DT>& r, const Scale& sc,
                                                 const Exp2Table& T, void* ws, int lane,
                                                 float4* tot_out, float4* sub_out) {
    constexpr int PV = Geo<DT>::kPerVec;
    float m = kNegInf;
#pragma unroll
    for (int v = 0; v < kLoads; ++v)
#pragma unroll
        for (int q = 0; q < PV; ++q) m = fmaxf(m, r.x[v][q]);
    m = warp_max(m);
    ddx em;
    bool any = m > kNegInf && precise_exp(m, sc, T, ws, em);
    if (!any) {
        bool nan = false;
#pragma unroll
        for (int v = 0; v < kLoads; ++v)
#pragma unroll
            for (int q = 0; q < PV; ++q) nan |= (r.x[v][q] != r.x[v][q]);
        if (__any_sync(0xffffffffu, nan) && lane == 0) raise_error(ws, kErrNonfinite);
        if (lane < kLoads) sub_out[lane] = pack_part(dd{0.0f, 0.0f}, kNoMass);
        if (lane == 0) *tot_out = pack_part(dd{0.0f, 0.0f}, kNoMass);
        return;
    }
    const int nref = em.n;
    float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
    dd total{0.0f, 0.0f};
#pragma unroll
    for (int v = 0; v < kLoads; ++v) {
        dd acc{kBias, 0.0f};
#pragma unroll
        for (int q = 0; q < PV; ++q) {
            ddx e;
            if (precise_exp(r.x[v][q], sc, T, ws, e)) acc_biased(acc, scaled(e, nref));
        }
        dd sv = warp_sum_dd(unbias(acc));
        total = dd_add(total, sv);
        if (lane == v) mine = pack_part(sv, nref);
    }
    if (lane < kLoads) sub_out[lane] = mine;
    if (lane == 0) *tot_out = pack_part(total, nref);
}

// ------------------------------------------------------------------------------------------
// row normalisers from fast partials
// ------------------------------------------------------------------------------------------

// Natural-log normalisers log sum_i exp(c z_i) of up to four rows whose fast partials start at
// part[r * stride] (cpr chunks each), written to out[r] (r < nrows) on every lane. The four
// rows' partial loads are in flight together. A row without mass gives NaN.
__device__ __forceinline__ void rows_lse_fast4(const float2* part, int stride, int nrows, int cpr,
                                               const Scale& sc, int lane, double (&out)[4]) {
    constexpr int RB = 4;
    float m[RB], s[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        m[b] = kNegInf;
        s[b] = 0.0f;
    }
    for (int c0 = 0; c0 < cpr; c0 += 4 * kWarp) {
        float2 v[RB][4];
#pragma unroll
        for (int b = 0; b < RB; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int c = c0 + lane + j * kWarp;
                v[b][j] = (b < nrows && c < cpr) ? ld_cg2(part + (size_t)b * stride + c)
                                                 : make_float2(kNegInf, 0.0f);
            }
#pragma unroll
        for (int b = 0; b < RB; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float pm = v[b][j].x, ps = v[b][j].y;
                if (pm == kNegInf) continue;
                if (pm > m[b]) {
                    s[b] = s[b] * hw_exp2((m[b] - pm) * sc.c2) + ps;
                    m[b] = pm;
                } else {
                    s[b] += ps * hw_exp2((pm - m[b]) * sc.c2);
                }
            }
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        float M = warp_max(m[b]);
        float t = (m[b] == kNegInf) ? 0.0f : s[b] * hw_exp2((m[b] - M) * sc.c2);
        float S = warp_sum(t);
        out[b] = (M == kNegInf || !(S > 0.0f)) ? __longlong_as_double(0x7ff8000000000000ll)
                                               : sc.c * (double)M + log((double)S);
    }
}

__device__ __forceinline__ double pick4(const double (&a)[4], int i) {
    return i == 0 ? a[0] : (i == 1 ? a[1] : (i == 2 ? a[2] : a[3]));
}

// ------------------------------------------------------------------------------------------
// inverse-CDF draw over a row described by precise partials
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ dd part_value(float4 p, int N) {
    int n = __float_as_int(p.z);
    if (n == kNoMass || !(p.x > 0.0f)) return dd{0.0f, 0.0f};
    float s = pow2i(n - N);
    return dd{f_mul(p.x, s), f_mul(p.y, s)};
}

// Draw token = min{ i : sum_{j<=i} w_j > u * sum_j w_j } over a row whose chunk totals `tot`
// [cpr] and slice partials `sub` [cpr * 8] were produced by precise_partials (or by the
// residual pass), rescanning one slice with `slice_weights(chunk, sub, lane, w[PV])`, which
// must reproduce the per-logit weights in units of 2^N exactly. Returns the token on every
// lane (-1 if the row has no mass). If `lse` is given it receives log(sum_j w_j) + N ln 2.
template <int PV, typename SliceFn>
__device__ int draw_inverse_cdf(const float4* tot, const float4* sub, int cpr, int chunk_elems,
                                int sub_elems, float u, int lane, SliceFn slice_weights,
                                double* lse) {
    // common exponent
    int N = kNoMass;
    for (int c = lane; c < cpr; c += kWarp) {
        float4 t = ld_cg4(tot + c);
        if (t.x > 0.0f) N = max(N, __float_as_int(t.z));
    }
    N = warp_max_i(N);
    if (N == kNoMass) return -1;

    // chunk level: lane l owns the contiguous chunks [l*cpl, l*cpl + cpl)
    const int cpl = (cpr + kWarp - 1) / kWarp;
    const int c_begin = min(lane * cpl, cpr), c_end = min(c_begin + cpl, cpr);
    dd loc{0.0f, 0.0f};
    for (int c = c_begin; c < c_end; ++c) loc = dd_add(loc, part_value(ld_cg4(tot + c), N));
    dd excl = warp_exclusive_scan_dd(loc, lane);
    dd incl = dd_add(excl, loc);
    dd R{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    if (lse) *lse = log(dd_to_double(R)) + (double)N * 0.69314718055994530942;
    const dd target = dd_mul_f(R, u);

    bool has = loc.hi > 0.0f && dd_gt(incl, target);
    unsigned bal = __ballot_sync(0xffffffffu, has);
    int owner;
    if (bal) {
        owner = __ffs(bal) - 1;
    } else {  // rounding put the target at or past the total: last lane with mass
        unsigned m = __ballot_sync(0xffffffffu, loc.hi > 0.0f);
        owner = 31 - __clz(m);
    }
    int c_star = -1;
    dd base{0.0f, 0.0f};
    if (lane == owner) {
        dd p = excl;
        int last_pos = -1;
        dd last_base = p;
        for (int c = c_begin; c < c_end; ++c) {
            dd v = part_value(ld_cg4(tot + c), N);
            if (v.hi > 0.0f) {
                last_pos = c;
                last_base = p;
                dd q = dd_add(p, v);
                if (dd_gt(q, target)) {
                    c_star = c;
                    base = p;
                    break;
                }
                p = q;
            }
        }
        if (c_star < 0) {
            c_star = last_pos;
            base = last_base;
        }
    }
    c_star = __shfl_sync(0xffffffffu, c_star, owner);
    base.hi = __shfl_sync(0xffffffffu, base.hi, owner);
    base.lo = __shfl_sync(0xffffffffu, base.lo, owner);

    // slice level
    dd sv = lane < kLoads ? part_value(ld_cg4(sub + (size_t)c_star * kLoads + lane), N) : dd{0.0f, 0.0f};
    dd sex = warp_exclusive_scan_dd(sv, lane);
    dd sin_ = dd_add(dd_add(base, sex), sv);
    has = sv.hi > 0.0f && dd_gt(sin_, target);
    bal = __ballot_sync(0xffffffffu, has);
    int s_star;
    if (bal) {
        s_star = __ffs(bal) - 1;
    } else {
        unsigned m = __ballot_sync(0xffffffffu, sv.hi > 0.0f);
        s_star = m ? 31 - __clz(m) : 0;
    }
    dd sbase = dd_add(base, sex);
    sbase.hi = __shfl_sync(0xffffffffu, sbase.hi, s_star);
    sbase.lo = __shfl_sync(0xffffffffu, sbase.lo, s_star);

    // logit level: rescan the slice
    dd w[PV];
    slice_weights(c_star, s_star, lane, w);
    dd lsum{0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < PV; ++q) lsum = dd_add(lsum, w[q]);
    dd lex = warp_exclusive_scan_dd(lsum, lane);
    dd p = dd_add(sbase, lex);
    int found = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < PV; ++q) {
        if (w[q].hi > 0.0f) {
            p = dd_add(p, w[q]);
            lastpos = q;
            if (found < 0 && dd_gt(p, target)) found = q;
        }
    }
    bal = __ballot_sync(0xffffffffu, found >= 0);
    int tok_lane, tok_q;
    if (bal) {
        tok_lane = __ffs(bal) - 1;
        tok_q = __shfl_sync(0xffffffffu, found, tok_lane);
    } else {
        unsigned m = __ballot_sync(0xffffffffu, lastpos >= 0);
        if (!m) return -1;
        tok_lane = 31 - __clz(m);
        tok_q = __shfl_sync(0xffffffffu, lastpos, tok_lane);
    }
    return c_star * chunk_elems + s_star * sub_elems + tok_lane * PV + tok_q;
}

// Weights exp(c z) / 2^N of one slice of a row (the rescan for draws from a precise row).
template <int DT>
struct PreciseSlice {
    const void* row;
    int V;
    bool vec;
    int N;
    Scale sc;
    const Exp2Table* T;
    void* ws;
    __device__ __forceinline__ void operator()(int chunk, int sub, int lane,
                                               dd (&w)[Geo<DT>::kPerVec]) const {
        float x[Geo<DT>::kPerVec];
        if (vec)
            load_slice<DT, true>(row, V, chunk, sub, lane, x);
        else
            load_slice<DT, false>(row, V, chunk, sub, lane, x);
#pragma unroll
        for (int q = 0; q < Geo<DT>::kPerVec; ++q) {
            ddx e;
            w[q] = precise_exp(x[q], sc, *T, ws, e) ? scaled(e, N) : dd{0.0f, 0.0f};
        }
    }
};

// The common exponent N of a precise row (max over its chunk totals), on every lane.
__device__ __forceinline__ int row_exponent(const float4* tot, int cpr, int lane) {
    int N = kNoMass;
    for (int c = lane; c < cpr; c += kWarp) {
        float4 t = ld_cg4(tot + c);
        if (t.x > 0.0f) N = max(N, __float_as_int(t.z));
    }
    return warp_max_i(N);
}

// Sum of a precise row in units of 2^N (double-float), on every lane.
__device__ __forceinline__ dd row_total(const float4* tot, int cpr, int N, int lane) {
    dd loc{0.0f, 0.0f};
    for (int c = lane; c < cpr; c += kWarp) loc = dd_add(loc, part_value(ld_cg4(tot + c), N));
    return warp_sum_dd(loc);
}

template <int DT>
__device__ __forceinline__ int draw_precise_row(const float4* tot, const float4* sub, int cpr,
                                                const void* row, int V, bool vec, const Scale& sc,
                                                const Exp2Table& T, float u, void* ws, int lane,
                                                double* lse) {
    PreciseSlice<DT> fn{row, V, vec, row_exponent(tot, cpr, lane), sc, &T, ws};
    return draw_inverse_cdf<Geo<DT>::kPerVec>(tot, sub, cpr, Geo<DT>::kChunk, Geo<DT>::kSub, u,
                                              lane, fn, lse);
}

// ------------------------------------------------------------------------------------------
// effective sample size and systematic resampling of one group (one warp)
// ------------------------------------------------------------------------------------------

// Number of children j in [0, N) with (j + U) / N < C, with the comparison evaluated exactly as
// written (double), so that it agrees with the definition a_j = min{ i : C_i > v_j }.
__device__ __forceinline__ int children_below(double C, double U, int N) {
    double est = floor(C * (double)N - U);
    long long j = (long long)est;
    if (j < -1) j = -1;
    if (j > N - 1) j = N - 1;
    while (j + 1 <= N - 1 && (((double)(j + 1) + U) / (double)N) < C) ++j;
    while (j >= 0 && !((((double)j + U) / (double)N) < C)) --j;
    return (int)(j + 1);
}

// logw [N] of one group (float, in/out). Writes ancestors [N], *ess_out, *res_out (if given).
// Returns whether the group was resampled (on every lane).
__device__ __forceinline__ bool group_resample(float* logw, int N, float thr, float U,
                                               int32_t* anc, float* ess_out, int32_t* res_out,
                                               void* ws, int lane) {
    double M = -__builtin_huge_val();
    bool bad = false;
    for (int i = lane; i < N; i += kWarp) {
        float v = __ldcg(logw + i);
        if (v != v || v == -kNegInf) bad = true;
        M = fmax(M, (double)v);
    }
    M = warp_max_d(M);
    bad = __any_sync(0xffffffffu, bad) || M == -__builtin_huge_val();
    if (bad) {
        if (lane == 0) raise_error(ws, kErrNonfinite);
        for (int j = lane; j < N; j += kWarp) anc[j] = j;
        if (lane == 0 && res_out) *res_out = 0;
        return false;
    }
    double W = 0.0, W2 = 0.0;
    for (int i = lane; i < N; i += kWarp) {
        double w = exp((double)__ldcg(logw + i) - M);
        W += w;
        W2 += w * w;
    }
    W = warp_sum_d(W);
    W2 = warp_sum_d(W2);
    const double ess = W * W / W2;
    const bool res = ess < (double)thr;
    if (lane == 0) {
        if (ess_out) *ess_out = (float)ess;
        if (res_out) *res_out = res ? 1 : 0;
    }
    if (!res) {
        for (int j = lane; j < N; j += kWarp) anc[j] = j;
        return false;
    }
    // CDF over contiguous blocks of particles per lane; children of particle i are the j with
    // C_{i-1} <= v_j < C_i, i.e. j in [J(C_{i-1}), J(C_i)).
    const int per = (N + kWarp - 1) / kWarp;
    const int i0 = min(lane * per, N), i1 = min(i0 + per, N);
    double loc = 0.0;
    for (int i = i0; i < i1; ++i) loc += exp((double)__ldcg(logw + i) - M);
    double run = warp_exclusive_scan_d(loc, lane);
    const double Ud = (double)U;
    int Jlast = 0;
    // J at the end of each lane's block, then the previous lane's value as this lane's start
    {
        double r = run;
        int J = 0;
        for (int i = i0; i < i1; ++i) {
            r += exp((double)__ldcg(logw + i) - M);
            double C = (i == N - 1) ? 1.0 : r / W;
            J = children_below(C, Ud, N);
        }
        Jlast = (i1 > i0) ? J : -1;
    }
    // propagate: a lane with an empty block passes its predecessor's value on
    int Jend = Jlast;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, Jend, o);
        if (lane >= o && Jend < 0) Jend = t;
    }
    int Jstart = __shfl_up_sync(0xffffffffu, Jend, 1);
    if (lane == 0 || Jstart < 0) Jstart = 0;
    double r = run;
    int Jprev = Jstart;
    for (int i = i0; i < i1; ++i) {
        r += exp((double)__ldcg(logw + i) - M);
        double C = (i == N - 1) ? 1.0 : r / W;
        int J = children_below(C, Ud, N);
        for (int j = Jprev; j < J; ++j) anc[j] = i;
        Jprev = max(Jprev, J);
    }
    __syncwarp();
    for (int i = lane; i < N; i += kWarp) logw[i] = 0.0f;
    return true;
}

}  // namespace smcsd
