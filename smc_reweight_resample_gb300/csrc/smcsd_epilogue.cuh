// smcsd_epilogue.cuh -- what the finishing passes (finish.cu) do with the streaming pass's chunk
// partials: one warp per row, then one warp per sequence, then, in the fused step, one block
// per group:
//   row   every row's normaliser log sum_i exp(c z_i); for the bonus row of a particle, the
//         (K+1)-th token drawn from pi at row K;
//   SD    ("Faster LLM Inference via Sequential Monte Carlo", sec. 1): the ratio tests
//         min(1, p/q) in position order, the acceptance length, and the hand-off of the row
//         (pair) to draw the final token from;
//   SMC   (same page, sec. 2 steps 3-4 and sec. 3): the log-weight update
//         sum_k log pi_k(x_k) - log q_k(x_k), or for the whole-sequence power target
//         sum_k alpha log p_k(x_k) - log q_k(x_k) + (alpha - 1) log p_K(b), plus an optional
//         additive log-reward (sec. 3 "flexibility", sec. 5);
//   step  additionally, per group of N particles: effective sample size, systematic
//         resampling and the page-table remap with refcounts.
#pragma once

#include <type_traits>

#include "smcsd_launch.cuh"

namespace smcsd {

__device__ __forceinline__ void load_exp2_table(const Exp2Table& src, Exp2Table& dst) {
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        dst.hi[i] = src.hi[i];
        dst.lo[i] = src.lo[i];
    }
    __syncthreads();
}

// The (K+1)-th token of particle s, drawn by inverse CDF from pi at target row ks with the row's
// precise partials (warp-wide; stores the token, the row's normaliser and the log-probability of
// the token where asked). Returns, on lane 0, the token's weight factor under the whole-sequence
// power target ((alpha - 1) log p(b) as a double-float; zero otherwise).
template <int DT>
__device__ __forceinline__ float2 bonus_draw(const StreamParams& p, const PreciseCtx& P, int s, int ks,
                                             int lane) {
    const Rows& R = p.R;
    const float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + (size_t)(s * 2) * p.cpr;
    const float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + (size_t)(s * 2) * p.cpr * kSubs;
    const long long row = trow_of(R, s, ks);
    float lse = 0.0f;
    const int tok = draw_precise_row<DT>(tot, sub, p.cpr, row_ptr<DT>(R.tgt, row, R.V), R.V, P,
                                         __ldg(p.uniforms + s), lane, &lse);
    float2 fac = make_float2(0.0f, 0.0f);
    if (lane == 0) {
        if (tok < 0) raise_error(p.ws, kErrNonfinite);
        p.bonus_token[s] = tok < 0 ? 0 : tok;
        if (p.lse_tgt) p.lse_tgt[row] = lse;
        if (p.target_seq || p.bonus_logq) {
            // log-probability of the drawn token, c z_tok - lse
            dd lp{0.0f, 0.0f};
            if (tok >= 0) {
                const float z = logit_at<DT>(row_ptr<DT>(R.tgt, row, R.V), tok);
                lp = dd_sub(dd_mul_f(dd{p.sc_t.c_hi, p.sc_t.c_lo}, z), dd{lse, 0.0f});
            }
            if (p.bonus_logq) p.bonus_logq[s] = f_add(lp.hi, lp.lo);
            if (p.target_seq && p.alpha != 1.0f) {
                // whole-sequence power target: the (K+1)-th token, drawn from p, carries the
                // weight factor p^(alpha-1), i.e. (alpha - 1) lp in log space
                const dd inc = dd_mul(lp, two_sum(p.alpha, -1.0f));  // exact alpha - 1
                fac = make_float2(inc.hi, inc.lo);
            }
        }
    }
    return fac;
}

// One row: the row's normaliser (into sL[slot], and the optional lse outputs), or, for the bonus
// row of a particle, the (K+1)-th token drawn from pi with the row's normaliser as a by-product.
template <int DT, int MODE>
__device__ __noinline__ void row_epilogue(const StreamParams& p, const PreciseCtx& P, int s, int slot,
                                          int ks, int lane, float2* sL) {
    const Rows& R = p.R;
    const int k = slot >> 1;
    if (MODE != kModeSD && slot == 2 * ks) {
        const float2 fac = bonus_draw<DT>(p, P, s, ks, lane);
        if (lane == 0 && p.target_seq) sL[slot] = fac;
        return;
    }
    const bool is_draft = slot < 2 * ks && (slot & 1);
    const size_t r = (size_t)s * p.slots + slot;
    const dd L = row_lse_fast(ws_ptr<float2>(p.ws, p.L.fast) + r * p.cpr, p.cpr,
                              is_draft ? p.sc_d : p.sc_t, lane);
    if (lane == 0) {
        if (!(L.hi == L.hi)) raise_error(p.ws, kErrNonfinite);  // a row without mass
        sL[slot] = make_float2(L.hi, L.lo);
        const float Lf = f_add(L.hi, L.lo);
        if (is_draft) {
            if (p.lse_drf) p.lse_drf[drow_of(R, s, k)] = Lf;
        } else if (p.lse_tgt) {
            p.lse_tgt[trow_of(R, s, k)] = Lf;
        }
    }
}

// Inputs of the sequence epilogue that do not depend on the streaming pass, read before waiting
// for it: the draft token of row `slot` (< 2ks) and the logit there, into sX[slot], sZ[slot].
template <int DT>
__device__ __forceinline__ void prefetch_token_logit(const StreamParams& p, int s, int slot, int* sX,
                                                     float* sZ) {
    const Rows& R = p.R;
    const int k = slot >> 1;
    const bool is_draft = slot & 1;
    const int x = __ldg(R.toks + drow_of(R, s, k));
    float z = 0.0f;
    if (is_draft && p.drf_logq)
        z = __ldg(p.drf_logq + drow_of(R, s, k));  // (draft slots then hold log q itself)
    else if (x >= 0 && x < R.V)
        z = is_draft ? logit_at<DT>(row_ptr<DT>(R.drf, drow_of(R, s, k), R.V), x)
                     : logit_at<DT>(row_ptr<DT>(R.tgt, trow_of(R, s, k), R.V), x);
    sX[slot] = x;
    sZ[slot] = z;
}

// log p_k(x_k) and log q_k(x_k) at position k, as double-floats, from the row normalisers sL and
// the draft token and logits there (sX, sZ) of this sequence's block. False (with an error raised)
// if the token is out of range.
__device__ __forceinline__ bool log_probs(const StreamParams& p, int k, const float2* sL, const int* sX,
                                          const float* sZ, dd& lt, dd& ld) {
    const int x = sX[2 * k];
    lt = ld = dd{0.0f, 0.0f};
    if (x < 0 || x >= p.R.V) {
        raise_error(p.ws, kErrRange);
        return false;
    }
    const float2 Lt = sL[2 * k];
    lt = dd_sub(dd_mul_f(dd{p.sc_t.c_hi, p.sc_t.c_lo}, sZ[2 * k]), dd{Lt.x, Lt.y});
    if (p.drf_logq) {
        ld = dd{sZ[2 * k + 1], 0.0f};  // the given log q_k(x_k)
    } else {
        const float2 Ld = sL[2 * k + 1];
        ld = dd_sub(dd_mul_f(dd{p.sc_d.c_hi, p.sc_d.c_lo}, sZ[2 * k + 1]), dd{Ld.x, Ld.y});
    }
    return true;
}

// log p_k(x_k) - log q_k(x_k) at position k (0 with an error raised if the token is out of range).
__device__ __forceinline__ bool log_ratio(const StreamParams& p, int k, const float2* sL, const int* sX,
                                          const float* sZ, dd& ell) {
    dd lt, ld;
    const bool ok = log_probs(p, k, sL, sX, sZ, lt, ld);
    ell = dd_sub(lt, ld);
    return ok;
}

// SD: the ratio tests min(1, p/q) in position order, the acceptance length and the hand-off of
// the row (pair) to draw the final token from. Position k is accepted iff u_k < exp(min(0, l_k)),
// with the exponential in double-float.
static __device__ __noinline__ void sd_seq_epilogue(const StreamParams& p, int s, int ks, int lane,
                                                    const float2* sL, const int* sX, const float* sZ,
                                                    const Exp2Table& T) {
    const Rows& R = p.R;
    const float* u = p.uniforms + (size_t)s * (R.K + 1);
    int acc = ks;
    for (int k0 = 0; k0 < ks; k0 += kWarp) {
        const int k = k0 + lane;
        bool rej = false;
        if (k < ks) {
            dd ell;
            const bool ok = log_ratio(p, k, sL, sX, sZ, ell);
            const float uk = __ldg(u + k);
            if (!ok || !(ell.hi == ell.hi)) {
                rej = true;
            } else if (ell.hi < 0.0f) {
                const ddx e = exp_split(ell, T);
                const float sc = pow2i(e.n);
                rej = !dd_gt(dd{f_mul(e.hi, sc), f_mul(e.lo, sc)}, dd{uk, 0.0f});
            }  // l_k >= 0: the ratio is at least 1 > u
        }
        const unsigned b = __ballot_sync(0xffffffffu, rej);
        if (b && acc == ks) acc = k0 + __ffs(b) - 1;
    }
    if (lane == 0) {
        p.accept_len[s] = acc;
        SeqState* st = ws_ptr<SeqState>(p.ws, p.L.seq) + s;
        st->mode = acc < ks ? 1 : 0;
        st->acc = acc;
        st->trow = trow_of(R, s, acc);
        st->drow = acc < ks ? drow_of(R, s, acc) : -1;
        // p_i > q_i iff c z_t,i - L_t > c z_d,i - L_d iff z_t,i - z_d,i > (L_t - L_d) / c
        if (acc < ks) {
            const float2 Lt = sL[2 * acc], Ld = sL[2 * acc + 1];
            const dd dl = dd_sub(dd{Lt.x, Lt.y}, dd{Ld.x, Ld.y});
            st->theta = f_div(f_add(dl.hi, dl.lo), p.sc_t.c_hi);
        }
    }
}

// SMC: log-weight update sum_k log pi_k(x_k) - log q_k(x_k) of particle s (double-float sums),
// from its old log-weight lw_old. With the whole-sequence power target the terms are
// alpha log p_k(x_k) - log q_k(x_k), plus the (K+1)-th token's factor that its row epilogue left
// in sL[2K]; a log-reward adds reward_scale * log_reward[s]. Returns the new log-weight on lane 0.
static __device__ __noinline__ float smc_particle_epilogue(const StreamParams& p, int s, int lane, float lw_old,
                                                          const float2* sL, const int* sX, const float* sZ) {
    dd inc{0.0f, 0.0f};
    for (int k = lane; k < p.R.K; k += kWarp) {
        dd lt, ld;
        if (log_probs(p, k, sL, sX, sZ, lt, ld))
            inc = dd_add(inc, dd_sub(p.target_seq ? dd_mul_f(lt, p.alpha) : lt, ld));
    }
    inc = warp_sum_dd(inc);
    if (lane == 0 && p.logw) {  // (no log-weights when only the draws are wanted)
        if (p.target_seq) {
            const float2 b = sL[2 * p.R.K];
            inc = dd_add(inc, dd{b.x, b.y});
        }
        if (p.log_reward) {
            const float r = __ldg(p.log_reward + s);
            if (!(fabsf(r) <= 3.402823466e38f)) raise_error(p.ws, kErrNonfinite);  // NaN or inf
            inc = dd_add(inc, two_prod(p.reward_scale, r));
        }
        const dd lw = dd_add(dd{lw_old, 0.0f}, inc);
        const float v = f_add(lw.hi, lw.lo);
        p.logw[s] = v;
        return v;
    }
    return 0.0f;
}

// The fused step's refcount array set to zero by the streaming pass (grid-stride), so that the
// finishing pass's remap, which starts only once the stream has completed, counts from zero.
__device__ __forceinline__ void zero_refcount(const StreamParams& p) {
    if (!p.refcount) return;
    const int stride = (int)(gridDim.x * blockDim.x);
    for (int i = (int)(blockIdx.x * blockDim.x + threadIdx.x); i < p.num_pages; i += stride)
        p.refcount[i] = 0;
}

// Page-table rows of one group after resampling, by threads 0..nthr-1 of a block: row j of the output
// is row anc[j] of the input (row j when the group was not resampled), W ints per access; every
// non-empty page id is counted in refcount. The input rows are read from `tin` (global memory),
// or from the block's staged copy `stage` (shared memory, the same layout) when it is given.
template <int W>
__device__ __forceinline__ void remap_rows_block(const StreamParams& p, const int32_t* tin, int32_t* tout,
                                                 const int32_t* anc, bool res, int N, int P, int nthr,
                                                 const int32_t* stage = nullptr) {
    using Vec = typename std::conditional<W == 4, int4, int>::type;
    const unsigned PW = (unsigned)(P / W);
    const unsigned n = (unsigned)N * PW;
    for (unsigned e = threadIdx.x; e < n; e += (unsigned)nthr) {
        const unsigned j = e / PW, col = e - j * PW;
        const int a = res ? anc[j] : (int)j;
        const Vec v = stage ? reinterpret_cast<const Vec*>(stage + (size_t)a * P)[col]
                            : __ldg(reinterpret_cast<const Vec*>(tin + (size_t)a * P) + col);
        reinterpret_cast<Vec*>(tout + (size_t)j * P)[col] = v;
        if (!p.refcount) continue;
        const int32_t* ids = reinterpret_cast<const int32_t*>(&v);
#pragma unroll
        for (int q = 0; q < W; ++q) {
            const int32_t id = ids[q];
            if (id == -1) continue;
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
// Chunk of the two-list dealing: `tag_item` is an index into the precise list (high bit set: the
// bonus row of a particle, cpr chunks per particle) or into the fast list (fslots rows of cpr
// chunks per sequence, row slots 0..fslots-1).
__device__ __forceinline__ ChunkRef chunk_ref_two_list(const StreamParams& p, uint32_t tag_item) {
    ChunkRef c;
    if (tag_item & 0x80000000u) {
        const uint32_t i = tag_item & 0x7fffffffu;
        c.s = (int)fast_div(i, p.div_cpr);
        c.chunk = (int)(i - (uint32_t)c.s * p.div_cpr.d);
        c.ks = seq_len(p.R, c.s, p.ws);
        c.slot = 2 * c.ks;
    } else {
        c.s = (int)fast_div(tag_item, p.div_fseq);
        const uint32_t rem = tag_item - (uint32_t)c.s * p.div_fseq.d;
        c.slot = (int)fast_div(rem, p.div_cpr);
        c.chunk = (int)(rem - (uint32_t)c.slot * p.div_cpr.d);
        if (p.drf_logq) c.slot *= 2;  // fast rows are the target rows 0 .. K-1 only
        c.ks = seq_len(p.R, c.s, p.ws);
    }
    c.valid = c.ks >= 0 && c.slot <= 2 * c.ks;
    c.is_draft = c.slot < 2 * c.ks && (c.slot & 1);
    const int k = c.slot >> 1;
    c.row = c.valid ? (c.is_draft ? drow_of(p.R, c.s, k) : trow_of(p.R, c.s, k)) : 0;
    return c;
}

// ------------------------------------------------------------------------------------------
// SD residual weights (the residual pass and the residual draw)
// ------------------------------------------------------------------------------------------

struct ResidualCtx {
    int n_t, n_d;
    dd inv_t, inv_d;  // 1 / (row total in units of 2^n)
    dd a_t, a_d;      // the same times 2^-n (exact), for the direct table
    bool direct;      // both rows' weights come straight from a direct table
};

// max(0, p_i - q_i), p_i = exp(c zt) / Z_t, q_i = exp(c zd) / Z_d, from raw logit bits. With a
// direct table both weights are one table entry times a_t (a_d); when float estimates of p_i and
// q_i (each within 2^-22 of the exact value) already put p_i below q_i, the result is 0 without
// the double-float products.
template <int DT>
__device__ __forceinline__ dd residual_weight(uint32_t bt, uint32_t bd, const ResidualCtx& c,
                                              const PreciseCtx& P) {
    dd pt, qd;
    const uint32_t ot = (bt & 0x7fffu) - kTabMagLo, od = (bd & 0x7fffu) - kTabMagLo;
    if (DT == 1 && c.direct && ot < kTabHalf && od < kTabHalf) {
        const float2 et = P.tab[ot + ((bt & 0x8000u) ? kTabStride : 0u)];
        const float2 ed = P.tab[od + ((bd & 0x8000u) ? kTabStride : 0u)];
        const float pf = f_mul(et.x, c.a_t.hi), qf = f_mul(ed.x, c.a_d.hi);
        if (pf < f_mul(qf, 1.0f - 0x1p-20f)) return dd{0.0f, 0.0f};
        pt = dd_mul(dd{et.x, et.y}, c.a_t);
        qd = dd_mul(dd{ed.x, ed.y}, c.a_d);
    } else {
        pt = precise_weight<DT>(bt, c.n_t, P);
        qd = precise_weight<DT>(bd, c.n_d, P);
        if (pt.hi > 0.0f) pt = dd_mul(pt, c.inv_t);
        if (qd.hi > 0.0f) qd = dd_mul(qd, c.inv_d);
    }
    dd d = two_sum(pt.hi, -qd.hi);
    d.lo = f_add(d.lo, f_sub(pt.lo, qd.lo));
    d = two_sum(d.hi, d.lo);
    return d.hi > 0.0f ? d : dd{0.0f, 0.0f};
}

// The direct-table products need n in [kDirectMinRef, kResidualMaxRef], so that the scaled
// reciprocals (and the products' low words) stay normal floats.
constexpr int kResidualMaxRef = 90;
__device__ __forceinline__ ResidualCtx residual_ctx(const SeqState* st, const PreciseCtx& P) {
    ResidualCtx c;
    c.n_t = __ldcg(&st->n_t);
    c.n_d = __ldcg(&st->n_d);
    c.inv_t = dd{__ldcg(&st->inv_t_hi), __ldcg(&st->inv_t_lo)};
    c.inv_d = dd{__ldcg(&st->inv_d_hi), __ldcg(&st->inv_d_lo)};
    c.direct = P.tab && P.direct && c.n_t >= kDirectMinRef && c.n_t <= kResidualMaxRef &&
               c.n_d >= kDirectMinRef && c.n_d <= kResidualMaxRef;
    const float st_ = pow2i(-c.n_t), sd_ = pow2i(-c.n_d);
    c.a_t = dd{f_mul(c.inv_t.hi, st_), f_mul(c.inv_t.lo, st_)};
    c.a_d = dd{f_mul(c.inv_d.hi, sd_), f_mul(c.inv_d.lo, sd_)};
    return c;
}

// Half item of the SD final-token pass (kModeSDFinal): item i (high bit set) is the target (i
// even) or draft (i odd) chunk of pair i >> 1 = sequence s's chunk `chunk` (pair = s * cpr +
// chunk); with `rows` the row is looked up in the hand-off state. Valid for the target half of every
// sequence and for the draft half of a sequence that draws a correction token; the target row is
// the one the sequence draws from (its bonus row, or the row of the rejected position).
__device__ __forceinline__ ChunkRef chunk_ref_sd_final(const StreamParams& p, uint32_t tag_item, bool rows) {
    ChunkRef c;
    const uint32_t i = tag_item & 0x7fffffffu;
    const int which = (int)(i & 1u);
    const uint32_t g = i >> 1;
    c.s = (int)fast_div(g, p.div_cpr);
    c.chunk = (int)(g - (uint32_t)c.s * p.div_cpr.d);
    c.slot = which;
    c.ks = 0;
    c.is_draft = which == 1;
    c.valid = true;
    c.row = 0;
    if (rows) {
        const int ks = seq_len(p.R, c.s, p.ws);
        const SeqState* st = ws_ptr<SeqState>(p.ws, p.L.seq) + c.s;
        c.valid = ks >= 0 && (which == 0 || __ldcg(&st->mode) == 1);
        c.row = c.valid ? (which ? __ldcg(&st->drow) : __ldcg(&st->trow)) : 0;
    }
    return c;
}

// Within a sequence the rows come bonus row first (position 0 is row slot 2ks, position q > 0 is
// slot q - 1), so that the bonus row's draw, the longest row epilogue, overlaps the streaming of
// the sequence's other rows instead of following its last chunk.
__device__ __forceinline__ ChunkRef chunk_ref(const StreamParams& p, uint32_t it) {
    ChunkRef c;
    c.s = (int)fast_div(it, p.div_seq);
    const uint32_t rem = it - (uint32_t)c.s * p.div_seq.d;
    const int pos = (int)fast_div(rem, p.div_cpr);
    c.chunk = (int)(rem - (uint32_t)pos * p.div_cpr.d);
    c.ks = seq_len(p.R, c.s, p.ws);
    c.slot = pos == 0 ? 2 * c.ks : pos - 1;
    c.valid = c.ks >= 0 && pos <= 2 * c.ks && !(p.drf_logq && pos > 0 && (c.slot & 1));
    c.is_draft = c.slot < 2 * c.ks && (c.slot & 1);
    const int k = c.slot >> 1;
    c.row = c.valid ? (c.is_draft ? drow_of(p.R, c.s, k) : trow_of(p.R, c.s, k)) : 0;
    return c;
}

}  // namespace smcsd
