// smcsd_sampling.cuh -- chunk partials (fast and precise), row normalisers, the inverse-CDF
// draw over a row, and per-group effective sample size with systematic resampling. Warp-level
// device code shared by the kernels.
#pragma once

#include <cuda_bf16.h>

#include "smcsd_internal.cuh"

namespace smcsd {

__device__ __forceinline__ float hw_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// floor(t) as an int for |t| < 2^22: add 1.5 * 2^23 rounding toward -inf, read the low bits.
__device__ __forceinline__ int floor_int(float t) {
    return __float_as_int(__fadd_rd(t, 12582912.0f)) - 0x4B400000;
}

// Scale c = alpha / T as a double-float (from the double quotient), c * log2(e) as float, and
// c in double for the normalisers.
struct Scale {
    float c_hi, c_lo;
    float c2;
    double c;
};

// ------------------------------------------------------------------------------------------
// precise weights exp(c z) of sampled rows
// ------------------------------------------------------------------------------------------
//
// exp(c z) is represented as e * 2^n with n = floor(z * c2) computed in float and e (about
// [1, 2)) a double-float. For bf16 logits with 2^-24 <= |z| < 64, e comes from a table over all
// such bf16 values (kTabSize entries with the zero entries, layout in smcsd_internal.cuh, filled
// from the general routine below, so both give identical bits); other logits use the general
// routine (double-float exp_split).

// the table is used only while |64 * c2| stays far inside floor_int's range
constexpr double kTabMaxScale = 4096.0;

struct PreciseCtx {
    Scale sc;
    const Exp2Table* T;  // shared memory
    const float2* tab;   // shared memory, or nullptr (float32 logits / very large scale)
    void* ws;
    bool direct;         // tab holds exp(c z) itself (c small enough to stay in float range)
};

// With c * 64 * log2(e) <= 125 every table value exp(c z), |z| < 64, is a normal float, so the
// table can hold the double-float value itself; then a logit's weight is one table load, and a
// block's sum is scaled by 2^-nref once. Chunks whose largest weight is below 2^-60 (their low
// words would be subnormal) or above 2^119 use the general routine instead.
constexpr double kDirectMaxScale = 1.35;
constexpr int kDirectMinRef = -60;

struct GW {
    float x, y;
    int n;
    int ok;
};

// exp(c z) = (x + y) * 2^n for any float z; ok = 0 for a weight of zero (-inf, or c z below
// -kMaxScaledLogit). NaN, +inf or c z above kMaxScaledLogit raise SMCSD_ERR_NONFINITE.
static __device__ __noinline__ GW general_weight(float z, float c_hi, float c_lo, float c2,
                                          const Exp2Table* T, void* ws) {
    GW r{0.0f, 0.0f, 0, 0};
    if (!(z > kNegInf)) {
        if (z != z) raise_error(ws, kErrNonfinite);
        return r;
    }
    const dd x = dd_mul_f(dd{c_hi, c_lo}, z);
    if (!(x.hi <= kMaxScaledLogit)) {
        raise_error(ws, kErrNonfinite);
        return r;
    }
    if (x.hi < -kMaxScaledLogit) return r;
    const ddx e = exp_split(x, *T);
    r.n = floor_int(f_mul(z, c2));
    const float s = pow2i(e.n - r.n);
    r.x = f_mul(e.hi, s);
    r.y = f_mul(e.lo, s);
    r.ok = 1;
    return r;
}

__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Fill a table (threads tid = 0..nthr-1 take part, then barrier `bar` over nthr threads).
__device__ __forceinline__ void build_exp_table(float2* tab, const Scale& sc, const Exp2Table* T,
                                                void* ws, bool direct, int tid, int nthr, int bar) {
    for (int i = tid; i < kTabSize; i += nthr) {
        const bool neg = i >= (int)kTabStride;
        const uint32_t m = (uint32_t)i - (neg ? kTabStride : 0u);
        if (m >= kTabHalf) {  // the zero entry after each half (and the unused entries)
            tab[i] = make_float2(0.0f, 0.0f);
            continue;
        }
        const uint32_t b = (kTabMagLo + m) | (neg ? 0x8000u : 0u);
        const GW g = general_weight(__uint_as_float(b << 16), sc.c_hi, sc.c_lo, sc.c2, T, ws);
        if (direct) {
            const float t = pow2i(g.n);
            tab[i] = make_float2(f_mul(g.x, t), f_mul(g.y, t));
        } else {
            tab[i] = make_float2(g.x, g.y);
        }
    }
    bar_sync(bar, nthr);
}

// The block's shared-memory table for scale sc. The first block that builds it for a workspace
// publishes it there (tag words: magic, then c_hi, c_lo, c2 bits); later calls with the same
// scale copy it instead of rebuilding. A published table is never overwritten, so a reader can
// never see a half-written one; calls with another scale build their own copy each time.
constexpr uint32_t kTabMagic = 0x54424c33u;
__device__ __forceinline__ void setup_exp_table(float2* tab, const Scale& sc, const Exp2Table* T,
                                                void* ws, uint32_t* gtag, float2* gtab, bool direct,
                                                int tid, int nthr, int bar) {
    __shared__ int state;  // 0: build and publish, 1: copy, 2: build only
    if (tid == 0) {
        uint32_t magic;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(magic) : "l"(gtag) : "memory");
        if (magic != kTabMagic)
            state = blockIdx.x == 0 ? 0 : 2;
        else
            state = (__ldcg(gtag + 1) == __float_as_uint(sc.c_hi) &&
                     __ldcg(gtag + 2) == __float_as_uint(sc.c_lo) &&
                     __ldcg(gtag + 3) == __float_as_uint(sc.c2))
                        ? 1
                        : 2;
    }
    bar_sync(bar, nthr);
    const int st = state;
    if (st == 1) {
        const uint4* src = reinterpret_cast<const uint4*>(gtab);
        uint4* dst = reinterpret_cast<uint4*>(tab);
        for (int i = tid; i < kTabSize / 2; i += nthr) dst[i] = __ldcg(src + i);
        bar_sync(bar, nthr);
        return;
    }
    build_exp_table(tab, sc, T, ws, direct, tid, nthr, bar);
    if (st == 0) {
        const uint4* src = reinterpret_cast<const uint4*>(tab);
        uint4* dst = reinterpret_cast<uint4*>(gtab);
        for (int i = tid; i < kTabSize / 2; i += nthr) dst[i] = src[i];
        __threadfence();
        bar_sync(bar, nthr);
        if (tid == 0) {
            gtag[1] = __float_as_uint(sc.c_hi);
            gtag[2] = __float_as_uint(sc.c_lo);
            gtag[3] = __float_as_uint(sc.c2);
            __threadfence();
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(gtag), "r"(kTabMagic) : "memory");
        }
    }
}

// Weight exp(c z) / 2^nref of one logit given its raw bits (see logit_bits), as a double-float.
template <int DT>
__device__ __forceinline__ dd precise_weight(uint32_t b, int nref, const PreciseCtx& P) {
    float ex, ey;
    int n;
    if (DT == 1 && P.tab && (!P.direct || nref >= kDirectMinRef)) {
        const uint32_t off = (b & 0x7fffu) - kTabMagLo;
        if (off < kTabHalf) {
            const float2 e = P.tab[off + ((b & 0x8000u) ? kTabStride : 0u)];
            ex = e.x;
            ey = e.y;
            n = P.direct ? 0 : floor_int(f_mul(bits_to_float<DT>(b), P.sc.c2));
        } else {
            const GW g = general_weight(bits_to_float<DT>(b), P.sc.c_hi, P.sc.c_lo, P.sc.c2, P.T, P.ws);
            if (!g.ok) return dd{0.0f, 0.0f};
            ex = g.x;
            ey = g.y;
            n = g.n;
        }
    } else {
        const GW g = general_weight(bits_to_float<DT>(b), P.sc.c_hi, P.sc.c_lo, P.sc.c2, P.T, P.ws);
        if (!g.ok) return dd{0.0f, 0.0f};
        ex = g.x;
        ey = g.y;
        n = g.n;
    }
    const float s = pow2i(n - nref);
    return dd{f_mul(ex, s), f_mul(ey, s)};
}

// Accumulate y (0 <= y <= ~2) into a biased accumulator whose high part stays >= 4, so that
// Dekker's fast-two-sum is exact. One packed f32x2 add forms both acc.hi + y.hi and
// acc.lo + y.lo; the exact rounding error of the first then joins the low part.
constexpr float kBias = 4.0f;
__device__ __forceinline__ void acc_biased(dd& acc, dd y) {
    float s, x;
    asm("{\n .reg .b64 a, b, c;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
        " add.rn.f32x2 c, a, b;\n mov.b64 {%0, %1}, c;\n}"
        : "=f"(s), "=f"(x)
        : "f"(acc.hi), "f"(acc.lo), "f"(y.hi), "f"(y.lo));
    const float err = f_sub(y.hi, f_sub(s, acc.hi));
    acc.lo = f_add(x, err);
    acc.hi = s;
}
__device__ __forceinline__ dd unbias(dd acc) { return fast_two_sum(f_sub(acc.hi, kBias), acc.lo); }

// Partial record of a sampled row: value = (x + y) * 2^n (z holds n's bits).
__device__ __forceinline__ float4 pack_part(dd v, int n) {
    return make_float4(v.hi, v.lo, __int_as_float(n), 0.0f);
}
constexpr int kNoMass = INT_MIN / 2;  // n of a chunk without mass

// ------------------------------------------------------------------------------------------
// chunk loads
// ------------------------------------------------------------------------------------------

// Interleaved chunk load for the fast path: vector v of lane l holds logits
// chunk*kChunk + v*(kChunk/8) + l*kPerVec + [0, kPerVec). Logits beyond V read as -inf.
template <int DT>
__device__ __forceinline__ void load_chunk_interleaved(const void* row, int V, bool vec, int chunk,
                                                       int lane, uint4 (&raw)[kLoads], uint64_t pol) {
    constexpr int PV = Geo<DT>::kPerVec;
    const long long base = (long long)chunk * Geo<DT>::kChunk + lane * PV;
    if (vec) {
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            const long long e = base + v * (Geo<DT>::kChunk / kLoads);
            raw[v] = e < V ? ld_stream16(static_cast<const char*>(row) + e * Geo<DT>::kBytes, pol)
                           : (DT == 0 ? make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u)
                                      : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u));
        }
    } else {
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (DT == 0) {
                    const long long e = base + v * (Geo<DT>::kChunk / kLoads) + j;
                    w[j] = e < V ? logit_bits_stream<0>(row, e, pol) : 0xff800000u;
                } else {
                    const long long e = base + v * (Geo<DT>::kChunk / kLoads) + 2 * j;
                    const uint32_t lo = e < V ? logit_bits_stream<1>(row, e, pol) : 0xff80u;
                    const uint32_t hi = e + 1 < V ? logit_bits_stream<1>(row, e + 1, pol) : 0xff80u;
                    w[j] = lo | (hi << 16);
                }
            }
            raw[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// A lane's contiguous block of kSub logits of a chunk (128 bytes) as 32 raw words; logits
// beyond V read as -inf.
template <int DT>
__device__ __forceinline__ void load_lane_block(const void* row, int V, bool vec, int chunk,
                                                int lane, uint32_t (&w)[32]) {
    constexpr int SUB = Geo<DT>::kSub;
    const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)lane * SUB;
    if (vec && e0 + SUB <= V) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + e0 * Geo<DT>::kBytes);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 q = __ldcg(p + i);
            w[4 * i] = q.x;
            w[4 * i + 1] = q.y;
            w[4 * i + 2] = q.z;
            w[4 * i + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (DT == 0) {
                w[j] = e0 + j < V ? logit_bits<0>(row, e0 + j) : 0xff800000u;
            } else {
                const uint32_t lo = e0 + 2 * j < V ? logit_bits<1>(row, e0 + 2 * j) : 0xff80u;
                const uint32_t hi = e0 + 2 * j + 1 < V ? logit_bits<1>(row, e0 + 2 * j + 1) : 0xff80u;
                w[j] = lo | (hi << 16);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// chunk partials
// ------------------------------------------------------------------------------------------

// Packed pairs of floats for the f32x2 instructions of sm_100 and later.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Fast partial of one chunk: {m, sum_i 2^(z_i c2 - fl(m c2))} with m the chunk's largest logit
// (raw, before scaling; c > 0 keeps the order), up to the rounding of the final rescaling. An
// all-masked chunk gives {-inf, 0}. The maximum runs as four independent chains; the exponent
// arguments and the sums as float pairs.
template <int DT>
__device__ __forceinline__ float2 fast_partial(const uint4 (&raw)[kLoads], float c2, void* ws) {
    float m;
    if (DT == 1) {
        __nv_bfloat162 mx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t w = j == 0 ? raw[0].x : j == 1 ? raw[0].y : j == 2 ? raw[0].z : raw[0].w;
            mx[j] = *reinterpret_cast<const __nv_bfloat162*>(&w);
        }
#pragma unroll
        for (int v = 1; v < kLoads; ++v) {
            const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) mx[j] = __hmax2(mx[j], *reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        }
        const __nv_bfloat162 mm = __hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3]));
        const uint32_t mw = *reinterpret_cast<const uint32_t*>(&mm);
        m = fmaxf(bf16_lo(mw), bf16_hi(mw));
    } else {
        float mf[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            mf[0] = fmaxf(mf[0], __uint_as_float(raw[v].x));
            mf[1] = fmaxf(mf[1], __uint_as_float(raw[v].y));
            mf[2] = fmaxf(mf[2], __uint_as_float(raw[v].z));
            mf[3] = fmaxf(mf[3], __uint_as_float(raw[v].w));
        }
        m = fmaxf(fmaxf(mf[0], mf[1]), fmaxf(mf[2], mf[3]));
    }
    // Each lane sums relative to its own maximum, so the exponentials need not wait for the
    // warp's; the lanes' sums are rescaled to the chunk maximum at the end.
    const bool live = m > kNegInf;
    const float q = live ? m * c2 : 0.0f;  // fl(m_lane c2)
    const unsigned long long C2 = f2_pack(c2, c2), NQ = f2_pack(-q, -q);
    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};  // (+0.0f, +0.0f) pairs
#pragma unroll
    for (int v = 0; v < kLoads; ++v) {
        const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
        if (DT == 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 t = f2_unpack(f2_fma(f2_pack(bf16_lo(w[j]), bf16_hi(w[j])), C2, NQ));
                acc[j] = f2_add(acc[j], f2_pack(hw_exp2(t.x), hw_exp2(t.y)));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 t = f2_unpack(f2_fma(f2_pack(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1])), C2, NQ));
                acc[j] = f2_add(acc[j], f2_pack(hw_exp2(t.x), hw_exp2(t.y)));
            }
        }
    }
    const float M = warp_max(m);
    if (M == kNegInf) {
        bool nan = false;
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (DT == 1)
                    nan |= (bf16_lo(w[j]) != bf16_lo(w[j])) | (bf16_hi(w[j]) != bf16_hi(w[j]));
                else
                    nan |= (__uint_as_float(w[j]) != __uint_as_float(w[j]));
            }
        }
        if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0) raise_error(ws, kErrNonfinite);
        return make_float2(kNegInf, 0.0f);
    }
    const float2 s0 = f2_unpack(f2_add(acc[0], acc[1])), s1 = f2_unpack(f2_add(acc[2], acc[3]));
    const float sl = (s0.x + s0.y) + (s1.x + s1.y);
    const float t = live ? sl * hw_exp2(q - M * c2) : 0.0f;
    const float s = warp_sum(t);
    if (!(s == s) || M == kPosInf) {  // NaN or +inf in the chunk
        if ((threadIdx.x & 31) == 0) raise_error(ws, kErrNonfinite);
    }
    return make_float2(M, s);
}

// Shared-memory load of one table entry through its shared-window byte address.
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
    float2 v;
    asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t shared_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// A lane block of kSub logits of a sampled row: piece(i) returns logits (i ^ sw) * PERP ..
// + PERP - 1 of the block as one 16-byte piece (PERP = 16 / element size), bits(q) the raw bits
// of logit q, those at or past V as -inf. GlobalSrc reads the row in global memory (16-byte
// loads when the row allows them, `vec`, else logit by logit); SharedSrc reads the block's 128
// bytes in shared memory, whose logits past V the caller has already overwritten with -inf.
template <int DT>
struct GlobalSrc {
    static constexpr int kUnroll = 1;  // pieces per step of the table pass
    const void* row;
    long long e0;
    int V;
    bool vec;
    __device__ __forceinline__ uint4 piece(int i) const {
        constexpr int PERP = 16 / Geo<DT>::kBytes;
        const long long e = e0 + (long long)i * PERP;
        if (vec && e + PERP <= V)
            return __ldca(reinterpret_cast<const uint4*>(static_cast<const char*>(row) + e * Geo<DT>::kBytes));
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (DT == 1) {
                const uint32_t lo = e + 2 * j < V ? logit_bits<DT>(row, e + 2 * j) : 0xff80u;
                const uint32_t hi = e + 2 * j + 1 < V ? logit_bits<DT>(row, e + 2 * j + 1) : 0xff80u;
                w[j] = lo | (hi << 16);
            } else {
                w[j] = e + j < V ? logit_bits<DT>(row, e + j) : 0xff800000u;
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ uint32_t bits(int q) const {
        return e0 + q < V ? logit_bits<DT>(row, e0 + q) : neg_inf_bits<DT>();
    }
    __device__ __forceinline__ bool live() const { return e0 < V; }  // the block holds a logit
};
template <int DT>
struct SharedSrc {
    static constexpr int kUnroll = 1;
    const unsigned char* base;  // the block's 128 bytes
    int sw;
    bool has;  // the block holds a logit
    __device__ __forceinline__ bool live() const { return has; }
    __device__ __forceinline__ uint4 piece(int i) const {
        return *reinterpret_cast<const uint4*>(base + ((i ^ sw) << 4));
    }
    __device__ __forceinline__ uint32_t bits(int q) const {
        return DT == 1 ? (uint32_t)reinterpret_cast<const unsigned short*>(base)[q]
                       : reinterpret_cast<const uint32_t*>(base)[q];
    }
};

// A lane block already in registers (pieces in natural order), for passes that load a block at
// once; only piece() with indices known at compile time (fully unrolled loops) keeps it there.
struct RegSrc {
    static constexpr int kUnroll = kLoads;
    uint4 v[kLoads];
    bool has;
    __device__ __forceinline__ uint4 piece(int i) const { return v[i]; }
    __device__ __forceinline__ bool live() const { return has; }
};

// With nref at most kDirectMaxRef the direct table pass can sum in absolute terms: its
// accumulator starts at 2^(nref+2) and stays below 2^(nref+8) <= 2^127.
constexpr int kDirectMaxRef = 119;

// Table byte offsets of both bf16 logits of a word, as 16-bit halves: |z|'s offset from kTabMagLo
// (taken modulo 2^16 without borrows between the halves) clamped to the zero entry kTabHalf,
// times 8, with the logit's sign bit kept in bit 15 (the negative half starts at byte 32768).
// `off` receives the unclamped offsets (a half >= kTabHalf: outside the table's domain).
__device__ __forceinline__ uint32_t tab_index2(uint32_t u, uint32_t& off) {
    off = ((u | 0x80008000u) - kTabMagLo * 0x10001u) ^ 0x80008000u;
    uint32_t c;
    asm("min.u16x2 %0, %1, %2;" : "=r"(c) : "r"(off), "r"(kTabHalf * 0x10001u));
    return (c << 3) | (u & 0x80008000u);  // (c < 4096: no bit crosses into the other half)
}

// Table pass over a bf16 lane block: the sum of exp(c z) / 2^nref over the logits inside the
// table's domain, as a double-float; bit i of `rare` is set when piece i holds a logit outside
// it (a zero entry stands in for it). KIND 0: the table holds exp(c z) itself and the pass adds
// the entries on an accumulator biased by 2^(nref+2), scaling the sum by 2^-nref once at the
// end; KIND 2: the table holds e with exp(c z) = e 2^n, n = floor(z c2), each entry scaled by
// 2^(n - nref) on the way in (bias 4). The low and high logit of every word feed two independent
// accumulators, renormalised after every piece. (The pass stays one piece per step: the hot
// loop of the streaming kernel has to fit the instruction cache.)
template <int KIND, typename Src>
__device__ __forceinline__ dd table_pass(const Src& src, uint32_t tab, int nref, float c2,
                                         unsigned& rare) {
    const float bias = KIND == 0 ? pow2i(nref + 2) : kBias;
    const float S = pow2i(-nref);
    dd a0{bias, 0.0f}, a1{bias, 0.0f};
    unsigned pieces = 0;
#pragma unroll(Src::kUnroll)
    for (int i = 0; i < kLoads; ++i) {
        const uint4 v = src.piece(i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t omax = 0;  // per half: the largest offset of the piece
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t u = w[j];
            uint32_t off;
            const uint32_t ix = tab_index2(u, off);
            asm("max.u16x2 %0, %1, %2;" : "=r"(omax) : "r"(omax), "r"(off));
            float2 e0 = lds_f2(tab + (ix & 0xffffu)), e1 = lds_f2(tab + (ix >> 16));
            if (KIND == 2) {
                const float s0 = pow2i(floor_int(f_mul(bf16_lo(u), c2)) - nref);
                const float s1 = pow2i(floor_int(f_mul(bf16_hi(u), c2)) - nref);
                e0 = make_float2(f_mul(e0.x, s0), f_mul(e0.y, s0));
                e1 = make_float2(f_mul(e1.x, s1), f_mul(e1.y, s1));
            }
            acc_biased(a0, dd{e0.x, e0.y});
            acc_biased(a1, dd{e1.x, e1.y});
        }
        if ((omax & 0xffffu) >= kTabHalf || (omax >> 16) >= kTabHalf) pieces |= 1u << i;
        a0 = fast_two_sum(a0.hi, a0.lo);
        a1 = fast_two_sum(a1.hi, a1.lo);
    }
    rare = pieces;
    dd s = dd_add(fast_two_sum(f_sub(a0.hi, bias), a0.lo), fast_two_sum(f_sub(a1.hi, bias), a1.lo));
    if (KIND == 0) s = dd{f_mul(s.hi, S), f_mul(s.lo, S)};
    return s;
}

// Precise partials of one chunk of a row that will be sampled. Lane l stores the double-float
// sum of exp(c z) / 2^nref over its block of kSub logits (read through `src`, see GlobalSrc) in
// sub_out[l]; lane 0 stores the chunk total in *tot_out. nref = floor(m c2) for the chunk's
// largest logit m. Logits the table does not cover (all of them when there is no table) are
// added by a second pass, which reads the pieces it needs through `again` (the same block).
template <int DT, typename Src, typename Again>
__device__ __forceinline__ void precise_core(const Src& src, const Again& again, int lane,
                                             const PreciseCtx& P, float4* tot_out,
                                             float4* sub_out) {
    // the block's largest logit (bf16: packed maxima; a NaN either comes out as the maximum or
    // lies outside the table's domain, and the second pass below reports it)
    float m = kNegInf;
    bool nan = false;
    if (DT == 1) {
        const uint4 v0 = src.piece(0);
        __nv_bfloat162 mx[2];
        mx[0] = *reinterpret_cast<const __nv_bfloat162*>(&v0.x);
        mx[1] = *reinterpret_cast<const __nv_bfloat162*>(&v0.y);
        mx[0] = __hmax2(mx[0], *reinterpret_cast<const __nv_bfloat162*>(&v0.z));
        mx[1] = __hmax2(mx[1], *reinterpret_cast<const __nv_bfloat162*>(&v0.w));
#pragma unroll
        for (int i = 1; i < kLoads; ++i) {
            const uint4 v = src.piece(i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mx[j & 1] = __hmax2(mx[j & 1], *reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        }
        const __nv_bfloat162 mm = __hmax2(mx[0], mx[1]);
        const uint32_t mw = *reinterpret_cast<const uint32_t*>(&mm);
        m = fmaxf(bf16_lo(mw), bf16_hi(mw));
        nan = (bf16_lo(mw) != bf16_lo(mw)) | (bf16_hi(mw) != bf16_hi(mw));
    } else {
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const uint4 v = src.piece(i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = __uint_as_float(w[j]);
                m = fmaxf(m, a);
                nan |= (a != a);
            }
        }
    }
    m = warp_max(m);
    nan = __any_sync(0xffffffffu, nan) || (m != m);
    const float cm = m * P.sc.c_hi;
    const bool ok = !nan && m > kNegInf && cm >= -kMaxScaledLogit && cm <= kMaxScaledLogit;
    if (!ok) {
        // NaN anywhere, +inf, or a scaled logit above the supported range is an error; a chunk
        // of -inf (or of logits whose weights all vanish) just has no mass
        const bool too_big = m > kNegInf && !(cm <= kMaxScaledLogit);  // includes +inf
        if ((nan || too_big) && lane == 0) raise_error(P.ws, kErrNonfinite);
        sub_out[lane] = pack_part(dd{0.0f, 0.0f}, kNoMass);
        if (lane == 0) *tot_out = pack_part(dd{0.0f, 0.0f}, kNoMass);
        return;
    }
    const int nref = floor_int(f_mul(m, P.sc.c2));
    dd sv{0.0f, 0.0f};
    unsigned rare = src.live() ? (1u << kLoads) - 1 : 0u;  // pieces left to the second pass
    bool covered = false;
    if (DT == 1 && P.tab && src.live()) {
        const uint32_t tab = shared_addr(P.tab);
        covered = true;
        if (!P.direct)
            sv = table_pass<2>(src, tab, nref, P.sc.c2, rare);
        else if (nref >= kDirectMinRef && nref <= kDirectMaxRef)
            sv = table_pass<0>(src, tab, nref, P.sc.c2, rare);
        else  // a chunk whose weights all lie below 2^-60, or above 2^119: the second pass alone
            covered = false;
    }
    if (__any_sync(0xffffffffu, rare != 0) && rare) {
        // second pass over the pieces of this lane's block with logits the table pass did not cover
        constexpr int PERP = 16 / Geo<DT>::kBytes;
        dd acc{kBias, 0.0f};
        do {
            const int i = __ffs(rare) - 1;
            rare &= rare - 1;
            const uint4 v = again.piece(i);
#pragma unroll 1
            for (int q = 0; q < PERP; ++q) {
                const int j = DT == 1 ? q >> 1 : q;
                const uint32_t wj = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
                const uint32_t b = DT == 1 ? ((q & 1) ? (wj >> 16) : (wj & 0xffffu)) : wj;
                if (b == neg_inf_bits<DT>()) continue;
                if (DT == 1 && covered && ((b & 0x7fffu) - kTabMagLo) < kTabHalf) continue;
                acc_biased(acc, precise_weight<DT>(b, nref, P));
            }
            acc = fast_two_sum(acc.hi, acc.lo);
        } while (rare);
        sv = dd_add(sv, unbias(acc));
    }
    sub_out[lane] = pack_part(sv, nref);
    const dd total = warp_total_fixed(sv);
    if (lane == 0) *tot_out = pack_part(total, nref);
}

// Precise partials of chunk `chunk` of a row in global memory: lane l's block of kSub logits
// from chunk * kChunk + l * kSub. With kRegs (and a 16-byte aligned row holding the whole
// block) the block's eight 16-byte loads are all in flight at once (kept in L2 for a later pass)
// and both passes run from registers; otherwise pieces are read as the passes go (cached in L1
// for the second).
template <int DT, bool kRegs = false>
__device__ __forceinline__ void precise_partials(const void* row, int V, bool vec, int chunk,
                                                 int lane, const PreciseCtx& P, float4* tot_out,
                                                 float4* sub_out) {
    const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)lane * Geo<DT>::kSub;
    const GlobalSrc<DT> g{row, e0, V, vec};
    if (kRegs && vec && __all_sync(0xffffffffu, e0 + Geo<DT>::kSub <= V)) {
        RegSrc r;
        const uint4* blk = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + e0 * Geo<DT>::kBytes);
#pragma unroll
        for (int i = 0; i < kLoads; ++i) r.v[i] = __ldg(blk + i);
        r.has = true;
        precise_core<DT>(r, g, lane, P, tot_out, sub_out);
    } else {
        precise_core<DT>(g, g, lane, P, tot_out, sub_out);
    }
}

// ------------------------------------------------------------------------------------------
// row normalisers from fast partials
// ------------------------------------------------------------------------------------------

// One fast partial {m, s} into a lane's running normaliser state: mq = fl(m c2) of its largest
// chunk so far, s the lane's sum relative to 2^mq, M its largest m. These three helpers spell
// out every rounding (no contraction left to the compiler), so that every lane layout that
// takes the same partials in the same order gets the same bits.
__device__ __forceinline__ void lse_acc(float& mq, float& s, float& M, float2 v, float c2) {
    const float pm = v.x, ps = v.y;
    if (pm == kNegInf) return;
    M = fmaxf(M, pm);
    const float q = f_mul(pm, c2);
    if (q > mq) {
        s = fmaf(s, hw_exp2(f_sub(mq, q)), ps);
        mq = q;
    } else {
        s = fmaf(ps, hw_exp2(f_sub(q, mq)), s);
    }
}
// A lane's sum relative to 2^Q, Q = fl(Mb c2) for the row's largest m, Mb.
__device__ __forceinline__ float lse_rescaled(float mq, float s, float Q) {
    return (mq == kNegInf) ? 0.0f : f_mul(s, hw_exp2(f_sub(mq, Q)));
}
// The normaliser from the row's largest m and the lanes' rescaled sums added up: c M exactly,
// plus the float log of the sum and the residual of fl(M c2).
__device__ __forceinline__ dd lse_final(float Mb, float Ssum, const Scale& sc) {
    if (Mb == kNegInf || !(Ssum > 0.0f)) return dd{__int_as_float(0x7fc00000), 0.0f};
    const float Q = f_mul(Mb, sc.c2);
    const float rQ = fmaf(Mb, sc.c2, -Q);  // exact residual of fl(M c2)
    const dd cM = dd_mul_f(dd{sc.c_hi, sc.c_lo}, Mb);
    return dd_add(cM, two_sum(logf(Ssum), f_mul(-rQ, SMCSD_LN2_HI)));
}

// Natural-log normaliser log sum_i exp(c z_i) of one row from its cpr fast partials, as a
// double-float on every lane (hi = NaN for a row without mass). Lane l takes partials
// l, l + 32, l + 64, ... in that order; the lanes' states meet in butterfly reductions. The
// partials' loads are all in flight together.
__device__ __forceinline__ dd row_lse_fast(const float2* part, int cpr, const Scale& sc, int lane) {
    float mq = kNegInf, s = 0.0f, M = kNegInf;
    for (int c0 = 0; c0 < cpr; c0 += 4 * kWarp) {
        float2 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + lane + j * kWarp;
            v[j] = c < cpr ? ld_cg2(part + c) : make_float2(kNegInf, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) lse_acc(mq, s, M, v[j], sc.c2);
    }
    const float Mb = warp_max(M);
    return lse_final(Mb, warp_sum(lse_rescaled(mq, s, f_mul(Mb, sc.c2))), sc);
}

// ------------------------------------------------------------------------------------------
// inverse-CDF draw over a row described by precise partials
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ dd part_value(float4 p, int N) {
    const int n = __float_as_int(p.z);
    if (n == kNoMass || !(p.x > 0.0f)) return dd{0.0f, 0.0f};
    const float s = pow2i(n - N);
    return dd{f_mul(p.x, s), f_mul(p.y, s)};
}

// Records of a row's partials in memory: chunk totals tot [cpr] and lane-block partials
// sub [cpr * kSubs], each {x, y, n bits, -} = (x + y) 2^n (see pack_part).
struct ArrayParts {
    const float4* tot;
    const float4* sub;
    __device__ __forceinline__ float4 chunk(int c) const { return ld_cg4(tot + c); }
    __device__ __forceinline__ float4 block(int c, int l) const { return ld_cg4(sub + (size_t)c * kSubs + l); }
};

// Draw token = min{ i : sum_{j<=i} w_j > u * sum_j w_j } over a row whose chunk totals
// (parts.chunk(c), c < cpr) and lane-block partials (parts.block(c, l)) describe the weights,
// rescanning one lane block with `block_weights(chunk, sub, lane, N, w[PL])` (PL = kSub / 32
// weights per lane, in units of 2^N, reproducing the partials exactly). Returns the token on
// every lane (-1 if the row has no mass). If `lse` is given it receives log(sum_j w_j) + N ln 2
// (in float). Lane l reads the contiguous chunk totals [l*cpl, l*cpl + cpl) once (kept in
// registers up to kDrawCache per lane) and serves both the common exponent and the chunk-level
// walk from them.
constexpr int kDrawCache = 4;
template <int PL, typename Parts, typename BlockFn>
__device__ int draw_inverse_cdf_parts(const Parts& parts, int cpr, int chunk_elems, int sub_elems,
                                      float u, int lane, BlockFn block_weights, float* lse) {
    const int cpl = (cpr + kWarp - 1) / kWarp;
    const int c_begin = min(lane * cpl, cpr), c_end = min(c_begin + cpl, cpr);
    const bool cached = cpl <= kDrawCache;
    float4 tc[kDrawCache];
    int N = kNoMass;
    if (cached) {
#pragma unroll
        for (int q = 0; q < kDrawCache; ++q) {
            tc[q] = c_begin + q < c_end ? parts.chunk(c_begin + q) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (tc[q].x > 0.0f) N = max(N, __float_as_int(tc[q].z));
        }
    } else {
        for (int c = lane; c < cpr; c += kWarp) {
            const float4 t = parts.chunk(c);
            if (t.x > 0.0f) N = max(N, __float_as_int(t.z));
        }
    }
    N = warp_max_i(N);
    if (N == kNoMass) return -1;

    // chunk level: lane l owns the contiguous chunks [c_begin, c_end)
    dd loc{0.0f, 0.0f};
    if (cached) {
#pragma unroll
        for (int q = 0; q < kDrawCache; ++q)
            if (c_begin + q < c_end) loc = dd_add(loc, part_value(tc[q], N));
    } else {
        for (int c = c_begin; c < c_end; ++c) loc = dd_add(loc, part_value(parts.chunk(c), N));
    }
    const dd excl = warp_exclusive_scan_dd(loc, lane);
    const dd incl = dd_add(excl, loc);
    const dd R{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    if (!(R.hi > 0.0f)) return -1;  // no mass (a residual whose records are all zero)
    if (lse) *lse = f_add(f_mul((float)N, SMCSD_LN2_HI), f_add(logf(R.hi), f_div(R.lo, R.hi)));
    const dd target = dd_mul_f(R, u);

    bool has = loc.hi > 0.0f && dd_gt(incl, target);
    unsigned bal = __ballot_sync(0xffffffffu, has);
    int owner;
    if (bal) {
        owner = __ffs(bal) - 1;
    } else {  // rounding put the target at or past the total: last lane with mass
        const unsigned m = __ballot_sync(0xffffffffu, loc.hi > 0.0f);
        owner = 31 - __clz(m);
    }
    int c_star = -1;
    dd base{0.0f, 0.0f};
    if (lane == owner) {
        dd p = excl;
        int last_pos = -1;
        dd last_base = p;
        bool found = false;
        auto visit = [&](int c, dd v) {
            if (found || !(v.hi > 0.0f)) return;
            last_pos = c;
            last_base = p;
            const dd qq = dd_add(p, v);
            if (dd_gt(qq, target)) {
                c_star = c;
                base = p;
                found = true;
            } else {
                p = qq;
            }
        };
        if (cached) {
#pragma unroll
            for (int q = 0; q < kDrawCache; ++q)
                if (c_begin + q < c_end) visit(c_begin + q, part_value(tc[q], N));
        } else {
            for (int c = c_begin; c < c_end; ++c) visit(c, part_value(parts.chunk(c), N));
        }
        if (c_star < 0) {
            c_star = last_pos;
            base = last_base;
        }
    }
    c_star = __shfl_sync(0xffffffffu, c_star, owner);
    base.hi = __shfl_sync(0xffffffffu, base.hi, owner);
    base.lo = __shfl_sync(0xffffffffu, base.lo, owner);
    block_weights.prefetch(c_star, lane);  // the rescan below reads from this chunk

    // lane-block level: one block per lane
    const dd sv = part_value(parts.block(c_star, lane), N);
    const dd sex = warp_exclusive_scan_dd(sv, lane);
    const dd sbase_l = dd_add(base, sex);
    has = sv.hi > 0.0f && dd_gt(dd_add(sbase_l, sv), target);
    bal = __ballot_sync(0xffffffffu, has);
    int s_star;
    if (bal) {
        s_star = __ffs(bal) - 1;
    } else {
        const unsigned m = __ballot_sync(0xffffffffu, sv.hi > 0.0f);
        s_star = m ? 31 - __clz(m) : 0;
    }
    dd sbase{__shfl_sync(0xffffffffu, sbase_l.hi, s_star), __shfl_sync(0xffffffffu, sbase_l.lo, s_star)};

    // logit level: rescan the block (lane l holds logits l*PL .. l*PL+PL-1 of it)
    dd w[PL];
    block_weights(c_star, s_star, lane, N, w);
    dd lsum{0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < PL; ++q) lsum = dd_add(lsum, w[q]);
    const dd lex = warp_exclusive_scan_dd(lsum, lane);
    dd p = dd_add(sbase, lex);
    int found = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < PL; ++q) {
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
        const unsigned m = __ballot_sync(0xffffffffu, lastpos >= 0);
        if (!m) return -1;
        tok_lane = 31 - __clz(m);
        tok_q = __shfl_sync(0xffffffffu, lastpos, tok_lane);
    }
    return c_star * chunk_elems + s_star * sub_elems + tok_lane * PL + tok_q;
}

template <int PL, typename BlockFn>
__device__ __forceinline__ int draw_inverse_cdf(const float4* tot, const float4* sub, int cpr,
                                                int chunk_elems, int sub_elems, float u, int lane,
                                                BlockFn block_weights, float* lse) {
    return draw_inverse_cdf_parts<PL>(ArrayParts{tot, sub}, cpr, chunk_elems, sub_elems, u, lane,
                                      block_weights, lse);
}

// Weights exp(c z) / 2^N of one lane block of a row (the rescan of a precise row).
template <int DT>
struct PreciseBlock {
    const void* row;
    int V;
    PreciseCtx P;
    static constexpr int PL = Geo<DT>::kSub / kWarp;
    __device__ __forceinline__ void operator()(int chunk, int sub, int lane, int N, dd (&w)[PL]) const {
        const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)sub * Geo<DT>::kSub + lane * PL;
#pragma unroll
        for (int q = 0; q < PL; ++q) {
            const long long e = e0 + q;
            w[q] = (e < V && check_ok(P.ws, e >= 0, -121, e))
                       ? precise_weight<DT>(logit_bits<DT>(row, e), N, P)
                       : dd{0.0f, 0.0f};
        }
    }
    // pull chunk `chunk` of the row towards L2 (lane l: its 128-byte piece)
    __device__ __forceinline__ void prefetch(int chunk, int lane) const {
        const long long e = (long long)chunk * Geo<DT>::kChunk + (long long)lane * (128 / Geo<DT>::kBytes);
        if (chunk >= 0 && e < V) l2_prefetch(static_cast<const char*>(row) + e * Geo<DT>::kBytes);
    }
};

// The common exponent N of a precise row (max over its chunk totals), on every lane.
__device__ __forceinline__ int row_exponent(const float4* tot, int cpr, int lane) {
    int N = kNoMass;
    for (int c = lane; c < cpr; c += kWarp) {
        const float4 t = ld_cg4(tot + c);
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
                                                const void* row, int V, const PreciseCtx& P,
                                                float u, int lane, float* lse) {
    PreciseBlock<DT> fn{row, V, P};
    return draw_inverse_cdf<PreciseBlock<DT>::PL>(tot, sub, cpr, Geo<DT>::kChunk, Geo<DT>::kSub,
                                                  u, lane, fn, lse);
}

// ------------------------------------------------------------------------------------------
// effective sample size and systematic resampling of one group (one warp)
// ------------------------------------------------------------------------------------------

// Number of children j in [0, N) with (j + U) / N < C, with the comparison evaluated exactly as
// written (double), so that it agrees with the definition a_j = min{ i : C_i > v_j }.
__device__ __forceinline__ int children_below(double C, double U, int N) {
    const double est = floor(C * (double)N - U);
    long long j = (long long)est;
    if (j < -1) j = -1;
    if (j > N - 1) j = N - 1;
    while (j + 1 <= N - 1 && (((double)(j + 1) + U) / (double)N) < C) ++j;
    while (j >= 0 && !((((double)j + U) / (double)N) < C)) --j;
    return (int)(j + 1);
}

// Resampling of a group of at most kWarp * PER particles with every weight computed
// once and held in registers (lane l holds particles l*per .. l*per+per-1), in double-float
// arithmetic on the FP32 pipes (about 2^-44 relative; this GPU's FP64 rate is far lower): the
// weights w_i = exp(logw_i - max) from the double-float exp, ESS = W^2 / W2, the CDF
// C_i = (prefix sum)/W with C_{N-1} = 1, the points v_j = (j + U)/N. The ancestor of child j is
// the number of particles i with C_i <= v_j (C is nondecreasing below 1 and C_{N-1} = 1 > v_j),
// found by a branch-free binary search over the C_i in the lanes' registers. The ancestors of
// the lane's children are also left in anc_reg (identity when not resampled).
constexpr int kResamplePer = 4;

// Value of register q of lane `src`, for a per-lane (src, q); `per` registers are live.
template <int PER>
__device__ __forceinline__ dd shfl_pick_dd(const dd (&v)[PER], int per, int src, int q) {
    dd r{0.0f, 0.0f};
#pragma unroll
    for (int q2 = 0; q2 < PER; ++q2) {
        if (q2 < per) {
            const float hi = __shfl_sync(0xffffffffu, v[q2].hi, src);
            const float lo = __shfl_sync(0xffffffffu, v[q2].lo, src);
            if (q2 == q) r = dd{hi, lo};
        }
    }
    return r;
}

// The log-weights are read from `logw` (global memory), or from lw_in (shared memory) when it is
// given; the zeros after a resampling always go to `logw`.
template <int PER>
__device__ __forceinline__ bool group_resample_small(float* logw, int N, float thr, float U,
                                                     int32_t* anc, float* ess_out, int32_t* res_out,
                                                     void* ws, int lane, const Exp2Table& T,
                                                     int (&anc_reg)[PER], const float* lw_in = nullptr) {
    const int per = (N + kWarp - 1) / kWarp;
    const int i0 = min(lane * per, N), i1 = min(i0 + per, N);
#pragma unroll
    for (int q = 0; q < PER; ++q) anc_reg[q] = i0 + q;
    float v[PER];
    bool bad = false;
    float m = kNegInf;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        v[q] = kNegInf;
        if (i0 + q < i1) {
            v[q] = lw_in ? lw_in[i0 + q] : __ldcg(logw + i0 + q);
            if (v[q] != v[q] || v[q] == kPosInf) bad = true;
            m = fmaxf(m, v[q]);
        }
    }
    const float M = warp_max(m);
    bad = __any_sync(0xffffffffu, bad) || M == kNegInf;
    if (bad) {
        if (lane == 0) raise_error(ws, kErrNonfinite);
        for (int j = lane; j < N; j += kWarp) anc[j] = j;
        if (lane == 0 && res_out) *res_out = 0;
        return false;
    }
    dd w[PER];
    dd loc{0.0f, 0.0f}, loc2{0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        w[q] = dd{0.0f, 0.0f};
        if (q < per && i0 + q < i1 && v[q] > kNegInf) {
            const ddx e = exp_split(two_sum(v[q], -M), T);  // logw_i - max, exact as a double-float
            const float sc = pow2i(e.n);
            w[q] = dd{f_mul(e.hi, sc), f_mul(e.lo, sc)};
            loc = dd_add(loc, w[q]);
            loc2 = dd_add(loc2, dd_mul(w[q], w[q]));
        }
    }
    const dd W = warp_sum_dd(loc), W2 = warp_sum_dd(loc2);
    const dd ess = dd_div(dd_mul(W, W), W2);
    const bool res = dd_gt(dd{thr, 0.0f}, ess);  // ESS < threshold
    if (lane == 0) {
        if (ess_out) *ess_out = f_add(ess.hi, ess.lo);
        if (res_out) *res_out = res ? 1 : 0;
    }
    if (!res) {
        for (int j = lane; j < N; j += kWarp) anc[j] = j;
        return false;
    }
    const dd rW = dd_recip(W), rN = dd_recip(dd{(float)N, 0.0f});
    dd C[PER], Vj[PER];
    dd r = warp_exclusive_scan_dd(loc, lane);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        C[q] = Vj[q] = dd{0.0f, 0.0f};
        if (q < per) {
            r = dd_add(r, w[q]);
            const int i = i0 + q;
            C[q] = i == N - 1 ? dd{1.0f, 0.0f} : dd_mul(r, rW);
            Vj[q] = dd_mul(two_sum((float)i, U), rN);
        }
    }
    int top = 1;
    while (top * 2 <= N) top *= 2;
    int cnt[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) cnt[q] = 0;
    for (int step = top; step > 0; step >>= 1) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            if (q < per) {
                const int probe = cnt[q] + step - 1;
                const int pc = min(probe, N - 1);
                const dd c = shfl_pick_dd(C, per, pc / per, pc - (pc / per) * per);
                if (probe < N && !dd_gt(c, Vj[q])) cnt[q] += step;
            }
        }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        anc_reg[q] = min(cnt[q], N - 1);
        if (i0 + q < i1) anc[i0 + q] = anc_reg[q];
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < PER; ++q)
        if (i0 + q < i1) logw[i0 + q] = 0.0f;
    return true;
}

// First attempt at the resampling of a group of at most kWarp particles (particle i on lane i), in
// float arithmetic, for the fused step's group part, whose single-warp chain sits on the step's
// critical path: w_i = exp(logw_i - max), ESS = W^2 / W2 with W = sum w_i, W2 = sum w_i^2, and
// ancestors a_j = #{ i : C_i <= v_j }, C_i = (w_0 + ... + w_i) / W, v_j = (j + U) / N, i.e.
// a_j = #{ i : x_i <= j } with x_i = C_i N - U. The rounding of each quantity is bounded (w_i and
// W within 1.3e-6 relative, W2 3.3e-6, ESS 6.1e-6, x_i N 2.7e-6 + 1e-6 absolute), and a decision
// is kept only when it lies farther from its boundary than a margin of about three times that
// bound: ESS not within 2e-5 relative of the threshold, and no x_i (i < N - 1; C_{N-1} = 1
// exactly) within 1e-5 (N + 1) of an integer. A kept decision is therefore the exact one, the same
// as the double-float path's. Otherwise (or for a weight that is not finite) nothing is written
// and false is returned; the caller then runs group_resample_small. On success writes what
// group_resample_small writes and returns true, with the lane's ancestor in anc_lane and the
// resampling flag in res (every lane). The log-weights are read from lw_in (shared memory) when it
// is given.
__device__ __forceinline__ bool group_resample_fast(float* logw, int N, float thr, float U, int32_t* anc,
                                                    float* ess_out, int32_t* res_out, int lane,
                                                    int& anc_lane, bool& res, const float* lw_in = nullptr) {
    const bool live = lane < N;
    const float v = live ? (lw_in ? lw_in[lane] : __ldcg(logw + lane)) : kNegInf;
    if (!__all_sync(0xffffffffu, !live || (v == v && v != kPosInf))) return false;
    const float M = warp_max(v);
    if (M == kNegInf) return false;
    const float w = v > kNegInf ? expf(v - M) : 0.0f;
    const float W = __shfl_sync(0xffffffffu, warp_sum(w), 0);
    const float W2 = __shfl_sync(0xffffffffu, warp_sum(w * w), 0);
    const float ess = W * W / W2;
    if (!(fabsf(ess - thr) > 2e-5f * ess)) return false;  // (also catches a NaN)
    res = ess < thr;
    if (!res) {
        anc_lane = lane;
        if (live) anc[lane] = lane;
        if (lane == 0) {
            if (ess_out) *ess_out = ess;
            if (res_out) *res_out = 0;
        }
        return true;
    }
    float S = w;  // inclusive prefix sum
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, S, o);
        if (lane >= o) S += t;
    }
    const float fN = (float)N;
    const float x = fmaf(S / W, fN, -U);
    const bool near = live && lane < N - 1 && fabsf(x - rintf(x)) <= 1e-5f * (fN + 1.0f);
    if (__any_sync(0xffffffffu, near)) return false;
    // k_i = ceil(x_i): particle i is counted by the children j >= k_i (never for i >= N - 1)
    const float k = lane < N - 1 ? ceilf(x) : 2.0f * fN;
    int a = lane;
    for (int j = 0; j < N; ++j) {
        const int c = __popc(__ballot_sync(0xffffffffu, k <= (float)j));
        if (lane == j) a = c < N - 1 ? c : N - 1;
    }
    anc_lane = a;
    if (live) anc[lane] = a;
    if (lane == 0) {
        if (ess_out) *ess_out = ess;
        if (res_out) *res_out = 1;
    }
    __syncwarp();
    if (live) logw[lane] = 0.0f;
    return true;
}

// logw [N] of one group (float, in/out). Writes ancestors [N], *ess_out, *res_out (if given).
// Returns whether the group was resampled (on every lane).
// The general path, for groups of any size (used above kWarp * kResamplePer particles).
static __device__ __noinline__ bool group_resample_general(float* logw, int N, float thr, float U,
                                                    int32_t* anc, float* ess_out, int32_t* res_out,
                                                    void* ws, int lane) {
    double M = -__builtin_huge_val();
    bool bad = false;
    for (int i = lane; i < N; i += kWarp) {
        const float v = __ldcg(logw + i);
        if (v != v || v == kPosInf) bad = true;
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
        const double w = exp((double)__ldcg(logw + i) - M);
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
    const double run = warp_exclusive_scan_d(loc, lane);
    const double Ud = (double)U;
    int Jend = -1;
    {
        double r = run;
        int J = 0;
        for (int i = i0; i < i1; ++i) {
            r += exp((double)__ldcg(logw + i) - M);
            const double C = (i == N - 1) ? 1.0 : r / W;
            J = children_below(C, Ud, N);
        }
        if (i1 > i0) Jend = J;
    }
    // a lane with an empty block passes its predecessor's value on
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, Jend, o);
        if (lane >= o && Jend < 0) Jend = t;
    }
    int Jstart = __shfl_up_sync(0xffffffffu, Jend, 1);
    if (lane == 0 || Jstart < 0) Jstart = 0;
    double r = run;
    int Jprev = Jstart;
    for (int i = i0; i < i1; ++i) {
        r += exp((double)__ldcg(logw + i) - M);
        const double C = (i == N - 1) ? 1.0 : r / W;
        const int J = children_below(C, Ud, N);
        for (int j = Jprev; j < J; ++j) anc[j] = i;
        Jprev = max(Jprev, J);
    }
    __syncwarp();
    for (int i = lane; i < N; i += kWarp) logw[i] = 0.0f;
    return true;
}

// logw [N] of one group (float, in/out). Writes ancestors [N], *ess_out, *res_out (if given).
// Returns whether the group was resampled (on every lane).
__device__ __forceinline__ bool group_resample(float* logw, int N, float thr, float U, int32_t* anc,
                                               float* ess_out, int32_t* res_out, void* ws, int lane,
                                               const Exp2Table& T) {
    if (N <= kWarp) {
        int a;
        bool res;
        if (group_resample_fast(logw, N, thr, U, anc, ess_out, res_out, lane, a, res)) return res;
    }
    if (N <= kWarp * kResamplePer) {
        int anc_reg[kResamplePer];
        return group_resample_small(logw, N, thr, U, anc, ess_out, res_out, ws, lane, T, anc_reg);
    }
    return group_resample_general(logw, N, thr, U, anc, ess_out, res_out, ws, lane);
}

}  // namespace smcsd
