// smcsd_internal.cuh -- shared device helpers, workspace layout and launch parameters of the
// GB300 verify / reweight / resample kernels.
//
// Work decomposition. Every logits row is cut into chunks of 4 KB (2048 bf16 or 1024 float32
// logits). One warp processes one chunk with eight 16-byte loads per lane issued back to back
// (each load instruction covers 512 contiguous bytes of the row), so a resident warp keeps 4 KB
// in flight. A chunk produces either
//   - a fast partial {max logit, sum exp((z - max) * c)} (hardware exp2), enough for the
//     normalisers that feed the accept tests and the weights, or
//   - for a row that will be sampled by inverse CDF, eight double-float sub-partials (one per
//     512-byte slice), each sum_i exp(c z_i) / 2^n_ref, plus their total, where n_ref is the
//     binary exponent of exp(c * max z) of the chunk. Inverse-CDF draws walk these totals, then
//     the sub-partials, then rescan one 512-byte slice.
// Counters in the workspace let the last warp that finishes a sequence's chunks run that
// sequence's epilogue ("last arriver finalises"): no block ever waits for another.
#pragma once

#include <cuda_runtime.h>
#include <float.h>
#include <limits.h>
#include <stdint.h>

#include "smcsd_math.cuh"

namespace smcsd {

constexpr int kWarp = 32;
constexpr int kChunkBytes = 4096;
constexpr int kLoads = 8;  // 16-byte loads per lane per chunk; also sub-partials per chunk
constexpr float kNegInf = -__builtin_huge_valf();

// status codes (values fixed by the public header)
constexpr int kOk = 0, kErrInvalid = -1, kErrDtype = -2, kErrWorkspace = -3, kErrCuda = -4,
              kErrNonfinite = -5, kErrRange = -6;

// largest |alpha * z / T| the double-float exponential accepts for a sampled row
constexpr float kMaxScaledLogit = 65536.0f;

template <int DT>
struct ElemT;
template <>
struct ElemT<0> {  // float32
    static constexpr int kBytes = 4;
    static constexpr int kPerVec = 4;
};
template <>
struct ElemT<1> {  // bf16
    static constexpr int kBytes = 2;
    static constexpr int kPerVec = 8;
};
template <int DT>
struct Geo {
    static constexpr int kChunk = kChunkBytes / ElemT<DT>::kBytes;  // logits per chunk
    static constexpr int kSub = kChunk / kLoads;                    // logits per sub-partial
    static constexpr int kPerVec = ElemT<DT>::kPerVec;              // logits per 16-byte load
};
__host__ __device__ inline int chunks_per_row(int V, int dtype) {
    int ch = kChunkBytes / (dtype == 0 ? 4 : 2);
    return (V + ch - 1) / ch;
}

// ------------------------------------------------------------------------------------------
// workspace layout
// ------------------------------------------------------------------------------------------

struct SeqState {  // per-sequence hand-off between the SD kernels
    int mode;      // 0: bonus draw from target row `trow`; 1: residual draw at (trow, drow)
    int acc;
    long long trow, drow;
    float inv_t_hi, inv_t_lo;  // 1 / (target row total) in units of 2^N_t
    float inv_d_hi, inv_d_lo;
    int n_t, n_d;
    int pad[2];
};

struct WsLayout {
    size_t flag;       // int32 error flag
    size_t cnt_seq1;   // uint32 [S]  first pass
    size_t cnt_seq2;   // uint32 [S]  second pass (SD)
    size_t cnt_seq3;   // uint32 [S]  third pass (SD)
    size_t cnt_group;  // uint32 [S]
    size_t cnt_misc;   // uint32 [16]
    size_t fast;       // float2 [S * (2K+1) * cpr]
    size_t ddtot;      // float4 [S * 2 * cpr]           chunk totals of sampled rows
    size_t ddsub;      // float4 [S * 2 * cpr * kLoads]  sub-partials of sampled rows
    size_t rtot;       // float4 [S * cpr]               residual chunk totals (SD)
    size_t rsub;       // float4 [S * cpr * kLoads]      residual sub-partials (SD)
    size_t seq;        // SeqState [S]
    size_t cdf;        // double [S]  resampling CDF scratch
    size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sized for the worst case over dtypes (float32 chunks are the smaller ones).
inline WsLayout ws_layout(int S, int K, int V) {
    WsLayout L{};
    const size_t s = (size_t)(S > 0 ? S : 1), k = (size_t)(K > 0 ? K : 0);
    const size_t cpr = (size_t)chunks_per_row(V > 0 ? V : 1, 0);
    size_t o = 0;
    L.flag = o;
    o = align256(o + 16);
    L.cnt_seq1 = o;
    o = align256(o + 4 * s);
    L.cnt_seq2 = o;
    o = align256(o + 4 * s);
    L.cnt_seq3 = o;
    o = align256(o + 4 * s);
    L.cnt_group = o;
    o = align256(o + 4 * s);
    L.cnt_misc = o;
    o = align256(o + 4 * 16);
    L.fast = o;
    o = align256(o + 8 * s * (2 * k + 1) * cpr);
    L.ddtot = o;
    o = align256(o + 16 * s * 2 * cpr);
    L.ddsub = o;
    o = align256(o + 16 * s * 2 * cpr * kLoads);
    L.rtot = o;
    o = align256(o + 16 * s * cpr);
    L.rsub = o;
    o = align256(o + 16 * s * cpr * kLoads);
    L.seq = o;
    o = align256(o + sizeof(SeqState) * s);
    L.cdf = o;
    o = align256(o + 8 * s);
    L.total = o;
    return L;
}

// Only the header, counters and CDF scratch are used by the resampling-only ops.
inline size_t ws_small_bytes(int S) {
    WsLayout L = ws_layout(S, 0, 1);
    return L.total;
}

template <typename T>
__device__ __forceinline__ T* ws_ptr(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

__device__ __forceinline__ void raise_error(void* ws, int code) {
    atomicCAS(reinterpret_cast<int*>(ws), 0, code);
}

// ------------------------------------------------------------------------------------------
// warp collectives
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_max_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ dd shfl_xor_dd(dd v, int o) {
    return dd{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ dd warp_sum_dd(dd v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = dd_add(v, shfl_xor_dd(v, o));
    return v;
}
// exclusive prefix of v over lanes (lane 0 gets 0), Kogge-Stone in double-float
__device__ __forceinline__ dd warp_exclusive_scan_dd(dd v, int lane) {
    dd incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        dd t{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
        if (lane >= o) incl = dd_add(incl, t);
    }
    dd ex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    return lane == 0 ? dd{0.0f, 0.0f} : ex;
}
__device__ __forceinline__ double warp_exclusive_scan_d(double v, int lane) {
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    double ex = __shfl_up_sync(0xffffffffu, incl, 1);
    return lane == 0 ? 0.0 : ex;
}

// ------------------------------------------------------------------------------------------
// loads
// ------------------------------------------------------------------------------------------

// Streaming 16-byte load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
// Coherent L2 load for data written by other blocks during the same kernel.
__device__ __forceinline__ float4 ld_cg4(const float4* p) { return __ldcg(p); }
__device__ __forceinline__ float2 ld_cg2(const float2* p) { return __ldcg(p); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Logit i of a row (scalar load), as float.
template <int DT>
__device__ __forceinline__ float logit_at(const void* row, long long i) {
    if (DT == 0) return __ldg(static_cast<const float*>(row) + i);
    uint16_t b = __ldg(static_cast<const unsigned short*>(row) + i);
    return __uint_as_float(((uint32_t)b) << 16);
}

// The logits of one chunk as seen by one lane: kLoads vectors of kPerVec logits each. Vector v
// of lane l covers logits chunk*kChunk + v*kSub + l*kPerVec + [0, kPerVec). Logits beyond V read
// as -inf.
template <int DT>
struct ChunkRegs {
    float x[kLoads][Geo<DT>::kPerVec];
};

template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(const void* row, int V, int chunk, int lane,
                                           ChunkRegs<DT>& r) {
    constexpr int PV = Geo<DT>::kPerVec;
    const long long base = (long long)chunk * Geo<DT>::kChunk + lane * PV;
    if (VEC) {
        uint4 raw[kLoads];
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            long long e = base + v * Geo<DT>::kSub;
            if (e < V) {
                raw[v] = ld_stream16(static_cast<const char*>(row) + e * ElemT<DT>::kBytes);
            } else {
                raw[v] = DT == 0 ? make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u)
                                 : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            }
        }
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
            if (DT == 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q) r.x[v][q] = __uint_as_float(w[q]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    r.x[v][2 * q] = bf16_lo(w[q]);
                    r.x[v][2 * q + 1] = bf16_hi(w[q]);
                }
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
#pragma unroll
            for (int q = 0; q < PV; ++q) {
                long long e = base + v * Geo<DT>::kSub + q;
                r.x[v][q] = e < V ? logit_at<DT>(row, e) : kNegInf;
            }
        }
    }
}

// Logits of one 512-byte slice (one vector per lane), for inverse-CDF rescans.
template <int DT, bool VEC>
__device__ __forceinline__ void load_slice(const void* row, int V, int chunk, int sub, int lane,
                                           float (&x)[Geo<DT>::kPerVec]) {
    constexpr int PV = Geo<DT>::kPerVec;
    const long long e0 = (long long)chunk * Geo<DT>::kChunk + sub * Geo<DT>::kSub + lane * PV;
    if (VEC && e0 < V) {
        uint4 raw = __ldcg(reinterpret_cast<const uint4*>(static_cast<const char*>(row) +
                                                          e0 * ElemT<DT>::kBytes));
        uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        if (DT == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) x[q] = __uint_as_float(w[q]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                x[2 * q] = bf16_lo(w[q]);
                x[2 * q + 1] = bf16_hi(w[q]);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < PV; ++q) x[q] = (e0 + q < V) ? logit_at<DT>(row, e0 + q) : kNegInf;
    }
}

// ------------------------------------------------------------------------------------------
// precise weights of sampled rows
// ------------------------------------------------------------------------------------------

// Scale c = alpha / T as a double-float (from the double quotient), and c * log2(e) as float.
struct Scale {
    float c_hi, c_lo;  // c as double-float
    float c2;          // c * log2(e), float, for the hardware exp2 path
    double c;          // c in double, for the normalisers
};

// exp(c * z) of one logit as (hi + lo) * 2^n. Returns false for a logit that contributes
// nothing (-inf, or c*z below -kMaxScaledLogit). NaN, +inf or c*z above kMaxScaledLogit raise
// SMCSD_ERR_NONFINITE and contribute nothing.
__device__ __forceinline__ bool precise_exp(float z, const Scale& sc, const Exp2Table& T,
                                            void* ws, ddx& out) {
    if (!(z > kNegInf)) {  // -inf or NaN
        if (z != z) raise_error(ws, kErrNonfinite);
        return false;
    }
    dd x = dd_mul_f(dd{sc.c_hi, sc.c_lo}, z);
    if (!(x.hi <= kMaxScaledLogit)) {
        raise_error(ws, kErrNonfinite);
        return false;
    }
    if (x.hi < -kMaxScaledLogit) return false;
    out = exp_split(x, T);
    return true;
}

// (hi + lo) * 2^(n - nref), n <= nref, as a double-float (flushes below 2^-126).
__device__ __forceinline__ dd scaled(const ddx& e, int nref) {
    float s = pow2i(e.n - nref);
    return dd{f_mul(e.hi, s), f_mul(e.lo, s)};
}

// Accumulate y (0 <= y <= 2) into a biased accumulator whose high part stays >= 4, so that
// Dekker's fast-two-sum is exact.
__device__ __forceinline__ void acc_biased(dd& acc, dd y) {
    float s = f_add(acc.hi, y.hi);
    float err = f_sub(y.hi, f_sub(s, acc.hi));
    acc.lo = f_add(acc.lo, f_add(err, y.lo));
    acc.hi = s;
}
constexpr float kBias = 4.0f;
__device__ __forceinline__ dd unbias(dd acc) {
    return fast_two_sum(f_sub(acc.hi, kBias), acc.lo);
}

// Partial record of a sampled row: value = (hi + lo) * 2^n.
__device__ __forceinline__ float4 pack_part(dd v, int n) {
    return make_float4(v.hi, v.lo, __int_as_float(n), 0.0f);
}
constexpr int kNoMass = INT_MIN / 2;  // n of an all-masked chunk

// ------------------------------------------------------------------------------------------
// per-sequence row layout (fixed K or ragged offsets)
// ------------------------------------------------------------------------------------------

struct Rows {
    const void* tgt;
    const void* drf;
    const int32_t* toks;
    const int32_t* toff;  // NULL = fixed layout
    const int32_t* doff;
    int S, K, V;
};

// Draft count of sequence s, or -1 (with an error raised) if its offsets are inconsistent.
__device__ __forceinline__ int seq_len(const Rows& R, int s, void* ws) {
    if (!R.toff) return R.K;
    int t0 = __ldg(R.toff + s), t1 = __ldg(R.toff + s + 1);
    int d0 = __ldg(R.doff + s), d1 = __ldg(R.doff + s + 1);
    int ks = d1 - d0;
    if (t0 < 0 || d0 < 0 || ks < 0 || ks > R.K || t1 - t0 != ks + 1) {
        raise_error(ws, kErrRange);
        return -1;
    }
    return ks;
}
__device__ __forceinline__ long long trow_of(const Rows& R, int s, int k) {
    return R.toff ? (long long)__ldg(R.toff + s) + k : (long long)s * (R.K + 1) + k;
}
__device__ __forceinline__ long long drow_of(const Rows& R, int s, int k) {
    return R.doff ? (long long)__ldg(R.doff + s) + k : (long long)s * R.K + k;
}
template <int DT>
__device__ __forceinline__ const void* row_ptr(const void* base, long long row, int V) {
    return static_cast<const char*>(base) + row * (long long)V * ElemT<DT>::kBytes;
}

// Hand-off of the last arriver: lane 0 counts the finished unit; the warp learns whether it
// was the last of `expected`; the last one resets the counter for the next call.
__device__ __forceinline__ bool arrive_last(unsigned* counter, unsigned expected, int lane) {
    unsigned last = 0;
    __threadfence();  // every lane's stores before the count
    __syncwarp();
    if (lane == 0) {
        unsigned old = atomicAdd(counter, 1u);
        last = (old == expected - 1);
        if (last) {
            atomicExch(counter, 0u);
            __threadfence();
        }
    }
    return __shfl_sync(0xffffffffu, last, 0) != 0;
}

}  // namespace smcsd
