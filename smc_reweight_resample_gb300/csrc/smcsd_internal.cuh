// smcsd_internal.cuh -- shared device helpers, workspace layout and constants of the GB300
// verify / reweight / resample kernels.
//
// Work decomposition. Every logits row is cut into chunks of 4 KB (2048 bf16 or 1024 float32
// logits); one warp processes one chunk with eight 16-byte loads per lane issued back to back,
// so each resident warp keeps 4 KB in flight. A chunk produces either
//   - a fast partial {max logit, sum exp(c (z - max))} (hardware exp2), enough for the
//     normalisers that feed the accept tests and the weights (lanes read interleaved 16-byte
//     vectors: every load instruction covers 512 contiguous bytes), or
//   - for a row that will be sampled by inverse CDF, double-float sums of exp(c z) / 2^nref,
//     one per lane over the lane's own contiguous block of 64 (bf16) or 32 (float32) logits,
//     plus their total; nref is the binary exponent of the chunk's largest weight. An
//     inverse-CDF draw walks the chunk totals, then one chunk's 32 lane blocks, then rescans
//     one block.
// Counters in the workspace let the last warp that finishes a sequence's chunks run that
// sequence's epilogue ("last arriver finalises"): no block ever waits for another.
#pragma once

#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "smcsd_fastdiv.h"
#include "smcsd_math.cuh"

namespace smcsd {

constexpr int kWarp = 32;
constexpr int kChunkBytes = 4096;
constexpr int kLoads = 8;   // 16-byte loads per lane per chunk
constexpr int kSubs = 32;   // sub-partials (lane blocks) per chunk of a precise row
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();

// status codes (values fixed by the public header)
constexpr int kOk = 0, kErrInvalid = -1, kErrDtype = -2, kErrWorkspace = -3, kErrCuda = -4,
              kErrNonfinite = -5, kErrRange = -6, kErrTimeout = -7;

// largest |alpha * z / T| the double-float exponential accepts for a sampled row
constexpr float kMaxScaledLogit = 65536.0f;

template <int DT>
struct Geo;
template <>
struct Geo<0> {  // float32
    static constexpr int kBytes = 4;
    static constexpr int kPerVec = 4;
    static constexpr int kChunk = kChunkBytes / 4;  // 1024 logits
    static constexpr int kSub = kChunk / kSubs;     // 32 logits per lane block
};
template <>
struct Geo<1> {  // bf16
    static constexpr int kBytes = 2;
    static constexpr int kPerVec = 8;
    static constexpr int kChunk = kChunkBytes / 2;  // 2048 logits
    static constexpr int kSub = kChunk / kSubs;     // 64 logits per lane block
};
__host__ __device__ inline int chunks_per_row(int V, int dtype) {
    int ch = kChunkBytes / (dtype == 0 ? 4 : 2);
    return (V + ch - 1) / ch;
}

// Geometry of the exp table of precise weights (bf16 logits): one entry per bf16 magnitude in
// [2^-24, 64) for each sign, the positive ones at [0, kTabHalf), the negative ones at
// [kTabStride, kTabStride + kTabHalf), each half followed by a zero entry (entries between the
// halves, and one of padding at the end, are zero too). The negative half starts at entry 4096,
// byte 32768 of the 8-byte entries: a logit's byte offset is its magnitude's times 8 with its
// sign bit in bit 15, both halves of a 32-bit word of logits at once (tab_index2).
constexpr uint32_t kTabMagLo = 0x3380u;                 // bf16 bits of 2^-24
constexpr uint32_t kTabMagHi = 0x4280u;                 // bf16 bits of 64
constexpr uint32_t kTabHalf = kTabMagHi - kTabMagLo;    // 3840 magnitudes per sign
constexpr uint32_t kTabStride = 4096u;                  // entry of the negative half's start
constexpr int kTabSize = (int)(kTabStride + kTabHalf + 2u);  // 7938 entries (an even count)
static_assert(kTabHalf * 8u < 32768u && kTabStride * 8u == 32768u, "exp table byte offsets");

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
    float theta;  // residual draw: p_i > q_i exactly when z_t,i - z_d,i > theta (to float accuracy)
    int pad;
};

struct WsLayout {
    size_t flag;       // int32 error flag
    size_t cnt_seq2;   // uint32 [S]  second pass (SD)
    size_t cnt_seq3;   // uint32 [S]  third pass (SD)
    size_t cnt_group;  // uint32 [S]
    size_t cnt_misc;   // uint32 [16]
    size_t claim;      // uint32 [64]  chunk claim counters (one per stripe) and a blocks-done count
    size_t fast;       // float2 [S * (2K+1) * cpr]
    size_t ddtot;      // float4 [S * 2 * cpr]          chunk totals of sampled rows
    size_t ddsub;      // float4 [S * 2 * cpr * kSubs]  lane-block partials of sampled rows
    size_t rtot;       // float4 [S * cpr]              residual chunk totals (SD)
    size_t rsub;       // float4 [S * cpr * kSubs]      residual lane-block partials (SD)
    size_t seq;        // SeqState [S]
    size_t tab;        // cached exp table: 4 tag words + kTabSize float2 (see setup_exp_table)
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
    L.cnt_seq2 = o;
    o = align256(o + 4 * s);
    L.cnt_seq3 = o;
    o = align256(o + 4 * s);
    L.cnt_group = o;
    o = align256(o + 4 * s);
    L.cnt_misc = o;
    o = align256(o + 4 * 16);
    L.claim = o;
    o = align256(o + 4 * 64);
    L.fast = o;
    o = align256(o + 8 * s * (2 * k + 1) * cpr);
    L.ddtot = o;
    o = align256(o + 16 * s * 2 * cpr);
    L.ddsub = o;
    o = align256(o + 16 * s * 2 * cpr * kSubs);
    L.rtot = o;
    o = align256(o + 16 * s * cpr);
    L.rsub = o;
    o = align256(o + 16 * s * cpr * kSubs);
    L.seq = o;
    o = align256(o + sizeof(SeqState) * s);
    L.tab = o;
    o = align256(o + 16 + 8 * (size_t)kTabSize);
    L.total = o;
    return L;
}

// Only the header and the counters are used by the resampling-only ops.
inline size_t ws_small_bytes(int S) { return ws_layout(S, 0, 1).cnt_misc + 256; }

template <typename T>
__device__ __forceinline__ T* ws_ptr(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

__device__ __forceinline__ void raise_error(void* ws, int code) {
    atomicCAS(reinterpret_cast<int*>(ws), 0, code);
}

// Opt-in self-checks (build with -DSMCSD_CHECKS): a failed check records a site code (-100 and
// below) in the error flag and the offending value in the next word, and the caller skips the
// access.
#ifdef SMCSD_CHECKS
__device__ __forceinline__ bool check_ok(void* ws, bool cond, int site, long long value) {
    if (!cond) {
        if (atomicCAS(reinterpret_cast<int*>(ws), 0, site) == 0)
            reinterpret_cast<long long*>(ws)[1] = value;
    }
    return cond;
}
#else
__device__ __forceinline__ bool check_ok(void*, bool, int, long long) { return true; }
#endif

// ------------------------------------------------------------------------------------------
// warp collectives
// ------------------------------------------------------------------------------------------

// Warp maxima in one instruction each (redux.sync: integers since sm_80, floats since sm_100),
// on every lane; a NaN lane is passed over, as fmaxf does.
__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ int warp_max_i(int v) {
    int r;
    asm("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
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
// Warp total of non-negative double-floats below 2^7 (a lane block's sum of at most 64 weights
// below 2, in units of its chunk's 2^n), valid on lane 0: each lane's parts are scaled exactly to
// fixed point with unit 2^-50 and rounded to integers (at most 2^-50 off per lane), the 64-bit
// integers are added exactly over the warp (32 lanes below 2^57 each stay below 2^62), and the
// total goes back to a double-float. Within 2^-45 of the exact total, for about a fifth of the
// instructions of a double-float butterfly.
__device__ __forceinline__ dd warp_total_fixed(dd v) {
    constexpr float kUp = 1125899906842624.0f;        // 2^50
    constexpr float kDown = 8.8817841970012523e-16f;  // 2^-50
    long long t = __float2ll_rn(v.hi * kUp) + __float2ll_rn(v.lo * kUp);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
    const float hi = __ll2float_rn(t);
    const float lo = __ll2float_rn(t - __float2ll_rn(hi));
    return fast_two_sum(hi * kDown, lo * kDown);
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

// L2 policy for data read exactly once (the logits): evicted first, so that the stream does not
// push the small per-row partials, the tables and the epilogues' code out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Streaming 16-byte load through the non-coherent path, not kept in L1, evicted first from L2.
__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ void l2_prefetch(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Coherent L2 loads for data written by other blocks during the same kernel.
__device__ __forceinline__ float4 ld_cg4(const float4* p) { return __ldcg(p); }
__device__ __forceinline__ float2 ld_cg2(const float2* p) { return __ldcg(p); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Raw bit pattern of logit i of a row: the bf16 bits in the low half (DT 1) or the float bits.
template <int DT>
__device__ __forceinline__ uint32_t logit_bits(const void* row, long long i) {
    if (DT == 0) return __ldg(static_cast<const unsigned*>(row) + i);
    return (uint32_t)__ldg(static_cast<const unsigned short*>(row) + i);
}
// The same for a streamed element, evicted first from L2.
template <int DT>
__device__ __forceinline__ uint32_t logit_bits_stream(const void* row, long long i, uint64_t pol) {
    if (DT == 0) {
        uint32_t v;
        asm volatile("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;"
                     : "=r"(v)
                     : "l"(static_cast<const unsigned*>(row) + i), "l"(pol));
        return v;
    }
    unsigned short v;
    asm volatile("ld.global.nc.L2::cache_hint.u16 %0, [%1], %2;"
                 : "=h"(v)
                 : "l"(static_cast<const unsigned short*>(row) + i), "l"(pol));
    return (uint32_t)v;
}
template <int DT>
__device__ __forceinline__ float bits_to_float(uint32_t b) {
    return DT == 0 ? __uint_as_float(b) : __uint_as_float(b << 16);
}
template <int DT>
__device__ __forceinline__ float logit_at(const void* row, long long i) {
    return bits_to_float<DT>(logit_bits<DT>(row, i));
}
template <int DT>
__device__ __forceinline__ uint32_t neg_inf_bits() {
    return DT == 0 ? 0xff800000u : 0xff80u;
}

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
    return static_cast<const char*>(base) + row * (long long)V * Geo<DT>::kBytes;
}

// Dynamic dealing of the chunks: the items of stripe j are j, j + n, j + 2n, ... (n stripes);
// claimer j of every block takes the next one from the stripe's counter. Returns -1 when the
// stripe is used up. The counters start at zero and the last block to finish resets them
// (reset_claims).
constexpr int kClaimDone = 63;  // index of the blocks-done count among the claim words
__device__ __forceinline__ long long claim_item(unsigned* claim, int j, int n, long long items) {
    const long long it = (long long)atomicAdd(claim + j, 1u) * n + j;
    return it < items ? it : -1;
}

// Programmatic dependent launch: the streaming pass lets the finishing pass be scheduled early;
// the finishing pass waits for the streaming pass to complete (and its writes to be visible)
// before it reads them. Both are no-ops without a programmatic dependency.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Completion count. Every arrival is a release at device scope (the warp's stores, ordered
// before lane 0 by the warp barrier, become visible before the count); only the last arriver
// then takes an acquire fence before it reads what the others stored. The last arriver resets
// the counter for the next call.
__device__ __forceinline__ unsigned atom_add_release(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}
__device__ __forceinline__ void fence_acquire() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ bool arrive_last(unsigned* counter, unsigned expected, int lane) {
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
        const unsigned old = atom_add_release(counter, 1u);
        last = (old == expected - 1);
        if (last) {
            fence_acquire();
            atomicExch(counter, 0u);
        }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    return last != 0;
}

// Called by one thread of each block once all of the block's claimers have stopped: the last
// block to get here resets the n stripe counters and the blocks-done count for the next call.
__device__ __forceinline__ void reset_claims(unsigned* claim, int n) {
    const unsigned old = atom_add_release(claim + kClaimDone, 1u);
    if (old == gridDim.x - 1) {
        fence_acquire();
        for (int j = 0; j < n; ++j) atomicExch(claim + j, 0u);
        atomicExch(claim + kClaimDone, 0u);
    }
}

}  // namespace smcsd
