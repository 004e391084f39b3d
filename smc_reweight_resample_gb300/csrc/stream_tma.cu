// stream_tma.cu -- the streaming pass over 16-byte-aligned logits rows as a TMA pipeline.
//
// One block per SM: two producer warps that move 4 KB chunks of logits from HBM into a ring of
// kRing = 32 shared-memory slots with the bulk-copy engine (cp.async.bulk, completion counted on
// one mbarrier per slot; lane j < 16 of producer warp w fills slot 16 w + j, so the two warps'
// refills run side by side on two sub-partitions), and kTmaConsumers consumer warps
// that take the slots in the order they were filled from a shared counter, wait for theirs and
// compute the chunk's partial (fast or precise, smcsd_sampling.cuh) into the workspace, where
// the finishing pass (finish.cu) picks the partials up. A fast chunk is copied into registers
// and its slot handed back (a second mbarrier per slot) before the arithmetic, so that nearly
// the whole ring stays in flight; a precise chunk, read from the slot twice, keeps it until done. Every
// logit crosses HBM exactly once.
//
// Chunks are dealt from two lists, each round-robin over the B blocks (smcsd_deal.h): the precise
// chunks (the rows that are sampled, one per particle) and the fast chunks (all other rows). Block
// b takes chunks b, b+B, b+2B, ... of the precise list and B-1-b, 2B-1-b, ... of the fast list (so
// the blocks left with one precise chunk more get no extra fast chunk), puts the precise chunks
// the fast ones cannot pair up first, then interleaves one precise chunk to fper fast ones (three
// quarters of the fast rows per sampled row), and ends on the fast chunks left over: every block
// gets the same share of each kind, the precise ones over the first four fifths of the pass, and
// finishes on cheap chunks, without a shared counter (a claim from one would put an atomic round
// trip on the producer's path). The producer lane of slot j loads the block's local chunks
// 32 * round + j.
//
// Every wait is bounded (about 2 s of wall time): a wait that runs out records
// SMCSD_ERR_TIMEOUT in the workspace and the warp leaves; the producer, before it leaves,
// waits (again bounded) for the copies it started.
#include "smcsd_epilogue.cuh"

namespace smcsd {

constexpr int kTmaConsumers = 18;
constexpr int kTmaProducers = 2;                      // producer warps, kRing / 2 slots each
constexpr int kTmaThreads = (kTmaConsumers + kTmaProducers) * kWarp;
constexpr int kRing = kWarp;  // one slot per producer lane
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

constexpr size_t kSmemRing = (size_t)kRing * kChunkBytes;
constexpr size_t kSmemTab = (size_t)kTabSize * sizeof(float2);
constexpr size_t kSmemBytes =
    kSmemRing + kSmemTab + sizeof(Exp2Table) + 2 * kRing * 8 + kRing * 8 + 16;
constexpr uint32_t kTagNone = 0xffffffffu;  // slot never loaded
constexpr uint32_t kTagDone = 0xfffffffeu;  // the slot's producer lane has no more chunks
// The tag word of a fast chunk (no kPreciseBit) carries what its consumer needs, decoded once by
// the producer (which decodes the chunk's list index anyway to address the copy): the index of
// the chunk's partial, (s * slots + row slot) * cpr + chunk, below 2^29 (2^29 chunks of 4 KB
// would be 2 TiB of logits), whether the row is a draft row, and whether the chunk is the row's
// last.
constexpr uint32_t kFastTailBit = 1u << 30, kFastDraftBit = 1u << 29, kFastIndexMask = kFastDraftBit - 1u;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Relaxed arrivals: they order nothing, so they never wait for this warp's outstanding global
// accesses (partial stores). Used where nothing written before the arrival is read by
// the waiting side (the data comes through the bulk copy or has already been read out).
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the phase of `parity` (try_wait may suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete, for at most `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
// Slot tags: one 64-bit word per slot, written by the producer once the slot's chunk is on its
// way: the block-local sequence number k of the load in the high half, the chunk's index in the
// low half. A consumer holding k waits for its tag first, so that the full barrier it then waits
// on is known to be in the phase of chunk k: a parity wait alone cannot tell that phase from the
// one two loads earlier, and the consumers take the slots from a shared counter, so a consumer
// can reach a slot before the previous chunk of that slot has landed. An aligned 8-byte access
// is single-copy atomic, so the chunk index comes with the tag and neither side needs a fence.
__device__ __forceinline__ void tag_store(uint32_t addr, uint32_t k, uint32_t item) {
    const unsigned long long v = ((unsigned long long)k << 32) | item;
    asm volatile("st.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tag_load(uint32_t addr) {
    unsigned long long v;
    asm volatile("ld.relaxed.cta.shared::cta.b64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}
// Wait (at most `limit_ns`) until the tag at `addr` reads k or kTagDone; the tag word seen is
// left in `seen`.
__device__ __forceinline__ bool tag_wait(uint32_t addr, uint32_t k, unsigned long long& seen,
                                         unsigned long long limit_ns = kWaitLimitNs) {
    seen = tag_load(addr);
    uint32_t hi = (uint32_t)(seen >> 32);
    if (hi == k || hi == kTagDone) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        __nanosleep(32);
        seen = tag_load(addr);
        hi = (uint32_t)(seen >> 32);
        if (hi == k || hi == kTagDone) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Diagnostic: the pipeline's two waits, run by one warp against a full barrier and a slot tag
// that nothing completes, each giving up after limit_ns and recording kErrTimeout, as the
// streaming pass does when its pipeline stalls. No copy is issued, so none is in flight when the
// kernel returns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(void* ws, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ __align__(8) unsigned long long tag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        tag = (unsigned long long)kTagNone << 32;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const bool got_bar = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), 0u, limit_ns));
    unsigned long long seen = 0;
    const bool got_tag = __all_sync(0xffffffffu, tag_wait(smem_u32(&tag), 0u, seen, limit_ns));
    if (threadIdx.x == 0 && (!got_bar || !got_tag)) raise_error(ws, kErrTimeout);
}

// Makes every word of `raw` an input of an (empty) instruction: what follows in program order
// is issued only after all of them have arrived in registers.
__device__ __forceinline__ void consume_all(const uint4 (&raw)[kLoads]) {
    uint32_t x = 0;
#pragma unroll
    for (int v = 0; v < kLoads; ++v) x ^= raw[v].x ^ raw[v].y ^ raw[v].z ^ raw[v].w;
    asm volatile("" ::"r"(x) : "memory");
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`, with L2 policy `pol`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// A producer lane: it owns slot `slot` and loads the block's chunks 32 * round + slot into it,
// each once the consumer of the slot's previous chunk has handed the slot back, then tags the
// slot with the block-local sequence number k = 32 * round + slot and the chunk's index. A lane out
// of chunks tags its slot kTagDone. The lanes poll their slots together (one non-blocking test per
// lane per pass), so no lane spins alone while the others wait on it.
// KIND 0: the two lists of the verify and SMC passes; 3: the SD final-token pass
// (kModeSDFinal), pairs of slots (2j, 2j+1) holding the target and draft chunk of one pair,
// pairs dealt round-robin over the blocks.
template <int DT, int KIND>
__device__ __noinline__ void tma_producer(const StreamParams& p, unsigned char* ring,
                                          uint64_t* full, uint64_t* empty,
                                          unsigned long long* tag, unsigned* n_done, int slot,
                                          bool active) {
    const long long row_bytes = (long long)p.R.V * Geo<DT>::kBytes;
    const uint32_t fb = smem_u32(&full[slot]), eb = smem_u32(&empty[slot]);
    const uint32_t tb = smem_u32(&tag[slot]);
    const uint32_t dst = smem_u32(ring + (size_t)slot * kChunkBytes);
    const uint64_t pol = l2_evict_first();
    uint32_t round = 0;
    bool done = !active;
    unsigned streak = 0;  // failed polls in a row, and when the streak began
    unsigned long long t_streak = 0;
    // This block's shares of the two lists and their order (smcsd_deal.h); lane `slot` walks
    // local chunks slot, slot + kRing, ...
    const uint32_t Bu = gridDim.x, bu = blockIdx.x;
    Deal d = deal_init(KIND == 0 ? p.n_precise : 0, KIND == 0 ? p.n_fast : 0, p.fper, Bu, bu,
                       (uint32_t)slot, kRing);
    const uint32_t Qb = deal_share(p.n_precise, Bu, bu);  // (KIND 3: pairs)
    auto local_item = [&]() -> long long {  // tag item of local chunk d.k, or -1
        if (KIND == 3) {  // final-pass pairs: local chunk k is half k & 1 of pair k >> 1
            const uint32_t jp = d.k >> 1;
            if (jp >= Qb) return -1;
            return (long long)((((jp * Bu + bu) << 1) | (d.k & 1u)) | kPreciseBit);
        }
        return deal_item(d);
    };
    bool moved = true;
    while (__any_sync(0xffffffffu, !done)) {
        // a pass in which no lane could refill its slot backs off briefly instead of spinning on
        // the issue slots the consumer warps of this sub-partition need
        if (!__any_sync(0xffffffffu, moved)) __nanosleep(200);
        moved = false;
        if (done) continue;
        long long it;
        if (round > 0 && !mbar_test_wait(eb, (round - 1) & 1u)) {
            if (streak++ == 0) {
                t_streak = global_ns();
                continue;
            }
            if ((streak & 1023u) != 0 || global_ns() - t_streak <= kWaitLimitNs) continue;
            raise_error(p.ws, kErrTimeout);
            it = -1;  // give the slot up below so that its consumers stop
        } else {
            streak = 0;
            it = local_item();
        }
        moved = true;
        if (it < 0) {
            atomicAdd(n_done, 1u);
            tag_store(tb, kTagDone, 0u);
            done = true;
            continue;
        }
        const ChunkRef c = KIND == 3 ? chunk_ref_sd_final(p, (uint32_t)it, true)
                                     : chunk_ref_two_list(p, (uint32_t)it);
        const long long off = (long long)c.chunk * kChunkBytes;
        const long long left = row_bytes - off;
        const uint32_t bytes = (uint32_t)(left < kChunkBytes ? left : kChunkBytes);
        const char* src = static_cast<const char*>(c.is_draft ? p.R.drf : p.R.tgt) +
                          c.row * row_bytes + off;
        const long long nrows = (long long)p.R.S * (c.is_draft ? p.R.K : p.R.K + 1);
        const bool sane = !c.valid ||
                          (check_ok(p.ws, c.s >= 0 && c.s < p.R.S, -101, it) &&
                           check_ok(p.ws, p.R.toff || (c.row >= 0 && c.row < nrows), -102, c.row) &&
                           check_ok(p.ws, left > 0 && (bytes & 15u) == 0, -103, left) &&
                           check_ok(p.ws, ((uintptr_t)src & 15u) == 0, -104,
                                    (long long)(uintptr_t)src));
        if (c.valid && sane) {
            mbar_arrive_expect_tx_relaxed(fb, bytes);
            bulk_load(dst, src, bytes, fb, pol);
        } else {
            mbar_arrive_relaxed(fb);
        }
        uint32_t word = (c.valid && sane) ? (uint32_t)it : 0xffffffffu;
        if (KIND == 0 && c.valid && sane && !(word & kPreciseBit))
            word = (uint32_t)(((long long)c.s * p.slots + c.slot) * p.cpr + c.chunk) |
                   (c.is_draft ? kFastDraftBit : 0u) | (c.chunk == p.cpr - 1 ? kFastTailBit : 0u);
        tag_store(tb, round * kRing + (uint32_t)slot, word);
        ++round;
        deal_advance(d, kRing);
    }
    // the copy of this lane's last chunk may still be in flight: wait for it before leaving
    if (round > 0) mbar_wait(fb, (round - 1) & 1u);
}

// The largest logit of a chunk in a slot (lane l reads its own block), on every lane, and whether
// a NaN is among them.
template <int DT>
__device__ __forceinline__ float slot_max(const SharedSrc<DT>& src, bool& nan) {
    float m = kNegInf;
    nan = false;
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
        const uint4 v = src.piece(i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (DT == 1) {
                const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
                m = fmaxf(m, fmaxf(a, b));
                nan |= (a != a) | (b != b);
            } else {
                const float a = __uint_as_float(w[j]);
                m = fmaxf(m, a);
                nan |= (a != a);
            }
        }
    }
    nan = __any_sync(0xffffffffu, nan);
    return warp_max(m);
}

// Reference exponent of a chunk whose largest logit is m (kNoMass for a chunk without mass);
// raises SMCSD_ERR_NONFINITE for NaN, +inf or a scaled logit above the supported range.
__device__ __forceinline__ int chunk_nref(float m, bool nan, const PreciseCtx& P, int lane) {
    const float cm = m * P.sc.c_hi;
    const bool ok = !nan && m > kNegInf && cm >= -kMaxScaledLogit && cm <= kMaxScaledLogit;
    if (ok) return floor_int(f_mul(m, P.sc.c2));
    const bool too_big = m > kNegInf && !(cm <= kMaxScaledLogit);
    if ((nan || too_big) && lane == 0) raise_error(P.ws, kErrNonfinite);
    return kNoMass;
}

// The four sums of one lane block of a (target, draft) chunk pair (see final_consumer), in units
// of 2^nt and 2^nd. With a direct bf16 table (exp(c z) itself in shared memory) and both
// exponents in its range, a table pass adds the entries of both rows on accumulators biased by
// 2^(n+2) (as table_pass does), the two halves of every word on separate accumulators, and a
// second pass adds, through the general weights, the positions outside the table's domain
// (pieces flagged by the first). Otherwise every position goes through precise_weight.
template <int DT>
__device__ __forceinline__ void pair_sums(const SharedSrc<DT>& src_t, const SharedSrc<DT>& src_d,
                                          int nt, int nd, float theta, const PreciseCtx& P,
                                          dd& st, dd& sd, dd& sa, dd& sb) {
    constexpr int PERP = 16 / Geo<DT>::kBytes;
    st = sd = sa = sb = dd{0.0f, 0.0f};
    if (!src_t.live()) return;
    unsigned rare = (1u << kLoads) - 1;  // pieces left to the per-position pass
    bool covered = false;                // whether the table pass took the in-domain positions
    if (DT == 1 && P.tab && P.direct && nt != kNoMass && nd != kNoMass && nt >= kDirectMinRef &&
        nt <= kDirectMaxRef && nd >= kDirectMinRef && nd <= kDirectMaxRef) {
        covered = true;
        const uint32_t tab = shared_addr(P.tab);
        const float bt = pow2i(nt + 2), bd = pow2i(nd + 2);
        dd t0{bt, 0.0f}, t1{bt, 0.0f}, a0{bt, 0.0f}, a1{bt, 0.0f};
        dd d0{bd, 0.0f}, d1{bd, 0.0f}, b0{bd, 0.0f}, b1{bd, 0.0f};
        unsigned pieces = 0;
#pragma unroll 1
        for (int i = 0; i < kLoads; ++i) {
            const uint4 vt = src_t.piece(i), vd = src_d.piece(i);
            const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
            uint32_t omax = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t ot, od;
                const uint32_t it = tab_index2(wt[j], ot), id = tab_index2(wd[j], od);
                asm("max.u16x2 %0, %1, %2;" : "=r"(omax) : "r"(omax), "r"(ot));
                asm("max.u16x2 %0, %1, %2;" : "=r"(omax) : "r"(omax), "r"(od));
                const float2 et0 = lds_f2(tab + (it & 0xffffu)), et1 = lds_f2(tab + (it >> 16));
                const float2 ed0 = lds_f2(tab + (id & 0xffffu)), ed1 = lds_f2(tab + (id >> 16));
                acc_biased(t0, dd{et0.x, et0.y});
                acc_biased(t1, dd{et1.x, et1.y});
                acc_biased(d0, dd{ed0.x, ed0.y});
                acc_biased(d1, dd{ed1.x, ed1.y});
                // p_i > q_i (a NaN difference, both masked, is not)
                const bool c0 = f_sub(bf16_lo(wt[j]), bf16_lo(wd[j])) > theta;
                const bool c1 = f_sub(bf16_hi(wt[j]), bf16_hi(wd[j])) > theta;
                // (predicated additions: adding an exact zero would leave the same bits)
                if (c0) {
                    acc_biased(a0, dd{et0.x, et0.y});
                    acc_biased(b0, dd{ed0.x, ed0.y});
                }
                if (c1) {
                    acc_biased(a1, dd{et1.x, et1.y});
                    acc_biased(b1, dd{ed1.x, ed1.y});
                }
            }
            if ((omax & 0xffffu) >= kTabHalf || (omax >> 16) >= kTabHalf) pieces |= 1u << i;
            t0 = fast_two_sum(t0.hi, t0.lo);
            t1 = fast_two_sum(t1.hi, t1.lo);
            d0 = fast_two_sum(d0.hi, d0.lo);
            d1 = fast_two_sum(d1.hi, d1.lo);
            a0 = fast_two_sum(a0.hi, a0.lo);
            a1 = fast_two_sum(a1.hi, a1.lo);
            b0 = fast_two_sum(b0.hi, b0.lo);
            b1 = fast_two_sum(b1.hi, b1.lo);
        }
        rare = pieces;
        const float ft = pow2i(-nt), fd = pow2i(-nd);
        auto fin = [](dd x, dd y, float bias, float f) {
            const dd v = dd_add(fast_two_sum(f_sub(x.hi, bias), x.lo), fast_two_sum(f_sub(y.hi, bias), y.lo));
            return dd{f_mul(v.hi, f), f_mul(v.lo, f)};
        };
        st = fin(t0, t1, bt, ft);
        sd = fin(d0, d1, bd, fd);
        sa = fin(a0, a1, bt, ft);
        sb = fin(b0, b1, bd, fd);
    }
    if (!rare) return;
    // positions the table pass did not take (all of them without it), through the general weights
    dd xt{kBias, 0.0f}, xd{kBias, 0.0f}, xa{kBias, 0.0f}, xb{kBias, 0.0f};
    do {
        const int i = __ffs(rare) - 1;
        rare &= rare - 1;
        const uint4 vt = src_t.piece(i), vd = src_d.piece(i);
        const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll 1
        for (int q = 0; q < PERP; ++q) {
            const uint32_t ut = DT == 1 ? ((q & 1) ? (wt[q >> 1] >> 16) : (wt[q >> 1] & 0xffffu)) : wt[q];
            const uint32_t ud = DT == 1 ? ((q & 1) ? (wd[q >> 1] >> 16) : (wd[q >> 1] & 0xffffu)) : wd[q];
            const bool in_t = covered && ((ut & 0x7fffu) - kTabMagLo) < kTabHalf;
            const bool in_d = covered && ((ud & 0x7fffu) - kTabMagLo) < kTabHalf;
            const dd et = (in_t || nt == kNoMass) ? dd{0.0f, 0.0f} : precise_weight<DT>(ut, nt, P);
            const dd ed = (in_d || nd == kNoMass) ? dd{0.0f, 0.0f} : precise_weight<DT>(ud, nd, P);
            acc_biased(xt, et);
            acc_biased(xd, ed);
            if (f_sub(bits_to_float<DT>(ut), bits_to_float<DT>(ud)) > theta) {
                acc_biased(xa, et);
                acc_biased(xb, ed);
            }
        }
        xt = fast_two_sum(xt.hi, xt.lo);
        xd = fast_two_sum(xd.hi, xd.lo);
        xa = fast_two_sum(xa.hi, xa.lo);
        xb = fast_two_sum(xb.hi, xb.lo);
    } while (rare);
    st = dd_add(st, unbias(xt));
    sd = dd_add(sd, unbias(xd));
    sa = dd_add(sa, unbias(xa));
    sb = dd_add(sb, unbias(xb));
}

// A consumer warp of the SD final-token pass: it claims both slots of a pair (target chunk in the
// even slot, draft chunk in the odd one). A sequence that accepted every draft has only the
// target half (its bonus row), whose precise partials go to ddtot/ddsub as in the SMC passes. For
// a sequence that rejected one, each lane sums over its block of the pair, in double-float
// units of 2^n_t and 2^n_d (each row's chunk exponent), S_t = sum exp(c z_t), S_d = sum exp(c z_d),
// A = the same over the positions with z_t - z_d > theta for the target row and B for the draft
// row: the row normalisers (S_t, S_d) and the residual's mass (A / Z_t - B / Z_d) then come from
// one read of the pair. Records: ddsub rows 2s and 2s+1 hold {S_t, A} and {S_d, B} per lane block,
// ddtot rows 2s and 2s+1 the chunk totals of S_t and S_d with their exponents, rtot {A, B} per
// chunk.
template <int DT>
__device__ __forceinline__ void final_consumer(const StreamParams& p, const PreciseCtx& P,
                                               unsigned char* ring, uint64_t* full, uint64_t* empty,
                                               unsigned long long* tag, unsigned* next,
                                               unsigned* n_done, int lane) {
    constexpr int SUB = Geo<DT>::kSub, PERP = 16 / Geo<DT>::kBytes;
    const SeqState* seq = ws_ptr<SeqState>(p.ws, p.L.seq);
    for (;;) {
        unsigned k = 0;
        if (lane == 0) k = atomicAdd(next, 2u);
        k = __shfl_sync(0xffffffffu, k, 0);
        const int slot0 = (int)(k % kRing), slot1 = slot0 + 1;
        unsigned long long seen0, seen1;
        if (!__all_sync(0xffffffffu, tag_wait(smem_u32(&tag[slot0]), k, seen0))) {
            if (lane == 0) raise_error(p.ws, kErrTimeout);
            break;
        }
        seen0 = __shfl_sync(0xffffffffu, seen0, 0);
        if ((uint32_t)(seen0 >> 32) == kTagDone) {
            unsigned nd = 0;
            if (lane == 0) nd = *reinterpret_cast<volatile unsigned*>(n_done);
            if (__shfl_sync(0xffffffffu, nd, 0) == (unsigned)kRing) break;
            continue;
        }
        if (!__all_sync(0xffffffffu, tag_wait(smem_u32(&tag[slot1]), k + 1, seen1))) {
            if (lane == 0) raise_error(p.ws, kErrTimeout);
            break;
        }
        seen1 = __shfl_sync(0xffffffffu, seen1, 0);
        const uint32_t item0 = (uint32_t)seen0, item1 = (uint32_t)seen1;  // 0xffffffff: not loaded
        ChunkRef c{};
        c.valid = false;
        if (item0 != 0xffffffffu) c = chunk_ref_sd_final(p, item0, false);
        int mode = 0;
        float theta = 0.0f;
        if (c.valid) {
            mode = __ldcg(&seq[c.s].mode);
            theta = __ldcg(&seq[c.s].theta);
        }
        const bool pair = c.valid && mode == 1 && item1 != 0xffffffffu;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[slot0]), (k / kRing) & 1u) &&
                                         mbar_wait(smem_u32(&full[slot1]), (k / kRing) & 1u))) {
            if (lane == 0) raise_error(p.ws, kErrTimeout);
            break;
        }
        bool wrote = false;
        if (c.valid) {
            const long long e0 = (long long)c.chunk * Geo<DT>::kChunk + (long long)lane * SUB;
            unsigned char* bt = ring + (size_t)slot0 * kChunkBytes + lane * 128;
            unsigned char* bd = ring + (size_t)slot1 * kChunkBytes + lane * 128;
            if (c.chunk == p.cpr - 1 && e0 + SUB > p.R.V) {
                // the rows end inside this block: the lane overwrites its logits past V with -inf
                // (the rest of the slots holds older chunks)
                for (int q = 0; q < SUB; ++q)
                    if (e0 + q >= p.R.V) {
                        if (DT == 1) {
                            reinterpret_cast<unsigned short*>(bt)[q] = 0xff80u;
                            reinterpret_cast<unsigned short*>(bd)[q] = 0xff80u;
                        } else {
                            reinterpret_cast<uint32_t*>(bt)[q] = 0xff800000u;
                            reinterpret_cast<uint32_t*>(bd)[q] = 0xff800000u;
                        }
                    }
                wrote = true;
            }
            const size_t prow = (size_t)c.s * 2;
            float4* tot_t = ws_ptr<float4>(p.ws, p.L.ddtot) + prow * p.cpr + c.chunk;
            float4* sub_t = ws_ptr<float4>(p.ws, p.L.ddsub) + (prow * p.cpr + c.chunk) * kSubs;
            const SharedSrc<DT> src_t{bt, lane & 7, e0 < p.R.V};
            if (!pair) {
                precise_core<DT>(src_t, src_t, lane, P, tot_t, sub_t);
            } else {
                const SharedSrc<DT> src_d{bd, lane & 7, e0 < p.R.V};
                bool nan_t, nan_d;
                const float mt = slot_max<DT>(src_t, nan_t), md = slot_max<DT>(src_d, nan_d);
                const int nt = chunk_nref(mt, nan_t, P, lane), nd = chunk_nref(md, nan_d, P, lane);
                dd vst, vsd, va, vb;
                pair_sums<DT>(src_t, src_d, nt, nd, theta, P, vst, vsd, va, vb);
                float4* sub_d = sub_t + (size_t)p.cpr * kSubs;
                sub_t[lane] = make_float4(vst.hi, vst.lo, va.hi, va.lo);
                sub_d[lane] = make_float4(vsd.hi, vsd.lo, vb.hi, vb.lo);
                const dd tst = warp_total_fixed(vst), tsd = warp_total_fixed(vsd);
                const dd ta = warp_total_fixed(va), tb = warp_total_fixed(vb);
                if (lane == 0) {
                    *tot_t = pack_part(tst, nt);
                    tot_t[p.cpr] = pack_part(tsd, nd);
                    ws_ptr<float4>(p.ws, p.L.rtot)[(size_t)c.s * p.cpr + c.chunk] =
                        make_float4(ta.hi, ta.lo, tb.hi, tb.lo);
                }
            }
            // stores into a slot must be ordered before the copy engine's next write to it
            if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        const bool any_wrote = __any_sync(0xffffffffu, wrote);
        __syncwarp();
        if (lane == 0) {
            if (any_wrote) {
                mbar_arrive(smem_u32(&empty[slot0]));
                mbar_arrive(smem_u32(&empty[slot1]));
            } else {
                mbar_arrive_relaxed(smem_u32(&empty[slot0]));
                mbar_arrive_relaxed(smem_u32(&empty[slot1]));
            }
        }
    }
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kTmaThreads, 1)
    stream_tma_kernel(const __grid_constant__ StreamParams p) {
    constexpr bool kPrecise = MODE != kModeSD;
    constexpr int kKind = MODE == kModeSDFinal ? 3 : 0;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    float2* sTab = reinterpret_cast<float2*>(smem + kSmemRing);
    Exp2Table* sT = reinterpret_cast<Exp2Table*>(smem + kSmemRing + kSmemTab);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemRing + kSmemTab + sizeof(Exp2Table));
    uint64_t* empty = full + kRing;
    unsigned long long* tag = reinterpret_cast<unsigned long long*>(empty + kRing);
    unsigned* next = reinterpret_cast<unsigned*>(tag + kRing);
    unsigned* n_done = next + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
            tag[i] = (unsigned long long)kTagNone << 32;
        }
        *next = 0;
        *n_done = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Launched as a programmatic dependent of the kernel before it on the stream (the previous
    // step's finishing pass, for instance): nothing global is read or written before that kernel
    // has completed and its writes are visible.
    griddep_wait();
    if (MODE == kModeSMCStep) zero_refcount(p);
    if (threadIdx.x == 0) griddep_launch_dependents();
    if (warp < kTmaProducers) {
        constexpr int kPer = kRing / kTmaProducers;
        tma_producer<DT, kKind>(p, ring, full, empty, tag, n_done, warp * kPer + (lane % kPer),
                                lane < kPer);
        return;
    }

    // consumers: tables first (while the producer already streams), then chunks
    const int tid = threadIdx.x - kTmaProducers * kWarp, nthr = kTmaConsumers * kWarp;
    for (int i = tid; i < 32; i += nthr) {
        sT->hi[i] = p.T.hi[i];
        sT->lo[i] = p.T.lo[i];
    }
    bar_sync(1, nthr);
    PreciseCtx P{p.sc_t, sT, nullptr, p.ws, p.direct};
    if (kPrecise && DT == 1 && p.use_table) {
        setup_exp_table(sTab, p.sc_t, sT, p.ws, ws_ptr<uint32_t>(p.ws, p.L.tab),
                        ws_ptr<float2>(p.ws, p.L.tab + 16), p.direct, tid, nthr, 1);
        P.tab = sTab;
    }
    if (MODE == kModeSDFinal) {
        final_consumer<DT>(p, P, ring, full, empty, tag, next, n_done, lane);
        return;
    }
    for (;;) {
        unsigned k = 0;
        if (lane == 0) k = atomicAdd(next, 1u);
        k = __shfl_sync(0xffffffffu, k, 0);
        const int slot = (int)(k % kRing);
        unsigned long long seen;
        if (!__all_sync(0xffffffffu, tag_wait(smem_u32(&tag[slot]), k, seen))) {
            if (lane == 0) raise_error(p.ws, kErrTimeout);
            break;
        }
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if ((uint32_t)(seen >> 32) == kTagDone) {
            // this slot has no more chunks; stop once no slot has any
            unsigned nd = 0;
            if (lane == 0) nd = *reinterpret_cast<volatile unsigned*>(n_done);
            if (__shfl_sync(0xffffffffu, nd, 0) == (unsigned)kRing) break;
            continue;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[slot]), (k / kRing) & 1u))) {
            if (lane == 0) raise_error(p.ws, kErrTimeout);
            break;
        }
        const uint32_t item = (uint32_t)seen;  // 0xffffffff: a chunk with nothing to load
        const unsigned char* cbuf = ring + (size_t)slot * kChunkBytes;
        if (item != 0xffffffffu && !(item & kPreciseBit)) {
            // a fast chunk, described by the producer (see fast_tag): its partial's index, whether
            // it is a draft row's and whether it is the row's last chunk
            const uint32_t fi = item & kFastIndexMask;
            const bool is_draft = (item & kFastDraftBit) != 0;
            check_ok(p.ws, (long long)fi < (long long)p.R.S * p.slots * p.cpr, -112, fi);
            {
                uint4 raw[kLoads];
#pragma unroll
                for (int v = 0; v < kLoads; ++v)
                    raw[v] = *reinterpret_cast<const uint4*>(cbuf + v * 512 + lane * 16);
                // the chunk now sits in registers: hand the slot back before the arithmetic, so
                // that the producer can refill it while this warp computes (the arrival follows
                // an instruction that consumed every loaded word, so the reads are complete)
                consume_all(raw);
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(smem_u32(&empty[slot]));
                if (item & kFastTailBit) {  // the row's last chunk: mask past V
                    const long long base = (long long)(p.cpr - 1) * Geo<DT>::kChunk + lane * Geo<DT>::kPerVec;
#pragma unroll
                    for (int v = 0; v < kLoads; ++v)
                        if (base + v * (Geo<DT>::kChunk / kLoads) >= p.R.V)
                            raw[v] = DT == 0 ? make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u)
                                             : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                }
                const float2 fp = fast_partial<DT>(raw, is_draft ? p.sc_d.c2 : p.sc_t.c2, p.ws);
                if (lane == 0) ws_ptr<float2>(p.ws, p.L.fast)[fi] = fp;
            }
            continue;
        }
        ChunkRef c{};
        c.valid = false;
        if (item != 0xffffffffu)
            c = chunk_ref_two_list(p, item);
        const int s = c.valid ? c.s : -1, rs = c.slot, chunk = c.chunk;
        const bool sane = s < 0 || (check_ok(p.ws, chunk >= 0 && chunk < p.cpr, -111, chunk) &&
                                    check_ok(p.ws, rs >= 0 && rs < p.slots, -112, rs));
        if (s >= 0 && sane) {
            {
                // a sampled row: lane l takes the contiguous block of kSub logits at l * 128
                // bytes, its pieces read with an XOR swizzle (piece v ^ (l & 7)) so that each
                // quarter-warp touches eight different bank groups; the slot goes back when the
                // partials are done
                constexpr int SUB = Geo<DT>::kSub;
                const long long e0 = (long long)chunk * Geo<DT>::kChunk + (long long)lane * SUB;
                unsigned char* blk = ring + (size_t)slot * kChunkBytes + lane * 128;
                const bool tail = chunk == p.cpr - 1;
                if (tail) {
                    // the row ends in this chunk: the lane overwrites its own logits past V with
                    // -inf (the rest of the slot holds an older chunk)
                    for (int q = 0; q < SUB; ++q)
                        if (e0 + q >= p.R.V) {
                            if (DT == 1) reinterpret_cast<unsigned short*>(blk)[q] = 0xff80u;
                            else reinterpret_cast<uint32_t*>(blk)[q] = 0xff800000u;
                        }
                }
                // the sampled row of sequence s (its bonus row) has its records at row 2s
                const size_t prow = (size_t)(s * 2);
                float4* tot = ws_ptr<float4>(p.ws, p.L.ddtot) + prow * p.cpr + chunk;
                float4* sub = ws_ptr<float4>(p.ws, p.L.ddsub) + (prow * p.cpr + chunk) * kSubs;
                const SharedSrc<DT> src{blk, lane & 7, e0 < p.R.V};
                precise_core<DT>(src, src, lane, P, tot, sub);
                // the stores above must be ordered before the copy engine's next write to the
                // slot: a proxy fence, and a releasing arrival
                if (tail) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if (tail) mbar_arrive(smem_u32(&empty[slot]));
                    else mbar_arrive_relaxed(smem_u32(&empty[slot]));
                }
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(smem_u32(&empty[slot]));
        }
    }
}

template <int DT, int MODE>
static cudaError_t launch_tma_t(const StreamParams& p0, cudaStream_t st) {
    auto kern = stream_tma_kernel<DT, MODE>;
    StreamParams p = p0;
    if (MODE == kModeSDFinal) {
        // (target, draft) chunk pairs of every sequence; n_precise counts pairs
        p.fslots = 0;
        p.fper = 0;
        p.n_precise = (long long)p.R.S * p.cpr;
        p.n_fast = 0;
        p.div_fseq = make_fastdiv(1u);
    } else {
        // the sampled rows (one per particle) form the precise list; in SD mode every row is fast
        const bool sampled = MODE != kModeSD;
        p.fslots = sampled ? (p.drf_logq ? p.R.K : p.slots - 1) : p.slots;
        p.n_precise = sampled ? (long long)p.R.S * p.cpr : 0;
        p.n_fast = (long long)p.R.S * p.fslots * p.cpr;
        p.div_fseq = make_fastdiv((uint32_t)(p.fslots > 0 ? p.fslots * p.cpr : 1));
        p.fper = sampled ? deal_fper(p.fslots) : p.fslots;
    }
    if ((long long)p.R.S * p.slots * p.cpr > (long long)kFastIndexMask) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long cap = device_sm_count();
    const long long units = (MODE == kModeSDFinal ? 2 : 1) * p.n_precise + p.n_fast;
    const long long want = (units + kTmaConsumers - 1) / kTmaConsumers;
    int grid = (int)(want < cap ? want : cap);
    if (grid < 1) grid = 1;
    // programmatic stream serialisation: the launch and the blocks' set-up overlap the tail of
    // the kernel before; the kernel's griddepcontrol.wait orders everything else after it
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kTmaThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
}

cudaError_t launch_wait_selftest(void* ws, unsigned long long limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(ws, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_stream_tma(const StreamParams& p, cudaStream_t st) {
    if (p.mode == kModeSDFinal)
        return p.dtype == 0 ? launch_tma_t<0, kModeSDFinal>(p, st) : launch_tma_t<1, kModeSDFinal>(p, st);
    if (p.dtype == 0) {
        if (p.mode == kModeSD) return launch_tma_t<0, kModeSD>(p, st);
        if (p.mode == kModeSMC) return launch_tma_t<0, kModeSMC>(p, st);
        return launch_tma_t<0, kModeSMCStep>(p, st);
    }
    if (p.mode == kModeSD) return launch_tma_t<1, kModeSD>(p, st);
    if (p.mode == kModeSMC) return launch_tma_t<1, kModeSMC>(p, st);
    return launch_tma_t<1, kModeSMCStep>(p, st);
}

}  // namespace smcsd
