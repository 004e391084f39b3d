// smcsd_deal.h -- how the streaming pass deals its chunks to the blocks (host and device code, so
// that the host tests can enumerate the dealing of every block).
//
// Two lists, each dealt round-robin over the B blocks: the precise list (chunks of the rows that
// are sampled, item i = chunk i % cpr of sampled row i / cpr) and the fast list (all other rows).
// Block b holds items b, b + B, b + 2B, ... of the precise list (Pb of them) and items B-1-b,
// 2B-1-b, ... of the fast list (Fb of them; reverse order, so that the blocks left with one precise
// chunk more get no extra fast chunk). Its local chunk sequence k = 0, 1, 2, ... is
//   phase 0: the E = Pb - G1 precise chunks the fast ones cannot pair up,
//   phase 1: G1 groups of one precise chunk and `fper` fast ones (L1 = G1 (fper + 1) chunks),
//   phase 2: the fast chunks left over,
// so that a block ends on cheap chunks; with fper below the number of fast rows per sampled row,
// the precise chunks run out before the fast ones do and the last part of the pass is fast chunks
// only. The producer lane of ring slot j walks k = j, j + R, j + 2R, ...; it tracks
// k1 = k - E = q (fper + 1) + r incrementally once k1 >= 0, in 32-bit arithmetic (every index is
// below 2^31), so a refill costs no division.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define SMCSD_DEAL_HD __host__ __device__ inline
#else
#define SMCSD_DEAL_HD inline
#endif

namespace smcsd {

constexpr uint32_t kPreciseBit = 0x80000000u;  // tag item of a precise chunk

// Number of items of a list of n dealt round-robin to block `pos` of B.
SMCSD_DEAL_HD uint32_t deal_share(long long n, uint32_t B, uint32_t pos) {
    return n > (long long)pos ? (uint32_t)((n - 1 - (long long)pos) / B) + 1u : 0u;
}

struct Deal {
    uint32_t B, b, bf, m, fper, Pb, Fb, G1, E, L1, dq, dr;
    uint32_t k, q, r;  // local chunk number and k - E = q m + r (once k >= E)
};

SMCSD_DEAL_HD Deal deal_init(long long n_precise, long long n_fast, int fper, uint32_t B,
                               uint32_t b, uint32_t first_k, uint32_t ring) {
    Deal d;
    d.B = B;
    d.b = b;
    d.bf = B - 1u - b;
    d.fper = (uint32_t)(fper > 0 ? fper : 0);
    d.m = d.fper + 1u;
    d.Pb = deal_share(n_precise, B, b);
    d.Fb = deal_share(n_fast, B, d.bf);
    const uint32_t fg = d.fper > 0 ? d.Fb / d.fper : 0u;
    d.G1 = d.fper > 0 ? (d.Pb < fg ? d.Pb : fg) : 0u;
    d.E = d.Pb - d.G1;
    d.L1 = d.G1 * d.m;
    d.dq = ring / d.m;
    d.dr = ring % d.m;
    d.k = first_k;
    d.q = d.r = 0;
    if (d.k >= d.E) {
        d.q = (d.k - d.E) / d.m;
        d.r = (d.k - d.E) % d.m;
    }
    return d;
}

// Tag item of local chunk d.k: a precise item (kPreciseBit set) or a fast item; -1 when the block
// has no chunk d.k.
SMCSD_DEAL_HD long long deal_item(const Deal& d) {
    uint32_t j;
    bool precise;
    if (d.k < d.E) {
        precise = true;
        j = d.k;
    } else if (d.k - d.E < d.L1) {
        precise = d.r == 0;
        j = precise ? d.E + d.q : d.q * d.fper + d.r - 1u;
    } else {
        precise = false;
        j = d.G1 * d.fper + (d.k - d.E - d.L1);
        if (j >= d.Fb) return -1;
    }
    return precise ? (long long)((j * d.B + d.b) | kPreciseBit) : (long long)(j * d.B + d.bf);
}

// Moves to local chunk d.k + ring.
SMCSD_DEAL_HD void deal_advance(Deal& d, uint32_t ring) {
    if (d.k >= d.E) {
        d.q += d.dq;
        d.r += d.dr;
        if (d.r >= d.m) {
            d.r -= d.m;
            ++d.q;
        }
    } else if (d.k + ring >= d.E) {  // k1 turns non-negative: one division
        d.q = (d.k + ring - d.E) / d.m;
        d.r = (d.k + ring - d.E) % d.m;
    }
    d.k += ring;
}

// Fast chunks paired with each precise chunk in phase 1, for `fslots` fast rows per sampled row:
// three quarters of them (at least one), so that the precise chunks are used up about a fifth of
// the way before the end of the pass.
SMCSD_DEAL_HD int deal_fper(int fslots) { return fslots > 0 ? (fslots * 3 / 4 > 0 ? fslots * 3 / 4 : 1) : 0; }

}  // namespace smcsd
