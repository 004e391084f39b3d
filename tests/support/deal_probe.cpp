// Host build of the streaming pass's chunk dealing (smcsd_deal.h), for CPU tests of coverage.
#include "smcsd_deal.h"

// For every block b < B and local chunk k, the tag item the producer lane of slot k % ring loads
// (walking its slot's chunks as the kernel does); items[b * max_local + k], -2 past the block's
// last chunk. Returns the largest local count, or -1 if it exceeds max_local.
extern "C" int probe_deal(long long n_precise, long long n_fast, int fper, unsigned B, unsigned ring,
                          long long* items, int max_local) {
    int most = 0;
    for (unsigned b = 0; b < B; ++b) {
        for (int k = 0; k < max_local; ++k) items[(long long)b * max_local + k] = -2;
        for (unsigned j = 0; j < ring; ++j) {
            smcsd::Deal d = smcsd::deal_init(n_precise, n_fast, fper, B, b, j, ring);
            for (;;) {
                const long long it = smcsd::deal_item(d);
                if (it < 0) break;
                if ((int)d.k >= max_local) return -1;
                items[(long long)b * max_local + d.k] = it;
                if ((int)d.k + 1 > most) most = (int)d.k + 1;
                smcsd::deal_advance(d, ring);
            }
        }
    }
    return most;
}

extern "C" int probe_fper(int fslots) { return smcsd::deal_fper(fslots); }
