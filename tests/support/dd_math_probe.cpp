// Host build of the CUDA library's double-float exponential, for CPU accuracy tests.
#include "smcsd_math.cuh"

extern "C" void probe_exp_split(const float* xh, const float* xl, int n, float* hi, float* lo, int* e) {
    smcsd::Exp2Table T = smcsd::make_exp2_table();
    for (int i = 0; i < n; ++i) {
        smcsd::ddx r = smcsd::exp_split(smcsd::dd{xh[i], xl[i]}, T);
        hi[i] = r.hi;
        lo[i] = r.lo;
        e[i] = r.n;
    }
}

extern "C" void probe_dd_recip(const float* ah, const float* al, int n, float* rh, float* rl) {
    for (int i = 0; i < n; ++i) {
        smcsd::dd r = smcsd::dd_recip(smcsd::dd{ah[i], al[i]});
        rh[i] = r.hi;
        rl[i] = r.lo;
    }
}

extern "C" void probe_dd_div(const float* ah, const float* al, const float* bh, const float* bl, int n,
                             float* qh, float* ql) {
    for (int i = 0; i < n; ++i) {
        smcsd::dd q = smcsd::dd_div(smcsd::dd{ah[i], al[i]}, smcsd::dd{bh[i], bl[i]});
        qh[i] = q.hi;
        ql[i] = q.lo;
    }
}

#include "smcsd_fastdiv.h"

// q = n / d through the launch-invariant division, for n in [0, count).
extern "C" int probe_fast_div_check(unsigned d, unsigned start, unsigned count, unsigned stride) {
    const smcsd::FastDiv f = smcsd::make_fastdiv(d);
    for (unsigned i = 0; i < count; ++i) {
        const unsigned n = start + i * stride;
        if (smcsd::fast_div(n, f) != n / d) return (int)i + 1;
    }
    return 0;
}
