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
