// resample_pacer.cu -- the stand-alone resampling, page-table and stop-rule kernels:
//   resample_kernel: effective sample size and systematic resampling, one warp per group
//     ("Faster LLM Inference via Sequential Monte Carlo", sec. 2 step 4);
//   remap_kernel: child rows of the paged-KV page table copied from their ancestors' rows, and
//     the page reference counts rebuilt (same page, sec. 3: a metadata update, no KV movement);
//   pacer_kernel: the PACER blockwise stop rule ("PACER: Blockwise Pre-verification for
//     Speculative Decoding with Adaptive Length", Methodik 1-3), one block per sequence, reading
//     hidden states (and position embeddings, Methodik 1) only up to the block that stops; the
//     last block to finish writes the ragged row offsets for the verify that follows.
#include "smcsd_launch.cuh"

namespace smcsd {

__global__ void __launch_bounds__(128) resample_kernel(const __grid_constant__ ResampleParams p) {
    // the exp table in shared memory: lanes index it at different entries
    __shared__ Exp2Table sT;
    for (int i = threadIdx.x; i < 32; i += blockDim.x) {
        sT.hi[i] = p.T.hi[i];
        sT.lo[i] = p.T.lo[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (g >= p.G) return;
    const size_t o = (size_t)g * p.N;
    group_resample(p.logw + o, p.N, p.ess_threshold, __ldg(p.uniforms + g), p.ancestors + o,
                   p.ess ? p.ess + g : nullptr, p.resampled ? p.resampled + g : nullptr, p.ws, lane,
                   sT);
}

__global__ void __launch_bounds__(256) remap_kernel(const __grid_constant__ RemapParams p) {
    const int P = p.pages_per_seq, N = p.N;
    const long long total = (long long)p.G * N * P;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / P;
        const int col = (int)(i - row * P);
        const int g = (int)(row / N), j = (int)(row - (long long)g * N);
        const bool moved = p.resampled ? __ldg(p.resampled + g) != 0 : true;
        const int a = moved ? __ldg(p.ancestors + row) : j;
        if (a < 0 || a >= N) {
            raise_error(p.ws, kErrRange);
            continue;
        }
        const int32_t id = __ldg(p.table_in + ((long long)g * N + a) * P + col);
        p.table_out[i] = id;
        if (p.refcount && id != -1) {
            if (id < 0 || id >= p.num_pages)
                raise_error(p.ws, kErrRange);
            else
                atomicAdd(p.refcount + id, 1);
        }
    }
}

constexpr int kPacerThreads = 128;
constexpr int kPacerMaxB = 64;

__global__ void __launch_bounds__(kPacerThreads) pacer_kernel(const __grid_constant__ PacerParams p) {
    __shared__ double score[kPacerMaxB];
    __shared__ int stop;
    __shared__ unsigned last;
    const int s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int P = p.max_blocks * p.b;
    double t = (double)p.t0;
    int len = P;
    int i = 0;
    for (; i < p.max_blocks; ++i) {
        for (int j = warp; j < p.b; j += nw) {
            const size_t pos = (size_t)i * p.b + j;  // draft position within the sequence
            const uint16_t* h = p.hidden + ((size_t)s * P + pos) * p.d;
            // w . (h + e) as w . h + w . e: each bf16 x bf16 product is exact in float
            const uint16_t* pe = p.pos_emb ? p.pos_emb + pos * p.d : nullptr;
            dd acc{0.0f, 0.0f};
            if (p.vec) {
                for (int e = lane * 8; e < p.d; e += 256) {
                    const uint4 hv = __ldg(reinterpret_cast<const uint4*>(h + e));
                    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.w + e));
                    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
                    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc = dd_add(acc, dd{f_mul(bf16_lo(hw[q]), bf16_lo(ww[q])), 0.0f});
                        acc = dd_add(acc, dd{f_mul(bf16_hi(hw[q]), bf16_hi(ww[q])), 0.0f});
                    }
                    if (pe) {
                        const uint4 ev = __ldg(reinterpret_cast<const uint4*>(pe + e));
                        const uint32_t ew[4] = {ev.x, ev.y, ev.z, ev.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            acc = dd_add(acc, dd{f_mul(bf16_lo(ew[q]), bf16_lo(ww[q])), 0.0f});
                            acc = dd_add(acc, dd{f_mul(bf16_hi(ew[q]), bf16_hi(ww[q])), 0.0f});
                        }
                    }
                }
            } else {
                for (int e = lane; e < p.d; e += 32) {
                    const float hv = __uint_as_float(((uint32_t)__ldg(h + e)) << 16);
                    const float wv = __uint_as_float(((uint32_t)__ldg(p.w + e)) << 16);
                    acc = dd_add(acc, dd{f_mul(hv, wv), 0.0f});
                    if (pe) {
                        const float ev = __uint_as_float(((uint32_t)__ldg(pe + e)) << 16);
                        acc = dd_add(acc, dd{f_mul(ev, wv), 0.0f});
                    }
                }
            }
            const dd dot = warp_sum_dd(acc);
            if (lane == 0) {
                const double a = dd_to_double(dot) + (double)p.c;
                if (a != a) raise_error(p.ws, kErrNonfinite);
                score[j] = 1.0 / (1.0 + exp(-a));
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            double m = 0.0;
            for (int j = 0; j < p.b; ++j) m += score[j];
            m /= (double)p.b;
            if (p.block_scores) p.block_scores[(size_t)s * p.max_blocks + i] = (float)m;
            stop = m < t;
            if (!stop) t *= (double)p.rho;
        }
        __syncthreads();
        if (stop) {
            len = (i + 1) * p.b;
            ++i;
            break;
        }
    }
    if (threadIdx.x == 0) {
        p.lengths[s] = len;
        if (p.block_scores)
            for (int r = i; r < p.max_blocks; ++r) p.block_scores[(size_t)s * p.max_blocks + r] = -1.0f;
    }
    if (!p.tgt_offsets) return;
    // the last block to finish writes the offsets: prefix sums of length+1 and length
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned* cnt = ws_ptr<unsigned>(p.ws, p.L.cnt_misc);
        const unsigned old = atomicAdd(cnt, 1u);
        last = (old == (unsigned)p.S - 1);
        if (last) {
            atomicExch(cnt, 0u);
            __threadfence();
        }
    }
    __syncthreads();
    if (!last) return;
    if (warp != 0) return;
    // one warp: contiguous blocks of sequences per lane
    const int per = (p.S + 31) / 32;
    const int s0 = min(lane * per, p.S), s1 = min(s0 + per, p.S);
    int loc = 0;
    for (int q = s0; q < s1; ++q) loc += __ldcg(p.lengths + q);
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - loc;  // drafts before this lane's block
    if (lane == 0) {
        p.tgt_offsets[0] = 0;
        p.drf_offsets[0] = 0;
    }
    for (int q = s0; q < s1; ++q) {
        run += __ldcg(p.lengths + q);
        p.drf_offsets[q + 1] = run;
        p.tgt_offsets[q + 1] = run + (q + 1);
    }
}

cudaError_t launch_resample(const ResampleParams& p, cudaStream_t st) {
    const int wpb = 4;
    resample_kernel<<<(p.G + wpb - 1) / wpb, wpb * 32, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_remap(const RemapParams& p, cudaStream_t st) {
    const long long total = (long long)p.G * p.N * p.pages_per_seq;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    remap_kernel<<<(int)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pacer(const PacerParams& p, cudaStream_t st) {
    pacer_kernel<<<p.S, kPacerThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace smcsd
