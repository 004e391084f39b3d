// smcsd_launch.cuh -- launch parameters of the kernels and the host-side launchers that the C ABI
// layer (api.cu) calls.
#pragma once

#include "smcsd_deal.h"
#include "smcsd_sampling.cuh"

namespace smcsd {

// kModeSDFinal: the SD final-token pass over (target, draft) chunk pairs: a sequence that drew
// all its drafts gets the precise partials of its bonus row, one that rejected one gets, per lane
// block of the pair, the sums of exp(c z_t) and exp(c z_d) over all positions and over the
// positions where z_t - z_d exceeds theta.
enum StreamMode { kModeSD = 0, kModeSMC = 1, kModeSMCStep = 2, kModeSDFinal = 5 };

// One streaming pass over all logits rows (SD first pass, SMC reweight, fused SMC step).
struct StreamParams {
    Rows R;
    int dtype;
    bool vec;        // 16-byte aligned rows: vector loads
    bool use_table;  // bf16 exp table for the sampled rows
    bool direct;     // the table holds exp(c z) itself
    int mode;
    Scale sc_t, sc_d;
    Exp2Table T;
    const float* uniforms;  // SD: [S*(K+1)]; SMC: bonus draws [S]
    // SD outputs
    int32_t* accept_len;
    float* lse_tgt;
    float* lse_drf;
    // SMC outputs
    float* logw;
    int32_t* bonus_token;
    // SMC tilted targets: whole-sequence power target (sc_t is then 1/T and draft-token log-
    // probabilities are weighted by alpha, the (K+1)-th token by alpha - 1), additive log-reward
    bool target_seq;
    float alpha;
    const float* log_reward;  // [S] or null
    float reward_scale;
    // log-probability of each particle's drawn (K+1)-th token at the target's scale, or null
    float* bonus_logq;
    // draft log-probabilities log q_k(x_k) given by the caller ([S*K], e.g. from the draft
    // sampler) in place of the draft logits: the draft rows are then neither streamed nor
    // normalised (SMC modes only)
    const float* drf_logq;
    // fused SMC step: per-group stage
    int G, N;
    float ess_threshold;
    const float* resample_uniforms;
    int32_t* ancestors;
    float* ess;
    int32_t* resampled;
    const int32_t* table_in;
    int32_t* table_out;
    int pages_per_seq;
    int32_t* refcount;
    int num_pages;
    // scratch
    void* ws;
    WsLayout L;
    int cpr, slots;
    long long items;       // chunks in the sequence-major order (< 2^31)
    FastDiv div_seq;       // by slots * cpr (chunks per sequence)
    FastDiv div_cpr;       // by cpr (chunks per row)
    // two-list dealing of the pipelined pass (set by its launcher): the precise chunks (rows that
    // are sampled) and the fast chunks (all other rows, fslots per sequence) as separate lists
    long long n_precise, n_fast;
    int fslots;
    int fper;              // fast chunks paired with each precise chunk (smcsd_deal.h)
    FastDiv div_fseq;      // by fslots * cpr
};

// SD second and third passes (precise sums of the rows to draw from, the residual draw).
struct SampleParams {
    Rows R;
    int dtype;
    bool vec;
    bool use_table;
    bool direct;
    Scale sc;
    Exp2Table T;
    const float* uniforms;
    int32_t* out_token;
    void* ws;
    WsLayout L;
    int cpr;
};

struct ResampleParams {
    float* logw;
    int G, N;
    float ess_threshold;
    const float* uniforms;
    int32_t* ancestors;
    float* ess;
    int32_t* resampled;
    void* ws;
    Exp2Table T;
};

struct RemapParams {
    const int32_t* ancestors;
    const int32_t* resampled;
    int G, N;
    const int32_t* table_in;
    int32_t* table_out;
    int pages_per_seq;
    int32_t* refcount;
    int num_pages;
    void* ws;
};

struct PacerParams {
    const uint16_t* hidden;
    const uint16_t* w;
    const uint16_t* pos_emb;  // [max_blocks*b, d] or null
    float c;
    int S, b, max_blocks, d;
    float t0, rho;
    bool vec;
    int32_t* lengths;
    float* block_scores;
    int32_t* tgt_offsets;
    int32_t* drf_offsets;
    void* ws;
    WsLayout L;
};

cudaError_t launch_stream(const StreamParams& p, cudaStream_t st);      // both passes
cudaError_t launch_finish(const StreamParams& p, cudaStream_t st);      // finishing pass
cudaError_t launch_stream_tma(const StreamParams& p, cudaStream_t st);  // aligned rows
cudaError_t launch_sd_sample(const SampleParams& p, cudaStream_t st);
cudaError_t launch_resample(const ResampleParams& p, cudaStream_t st);
cudaError_t launch_remap(const RemapParams& p, cudaStream_t st);
cudaError_t launch_pacer(const PacerParams& p, cudaStream_t st);
cudaError_t launch_wait_selftest(void* ws, unsigned long long limit_ns, cudaStream_t st);

int device_sm_count();

}  // namespace smcsd
