// api.cu -- the C ABI declared in include/smcsd.h: host-side argument validation, workspace
// sizing and kernel launches. No allocation, no state kept between calls.
#include <math.h>
#include <stdint.h>

#include "smcsd.h"
#include "smcsd_launch.cuh"

using namespace smcsd;

namespace {

Scale make_scale(double c) {
    Scale s;
    s.c = c;
    s.c_hi = (float)c;
    s.c_lo = (float)(c - (double)s.c_hi);
    s.c2 = (float)(c * 1.4426950408889634074);
    return s;
}

const Exp2Table& exp2_table() {
    static const Exp2Table T = make_exp2_table();
    return T;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool finite_pos(float v) { return v > 0.0f && isfinite(v); }
int from_cuda(cudaError_t e) { return e == cudaSuccess ? SMCSD_OK : SMCSD_ERR_CUDA; }

int check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (!ws) return SMCSD_ERR_INVALID_ARG;
    if (((uintptr_t)ws & 255u) != 0 || ws_bytes < need) return SMCSD_ERR_WORKSPACE;
    return SMCSD_OK;
}

int elem_bytes(int dtype) { return dtype == SMCSD_F32 ? 4 : 2; }

}  // namespace

extern "C" size_t smcsd_workspace_size(int op, int S, int K, int V) {
    if (S <= 0) return 0;
    switch (op) {
        case SMCSD_OP_SD_VERIFY:
        case SMCSD_OP_SMC_REWEIGHT:
        case SMCSD_OP_SMC_STEP:
            if (K < 0 || V <= 0) return 0;
            return ws_layout(S, K, V).total;
        case SMCSD_OP_DRAFT_SAMPLE:
            if (V <= 0) return 0;
            return ws_layout(S, 0, V).total;
        case SMCSD_OP_ESS_RESAMPLE:
        case SMCSD_OP_PAGETABLE_REMAP:
        case SMCSD_OP_PACER_BLOCK_STOP:
            return ws_small_bytes(S);
        default:
            return 0;
    }
}

extern "C" int smcsd_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes == 0) return SMCSD_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

extern "C" int smcsd_check_status(void* ws, void* stream) {
    if (!ws) return SMCSD_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SMCSD_ERR_CUDA;
    int flag = 0;
    if (cudaMemcpy(&flag, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SMCSD_ERR_CUDA;
    if (flag != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return SMCSD_ERR_CUDA;
    return flag;
}

extern "C" int smcsd_selftest_wait(unsigned int limit_us, void* ws, size_t ws_bytes, void* stream) {
    if (limit_us == 0 || limit_us > 2000000u) return SMCSD_ERR_INVALID_ARG;
    int rc = check_ws(ws, ws_bytes, sizeof(int));
    if (rc) return rc;
    return from_cuda(launch_wait_selftest(ws, 1000ull * limit_us, (cudaStream_t)stream));
}

extern "C" const char* smcsd_status_string(int code) {
    switch (code) {
        case SMCSD_OK: return "ok";
        case SMCSD_ERR_INVALID_ARG: return "invalid argument";
        case SMCSD_ERR_DTYPE: return "unsupported dtype";
        case SMCSD_ERR_WORKSPACE: return "workspace too small or misaligned";
        case SMCSD_ERR_CUDA: return "CUDA launch or runtime error";
        case SMCSD_ERR_NONFINITE: return "non-finite input (NaN/+inf logit or weight, or an all-masked row)";
        case SMCSD_ERR_RANGE: return "index out of range (token id, offsets, ancestor or page id)";
        case SMCSD_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        default: return "unknown status";
    }
}

extern "C" int sd_verify(const void* tgt_logits, const void* drf_logits, int dtype,
                         const int32_t* draft_tokens, const int32_t* tgt_offsets,
                         const int32_t* drf_offsets, int S, int K, int V, float temperature,
                         const float* uniforms, int32_t* accept_len, int32_t* out_token,
                         float* lse_tgt, float* lse_drf, void* ws, size_t ws_bytes, void* stream) {
    if (dtype != SMCSD_F32 && dtype != SMCSD_BF16) return SMCSD_ERR_DTYPE;
    if (!tgt_logits || !uniforms || !accept_len || !out_token) return SMCSD_ERR_INVALID_ARG;
    if (S <= 0 || K < 0 || V <= 0 || !finite_pos(temperature)) return SMCSD_ERR_INVALID_ARG;
    if (K > 0 && (!drf_logits || !draft_tokens)) return SMCSD_ERR_INVALID_ARG;
    if ((tgt_offsets == nullptr) != (drf_offsets == nullptr)) return SMCSD_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(S, K, V);
    int rc = check_ws(ws, ws_bytes, L.total);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;

    StreamParams p{};
    p.R = Rows{tgt_logits, drf_logits, draft_tokens, tgt_offsets, drf_offsets, S, K, V};
    p.dtype = dtype;
    p.vec = aligned16(tgt_logits) && (K == 0 || aligned16(drf_logits)) &&
            ((size_t)V * elem_bytes(dtype)) % 16 == 0;
    p.mode = kModeSD;
    p.sc_t = p.sc_d = make_scale(1.0 / (double)temperature);
    p.use_table = dtype == SMCSD_BF16 && p.sc_t.c <= kTabMaxScale;
    p.direct = p.use_table && p.sc_t.c <= kDirectMaxScale;
    p.T = exp2_table();
    p.uniforms = uniforms;
    p.accept_len = accept_len;
    p.lse_tgt = lse_tgt;
    p.lse_drf = lse_drf;
    p.ws = ws;
    p.L = L;
    p.cpr = chunks_per_row(V, dtype);
    p.slots = 2 * K + 1;
    if (p.slots >= (1 << 15)) p.vec = false;  // the pipelined pass packs row slot and draft count in 16 bits each
    p.items = (long long)S * p.slots * p.cpr;
    if (p.items >= (1ll << 31)) return SMCSD_ERR_INVALID_ARG;
    p.div_seq = make_fastdiv((uint32_t)(p.slots * p.cpr));
    p.div_cpr = make_fastdiv((uint32_t)p.cpr);
    cudaError_t e = launch_stream(p, st);
    if (e != cudaSuccess) return SMCSD_ERR_CUDA;

    SampleParams q{};
    q.R = p.R;
    q.dtype = dtype;
    q.vec = p.vec;
    q.use_table = p.use_table;
    q.direct = p.direct;
    q.sc = p.sc_t;
    q.T = p.T;
    q.uniforms = uniforms;
    q.out_token = out_token;
    q.ws = ws;
    q.L = L;
    q.cpr = p.cpr;
    return from_cuda(launch_sd_sample(q, st));
}

static int smc_common(const void* tgt_logits, const void* drf_logits, int dtype,
                      const int32_t* draft_tokens, int S, int K, int V, float temperature,
                      float alpha, int target, const float* log_reward, float reward_scale,
                      const float* uniforms, float* logw, int32_t* bonus_token,
                      void* ws, size_t ws_bytes, StreamParams& p,
                      const float* drf_logq = nullptr) {
    if (dtype != SMCSD_F32 && dtype != SMCSD_BF16) return SMCSD_ERR_DTYPE;
    if (!tgt_logits || !uniforms || !bonus_token) return SMCSD_ERR_INVALID_ARG;
    if (S <= 0 || K < 0 || V <= 0) return SMCSD_ERR_INVALID_ARG;
    if (!finite_pos(temperature) || !finite_pos(alpha)) return SMCSD_ERR_INVALID_ARG;
    if (target != SMCSD_TARGET_TOKEN && target != SMCSD_TARGET_SEQUENCE) return SMCSD_ERR_INVALID_ARG;
    if (log_reward && !isfinite(reward_scale)) return SMCSD_ERR_INVALID_ARG;
    if (K > 0 && ((!drf_logits && !drf_logq) || !draft_tokens)) return SMCSD_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(S, K, V);
    int rc = check_ws(ws, ws_bytes, L.total);
    if (rc) return rc;
    if (drf_logq) drf_logits = nullptr;  // the draft rows are not read
    p.R = Rows{tgt_logits, drf_logits, draft_tokens, nullptr, nullptr, S, K, V};
    p.drf_logq = K > 0 ? drf_logq : nullptr;
    p.dtype = dtype;
    p.vec = aligned16(tgt_logits) && (K == 0 || aligned16(drf_logits)) &&
            ((size_t)V * elem_bytes(dtype)) % 16 == 0;
    // per-position target: pi = softmax(alpha z / T); whole sequence: p = softmax(z / T), with
    // alpha applied to the log-probabilities in the weight
    p.target_seq = target == SMCSD_TARGET_SEQUENCE;
    p.alpha = alpha;
    p.log_reward = log_reward;
    p.reward_scale = reward_scale;
    p.sc_t = make_scale((p.target_seq ? 1.0 : (double)alpha) / (double)temperature);
    p.sc_d = make_scale(1.0 / (double)temperature);
    p.use_table = dtype == SMCSD_BF16 && p.sc_t.c <= kTabMaxScale;
    p.direct = p.use_table && p.sc_t.c <= kDirectMaxScale;
    p.T = exp2_table();
    p.uniforms = uniforms;
    p.logw = logw;
    p.bonus_token = bonus_token;
    p.ws = ws;
    p.L = L;
    p.cpr = chunks_per_row(V, dtype);
    p.slots = 2 * K + 1;
    if (p.slots >= (1 << 15)) p.vec = false;  // the pipelined pass packs row slot and draft count in 16 bits each
    p.items = (long long)S * p.slots * p.cpr;
    if (p.items >= (1ll << 31)) return SMCSD_ERR_INVALID_ARG;
    p.div_seq = make_fastdiv((uint32_t)(p.slots * p.cpr));
    p.div_cpr = make_fastdiv((uint32_t)p.cpr);
    return SMCSD_OK;
}

extern "C" int smc_reweight_tilted(const void* tgt_logits, const void* drf_logits, int dtype,
                                   const int32_t* draft_tokens, int S, int K, int V,
                                   float temperature, float alpha, int target,
                                   const float* log_reward, float reward_scale,
                                   const float* uniforms, float* logw, int32_t* bonus_token,
                                   float* lse_tgt, float* lse_drf, void* ws, size_t ws_bytes,
                                   void* stream) {
    if (!logw) return SMCSD_ERR_INVALID_ARG;
    StreamParams p{};
    int rc = smc_common(tgt_logits, drf_logits, dtype, draft_tokens, S, K, V, temperature, alpha,
                        target, log_reward, reward_scale, uniforms, logw, bonus_token, ws,
                        ws_bytes, p);
    if (rc) return rc;
    p.mode = kModeSMC;
    p.lse_tgt = lse_tgt;
    p.lse_drf = lse_drf;
    return from_cuda(launch_stream(p, (cudaStream_t)stream));
}

extern "C" int smc_reweight(const void* tgt_logits, const void* drf_logits, int dtype,
                            const int32_t* draft_tokens, int S, int K, int V, float temperature,
                            float alpha, const float* uniforms, float* logw, int32_t* bonus_token,
                            float* lse_tgt, float* lse_drf, void* ws, size_t ws_bytes,
                            void* stream) {
    return smc_reweight_tilted(tgt_logits, drf_logits, dtype, draft_tokens, S, K, V, temperature,
                               alpha, SMCSD_TARGET_TOKEN, nullptr, 0.0f, uniforms, logw,
                               bonus_token, lse_tgt, lse_drf, ws, ws_bytes, stream);
}

static int smc_step_impl(const void* tgt_logits, const void* drf_logits, const float* drf_logq,
                         int dtype, const int32_t* draft_tokens, int G, int N, int K, int V,
                         float temperature, float alpha, int target, const float* log_reward,
                         float reward_scale, const float* bonus_uniforms, float* logw,
                         int32_t* bonus_token, float ess_threshold, const float* resample_uniforms,
                         int32_t* ancestors, float* ess, int32_t* resampled,
                         const int32_t* table_in, int32_t* table_out, int pages_per_seq,
                         int32_t* refcount, int num_pages, void* ws, size_t ws_bytes,
                         void* stream) {
    if (G <= 0 || N <= 0 || (long long)G * N > 0x7fffffffLL) return SMCSD_ERR_INVALID_ARG;
    if (!logw || !resample_uniforms || !ancestors || isnan(ess_threshold)) return SMCSD_ERR_INVALID_ARG;
    const bool remap = table_in != nullptr;
    if (remap) {
        if (!table_out || table_out == table_in || pages_per_seq <= 0) return SMCSD_ERR_INVALID_ARG;
        if (refcount && num_pages <= 0) return SMCSD_ERR_INVALID_ARG;
    } else if (table_out || refcount) {
        return SMCSD_ERR_INVALID_ARG;
    }
    StreamParams p{};
    int rc = smc_common(tgt_logits, drf_logits, dtype, draft_tokens, G * N, K, V, temperature,
                        alpha, target, log_reward, reward_scale, bonus_uniforms, logw,
                        bonus_token, ws, ws_bytes, p, drf_logq);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    p.mode = kModeSMCStep;
    p.G = G;
    p.N = N;
    p.ess_threshold = ess_threshold;
    p.resample_uniforms = resample_uniforms;
    p.ancestors = ancestors;
    p.ess = ess;
    p.resampled = resampled;
    p.table_in = table_in;
    p.table_out = table_out;
    p.pages_per_seq = pages_per_seq;
    p.refcount = remap ? refcount : nullptr;  // zeroed by the streaming pass
    p.num_pages = num_pages;
    return from_cuda(launch_stream(p, st));
}

extern "C" int smc_step_tilted(const void* tgt_logits, const void* drf_logits, int dtype,
                               const int32_t* draft_tokens, int G, int N, int K, int V,
                               float temperature, float alpha, int target,
                               const float* log_reward, float reward_scale,
                               const float* bonus_uniforms, float* logw, int32_t* bonus_token,
                               float ess_threshold, const float* resample_uniforms,
                               int32_t* ancestors, float* ess, int32_t* resampled,
                               const int32_t* table_in, int32_t* table_out, int pages_per_seq,
                               int32_t* refcount, int num_pages, void* ws, size_t ws_bytes,
                               void* stream) {
    return smc_step_impl(tgt_logits, drf_logits, nullptr, dtype, draft_tokens, G, N, K, V,
                         temperature, alpha, target, log_reward, reward_scale, bonus_uniforms,
                         logw, bonus_token, ess_threshold, resample_uniforms, ancestors, ess,
                         resampled, table_in, table_out, pages_per_seq, refcount, num_pages, ws,
                         ws_bytes, stream);
}

extern "C" int smc_step_logq(const void* tgt_logits, int dtype, const int32_t* draft_tokens,
                             const float* drf_logq, int G, int N, int K, int V, float temperature,
                             float alpha, const float* bonus_uniforms, float* logw,
                             int32_t* bonus_token, float ess_threshold,
                             const float* resample_uniforms, int32_t* ancestors, float* ess,
                             int32_t* resampled, const int32_t* table_in, int32_t* table_out,
                             int pages_per_seq, int32_t* refcount, int num_pages, void* ws,
                             size_t ws_bytes, void* stream) {
    if (K > 0 && !drf_logq) return SMCSD_ERR_INVALID_ARG;
    return smc_step_impl(tgt_logits, nullptr, drf_logq, dtype, draft_tokens, G, N, K, V,
                         temperature, alpha, SMCSD_TARGET_TOKEN, nullptr, 0.0f, bonus_uniforms,
                         logw, bonus_token, ess_threshold, resample_uniforms, ancestors, ess,
                         resampled, table_in, table_out, pages_per_seq, refcount, num_pages, ws,
                         ws_bytes, stream);
}

extern "C" int smc_step(const void* tgt_logits, const void* drf_logits, int dtype,
                        const int32_t* draft_tokens, int G, int N, int K, int V,
                        float temperature, float alpha, const float* bonus_uniforms, float* logw,
                        int32_t* bonus_token, float ess_threshold, const float* resample_uniforms,
                        int32_t* ancestors, float* ess, int32_t* resampled,
                        const int32_t* table_in, int32_t* table_out, int pages_per_seq,
                        int32_t* refcount, int num_pages, void* ws, size_t ws_bytes,
                        void* stream) {
    return smc_step_tilted(tgt_logits, drf_logits, dtype, draft_tokens, G, N, K, V, temperature,
                           alpha, SMCSD_TARGET_TOKEN, nullptr, 0.0f, bonus_uniforms, logw,
                           bonus_token, ess_threshold, resample_uniforms, ancestors, ess,
                           resampled, table_in, table_out, pages_per_seq, refcount, num_pages,
                           ws, ws_bytes, stream);
}

extern "C" int draft_sample(const void* logits, int dtype, int R, int V, float temperature,
                            const float* uniforms, int32_t* tokens, float* logq, float* lse,
                            void* ws, size_t ws_bytes, void* stream) {
    // each row is a "particle" with no draft positions: its (K+1)-th token is the draw
    StreamParams p{};
    int rc = smc_common(logits, nullptr, dtype, nullptr, R, 0, V, temperature, 1.0f,
                        SMCSD_TARGET_TOKEN, nullptr, 0.0f, uniforms, nullptr, tokens, ws, ws_bytes,
                        p);
    if (rc) return rc;
    p.mode = kModeSMC;
    p.lse_tgt = lse;
    p.bonus_logq = logq;
    return from_cuda(launch_stream(p, (cudaStream_t)stream));
}

extern "C" int smc_ess_resample(float* logw, int G, int N, float ess_threshold,
                                const float* uniforms, int32_t* ancestors, float* ess,
                                int32_t* resampled, void* ws, size_t ws_bytes, void* stream) {
    if (!logw || !uniforms || !ancestors || G <= 0 || N <= 0 || isnan(ess_threshold))
        return SMCSD_ERR_INVALID_ARG;
    int rc = check_ws(ws, ws_bytes, ws_small_bytes(G));
    if (rc) return rc;
    ResampleParams p{logw, G, N, ess_threshold, uniforms, ancestors, ess, resampled, ws, exp2_table()};
    return from_cuda(launch_resample(p, (cudaStream_t)stream));
}

extern "C" int kv_pagetable_remap(const int32_t* ancestors, const int32_t* resampled, int G,
                                  int N, const int32_t* table_in, int32_t* table_out,
                                  int pages_per_seq, int32_t* refcount, int num_pages, void* ws,
                                  size_t ws_bytes, void* stream) {
    if (!ancestors || !table_in || !table_out || table_in == table_out) return SMCSD_ERR_INVALID_ARG;
    if (G <= 0 || N <= 0 || pages_per_seq <= 0) return SMCSD_ERR_INVALID_ARG;
    if (refcount && num_pages <= 0) return SMCSD_ERR_INVALID_ARG;
    int rc = check_ws(ws, ws_bytes, ws_small_bytes(G));
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (refcount && cudaMemsetAsync(refcount, 0, (size_t)num_pages * sizeof(int32_t), st) != cudaSuccess)
        return SMCSD_ERR_CUDA;
    RemapParams p{ancestors, resampled, G, N, table_in, table_out, pages_per_seq, refcount, num_pages, ws};
    return from_cuda(launch_remap(p, st));
}

extern "C" int pacer_block_stop_pos(const void* hidden, const void* w, const void* pos_emb,
                                    float c, int S, int b, int max_blocks, int d, float t0,
                                    float rho, int32_t* lengths, float* block_scores,
                                    int32_t* tgt_offsets, int32_t* drf_offsets, void* ws,
                                    size_t ws_bytes, void* stream) {
    if (!hidden || !w || !lengths) return SMCSD_ERR_INVALID_ARG;
    if (S <= 0 || b <= 0 || b > 64 || max_blocks <= 0 || d <= 0) return SMCSD_ERR_INVALID_ARG;
    if (!isfinite(c) || !isfinite(t0) || !finite_pos(rho)) return SMCSD_ERR_INVALID_ARG;
    if ((tgt_offsets == nullptr) != (drf_offsets == nullptr)) return SMCSD_ERR_INVALID_ARG;
    int rc = check_ws(ws, ws_bytes, ws_small_bytes(S));
    if (rc) return rc;
    PacerParams p{};
    p.hidden = static_cast<const uint16_t*>(hidden);
    p.w = static_cast<const uint16_t*>(w);
    p.pos_emb = static_cast<const uint16_t*>(pos_emb);
    p.c = c;
    p.S = S;
    p.b = b;
    p.max_blocks = max_blocks;
    p.d = d;
    p.t0 = t0;
    p.rho = rho;
    p.vec = aligned16(hidden) && aligned16(w) && (!pos_emb || aligned16(pos_emb)) && (d % 8) == 0;
    p.lengths = lengths;
    p.block_scores = block_scores;
    p.tgt_offsets = tgt_offsets;
    p.drf_offsets = drf_offsets;
    p.ws = ws;
    p.L = ws_layout(S, 0, 1);
    return from_cuda(launch_pacer(p, (cudaStream_t)stream));
}

extern "C" int pacer_block_stop(const void* hidden, const void* w, float c, int S, int b,
                                int max_blocks, int d, float t0, float rho, int32_t* lengths,
                                float* block_scores, int32_t* tgt_offsets, int32_t* drf_offsets,
                                void* ws, size_t ws_bytes, void* stream) {
    return pacer_block_stop_pos(hidden, w, nullptr, c, S, b, max_blocks, d, t0, rho, lengths,
                                block_scores, tgt_offsets, drf_offsets, ws, ws_bytes, stream);
}
