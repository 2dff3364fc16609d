// api.cu -- the exported C ABI of libdlm: argument checks, then launches.
//
// Every check runs on the host before anything is enqueued, so a rejected
// call leaves the stream untouched.  Device attributes (SM count) are read
// once per device and cached.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not read yet (static storage starts zeroed)

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
    if (dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int dtype_size(int dt) { return dt == DLM_F32 ? 4 : 2; }

inline bool dtype_ok(int dt) { return dt == DLM_F32 || dt == DLM_BF16 || dt == DLM_F16; }

inline dlm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DLM_OK : DLM_ERR_CUDA; }

}  // namespace

extern "C" {

const char* dlm_status_string(dlm_status s) {
    switch (s) {
    case DLM_OK: return "ok";
    case DLM_ERR_INVALID_ARG: return "invalid argument";
    case DLM_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case DLM_ERR_UNSUPPORTED: return "unsupported dtype";
    case DLM_ERR_WORKSPACE: return "workspace missing or too small";
    case DLM_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

int dlm_version(void) { return 100; }

// CTAs per row: split a row over a cluster of CTAs only when the rows alone
// cannot fill the GPU and each CTA still gets at least two vectors per thread.
static int row_split(dlm_dtype dtype, int64_t n_rows, int64_t vocab) {
    const int64_t nvec = vocab / dlm::row_stats_elems_per_vector(dtype);
    const int threads = dlm::row_stats_threads();
    const int64_t target = 2LL * sm_count();
    int split = 1;
    while (split < 8 && n_rows * split < target && nvec / (split * 2) >= 2LL * threads) split *= 2;
    return split;
}

// Validation and launch shape shared by the whole-row and the slice calls.
static dlm_status row_stats_prepare(dlm::RowStatsArgs& a, const void* cur, const void* prev, dlm_dtype dtype,
                                    int64_t n_rows, int64_t vocab, int64_t row_stride, const int32_t* row_index) {
    if (!dtype_ok(dtype)) return DLM_ERR_UNSUPPORTED;
    if (n_rows < 0 || vocab < 1 || vocab > 0x7fffffffLL || row_stride < vocab) return DLM_ERR_INVALID_ARG;
    if (n_rows == 0) return DLM_OK;
    if (!cur) return DLM_ERR_INVALID_ARG;
    const int esz = dtype_size(dtype);
    if (!aligned16(cur) || (prev && !aligned16(prev)) || (row_stride * esz) % 16 != 0) return DLM_ERR_ALIGNMENT;
    const int split = row_split(dtype, n_rows, vocab);
    const int64_t target = 2LL * sm_count();
    if (n_rows * split > 0x7fffffffLL) return DLM_ERR_INVALID_ARG;
    a = dlm::RowStatsArgs{};
    a.cur = cur;
    a.prev = prev;
    a.n_rows = n_rows;
    a.vocab = vocab;
    a.row_stride = row_stride;
    a.row_index = row_index;
    a.split = split;
    a.num_sms = (int)(target / 2);
    return DLM_OK;
}

dlm_status dlm_row_stats_ex(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows, int64_t vocab,
                            int64_t row_stride, const int32_t* row_index, int64_t n_src_rows, int32_t* argmax,
                            float* conf, float* lse, float* entropy, float* kl, float* lse_prev,
                            uint32_t* dev_status, uint32_t flags, dlm_stream_t stream) {
    if ((flags & ~(DLM_ROWS_SINGLE_GRID | DLM_ROWS_GATHER)) || n_src_rows < 0) return DLM_ERR_INVALID_ARG;
    if (!row_index && n_src_rows > 0 && n_rows > n_src_rows) return DLM_ERR_INVALID_ARG;
    dlm::RowStatsArgs a{};
    const dlm_status st = row_stats_prepare(a, cur, prev, dtype, n_rows, vocab, row_stride, row_index);
    if (st != DLM_OK || n_rows == 0) return st;
    if (!argmax || !conf || !lse || !entropy) return DLM_ERR_INVALID_ARG;
    a.n_src = n_src_rows;
    a.gather = (flags & DLM_ROWS_GATHER) ? 1 : 0;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.entropy = entropy;
    a.kl = kl;
    a.lse_prev = lse_prev;
    a.dev_status = dev_status;
    a.single_grid = (flags & DLM_ROWS_SINGLE_GRID) ? 1 : 0;
    return from_cuda(dlm::launch_row_stats(a, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_row_stats(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows,
                         int64_t vocab, int64_t row_stride, const int32_t* row_index,
                         int32_t* argmax, float* conf, float* lse, float* entropy, float* kl,
                         float* lse_prev, uint32_t* dev_status, dlm_stream_t stream) {
    return dlm_row_stats_ex(cur, prev, dtype, n_rows, vocab, row_stride, row_index, 0, argmax, conf, lse, entropy,
                            kl, lse_prev, dev_status, 0u, stream);
}

int32_t dlm_row_stats_launches(dlm_dtype dtype, int32_t has_prev, int64_t n_rows, int64_t vocab,
                               uint32_t flags) {
    if (!dtype_ok(dtype) || n_rows < 0 || vocab < 1 || vocab > 0x7fffffffLL ||
        (flags & ~(DLM_ROWS_SINGLE_GRID | DLM_ROWS_GATHER)))
        return -1;
    if (n_rows == 0) return 0;
    dlm::RowStatsArgs a{};
    // alignment does not change the launch shape: use a dummy aligned pointer
    static const uint4 dummy = {0, 0, 0, 0};
    const int esz = dtype_size(dtype);
    const int64_t stride = (vocab * esz + 15) / 16 * 16 / esz;
    if (row_stats_prepare(a, &dummy, has_prev ? &dummy : nullptr, dtype, n_rows, vocab, stride, nullptr) != DLM_OK)
        return -1;
    a.single_grid = (flags & DLM_ROWS_SINGLE_GRID) ? 1 : 0;
    return dlm::row_stats_grids(a, dtype);
}

dlm_status dlm_row_stats_partial(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows,
                                 int64_t vocab, int64_t row_stride, const int32_t* row_index,
                                 int64_t vocab_offset, dlm_row_partial* partial, dlm_stream_t stream) {
    dlm::RowStatsArgs a{};
    const dlm_status st = row_stats_prepare(a, cur, prev, dtype, n_rows, vocab, row_stride, row_index);
    if (st != DLM_OK || n_rows == 0) return st;
    if (!partial || vocab_offset < 0 || vocab_offset + vocab > 0x7fffffffLL) return DLM_ERR_INVALID_ARG;
    a.partial = partial;
    a.vocab_offset = vocab_offset;
    return from_cuda(dlm::launch_row_stats(a, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_row_stats_merge(const dlm_row_partial* partials, int32_t n_shards, int64_t shard_stride,
                               int64_t n_rows, const int32_t* row_index, int32_t has_prev, int32_t* argmax,
                               float* conf, float* lse, float* entropy, float* kl, float* lse_prev,
                               uint32_t* dev_status, dlm_stream_t stream) {
    if (n_shards < 1 || n_rows < 0 || shard_stride < 0 || (n_shards > 1 && shard_stride < 1) ||
        (has_prev != 0 && has_prev != 1))
        return DLM_ERR_INVALID_ARG;
    if (n_rows == 0) return DLM_OK;
    if (!partials || !argmax || !conf || !lse || !entropy) return DLM_ERR_INVALID_ARG;
    dlm::RowStatsArgs a{};
    a.n_rows = n_rows;
    a.row_index = row_index;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.entropy = entropy;
    a.kl = kl;
    a.lse_prev = lse_prev;
    a.dev_status = dev_status;
    return from_cuda(dlm::launch_row_merge(a, partials, n_shards, shard_stride, has_prev != 0,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

size_t dlm_row_stats_rules_workspace_size(int32_t batch) {
    if (batch < 0 || batch > DLM_MAX_BATCH) return 0;
    return ((size_t)batch * sizeof(unsigned) + 255) & ~(size_t)255;
}

dlm_status dlm_row_stats_rules(const void* cur, const void* prev, dlm_dtype dtype, int32_t batch, int32_t blk,
                               int64_t vocab, int64_t row_stride, const uint8_t* masked,
                               const dlm_step_rules* rules, int32_t* argmax, float* conf, float* lse,
                               float* entropy, float* kl, float* lse_prev, uint8_t* thr_selected,
                               int32_t* thr_n_selected, int32_t* block_len, float* score, uint8_t* cap_selected,
                               int32_t* cap_n_selected, void* workspace, size_t ws_bytes, uint32_t* dev_status,
                               dlm_stream_t stream) {
    if (!rules || batch < 0 || batch > DLM_MAX_BATCH || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    const uint32_t on = rules->rules;
    const uint32_t all = DLM_RULE_THRESHOLD | DLM_RULE_BOUNDARY | DLM_RULE_CAP;
    if (on == 0 || (on & ~all)) return DLM_ERR_INVALID_ARG;
    const bool thr = on & DLM_RULE_THRESHOLD, bnd = on & DLM_RULE_BOUNDARY, cap = on & DLM_RULE_CAP;
    if (rules->cap_scope_from_boundary != 0 && rules->cap_scope_from_boundary != 1) return DLM_ERR_INVALID_ARG;
    if (rules->cap_scope_from_boundary && !(bnd && cap)) return DLM_ERR_INVALID_ARG;
    if (bnd) {
        const dlm_depcap_params& d = rules->depcap;
        if (d.L_min < 1 || d.smooth_w < 1 || d.smooth_w > 63 || (d.smooth_w % 2) == 0 || d.norm_mode < 0 ||
            d.norm_mode > 2 || !isfinite(d.lambda))
            return DLM_ERR_INVALID_ARG;
    }
    if (cap) {
        const dlm_cap_params& c = rules->cap;
        if (c.p_max < 1 || c.p_max > 64 || (c.high_tier_unconditional != 0 && c.high_tier_unconditional != 1))
            return DLM_ERR_INVALID_ARG;
    }
    const int64_t n_rows = (int64_t)batch * blk;
    dlm::RowStatsArgs a{};
    const dlm_status st = row_stats_prepare(a, cur, prev, dtype, n_rows, vocab, row_stride, nullptr);
    if (st != DLM_OK || batch == 0) return st;
    if (!masked || !argmax || !conf || !lse || !entropy) return DLM_ERR_INVALID_ARG;
    if (thr && (!thr_selected || !thr_n_selected)) return DLM_ERR_INVALID_ARG;
    if (bnd && (!prev || !kl || !block_len)) return DLM_ERR_INVALID_ARG;
    if (cap && (!cap_selected || !cap_n_selected)) return DLM_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < dlm_row_stats_rules_workspace_size(batch)) return DLM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DLM_ERR_ALIGNMENT;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.entropy = entropy;
    a.kl = kl;
    a.lse_prev = lse_prev;
    a.dev_status = dev_status;
    dlm::RowRules r{};
    r.counter = static_cast<unsigned*>(workspace);
    r.blk = blk;
    r.thr = thr;
    r.bnd = bnd;
    r.cap = cap;
    r.t = dlm::ThresholdArgs{conf, masked, batch, blk, rules->tau, thr_selected, thr_n_selected};
    r.d = dlm::BoundaryArgs{kl, entropy, batch, blk, nullptr, rules->cold_start, rules->depcap.lambda,
                            rules->depcap.L_min, rules->depcap.smooth_w, rules->depcap.norm_mode, block_len, score};
    dlm::CapArgs& c = r.c;
    c.logits = cur;
    c.dtype = dtype;
    c.vocab = vocab;
    c.row_stride = row_stride;
    c.argmax = argmax;
    c.conf = conf;
    c.lse = lse;
    c.masked = masked;
    c.scope_len = rules->cap_scope_from_boundary ? block_len : nullptr;
    c.row_index = nullptr;
    c.n_rows = n_rows;
    c.batch = batch;
    c.blk = blk;
    c.tau_low = rules->cap.tau_low;
    c.tau_high = rules->cap.tau_high;
    c.gamma = rules->cap.gamma;
    c.p_max = rules->cap.p_max;
    c.high_tier_unconditional = rules->cap.high_tier_unconditional;
    c.selected = cap_selected;
    c.n_selected = cap_n_selected;
    c.D_out = nullptr;
    c.dev_status = dev_status;
    return from_cuda(dlm::launch_row_stats_rules(a, r, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_select_threshold(const float* conf, const uint8_t* masked, int32_t batch,
                                int32_t blk, float tau, uint8_t* selected, int32_t* n_selected,
                                dlm_stream_t stream) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!conf || !masked || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    dlm::ThresholdArgs a{conf, masked, batch, blk, tau, selected, n_selected};
    return from_cuda(dlm::launch_threshold(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_select_topk(const float* conf, const uint8_t* masked, int32_t batch, int32_t blk, int32_t k,
                           uint8_t* selected, int32_t* n_selected, dlm_stream_t stream) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK || k < 0) return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!conf || !masked || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    dlm::RankSelectArgs a{conf, masked, batch, blk, 0, k, 0.f, selected, n_selected};
    return from_cuda(dlm::launch_rank_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_select_factor(const float* conf, const uint8_t* masked, int32_t batch, int32_t blk, float f,
                             uint8_t* selected, int32_t* n_selected, dlm_stream_t stream) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK || !isfinite(f)) return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!conf || !masked || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    dlm::RankSelectArgs a{conf, masked, batch, blk, 1, 0, f, selected, n_selected};
    return from_cuda(dlm::launch_rank_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_parallel_certificate(const float* conf, const uint8_t* selected, int32_t batch, int32_t blk,
                                    uint8_t* certified, dlm_stream_t stream) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!conf || !selected || !certified) return DLM_ERR_INVALID_ARG;
    dlm::CertificateArgs a{conf, selected, batch, blk, certified};
    return from_cuda(dlm::launch_certificate(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_depcap_boundary(const float* kl, const float* entropy, int32_t batch,
                               int32_t L_window, const uint8_t* cold_start,
                               const dlm_depcap_params* params, int32_t* block_len,
                               float* score, dlm_stream_t stream) {
    if (!params || batch < 0 || L_window < 1 || L_window > 1024) return DLM_ERR_INVALID_ARG;
    if (params->L_min < 1 || params->smooth_w < 1 || params->smooth_w > 63 || (params->smooth_w % 2) == 0 ||
        params->norm_mode < 0 || params->norm_mode > 2 || !isfinite(params->lambda))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!kl || !entropy || !block_len) return DLM_ERR_INVALID_ARG;
    dlm::BoundaryArgs a{kl, entropy, batch, L_window, nullptr, cold_start, params->lambda,
                        params->L_min, params->smooth_w, params->norm_mode, block_len, score};
    return from_cuda(dlm::launch_boundary(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_depcap_boundary_ragged(const float* kl, const float* entropy, int32_t batch,
                                      int32_t L_stride, const int32_t* window_len,
                                      const uint8_t* cold_start, const dlm_depcap_params* params,
                                      int32_t* block_len, float* score, dlm_stream_t stream) {
    if (!params || batch < 0 || L_stride < 1 || L_stride > 1024) return DLM_ERR_INVALID_ARG;
    if (params->L_min < 1 || params->smooth_w < 1 || params->smooth_w > 63 || (params->smooth_w % 2) == 0 ||
        params->norm_mode < 0 || params->norm_mode > 2 || !isfinite(params->lambda))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!kl || !entropy || !block_len || !window_len) return DLM_ERR_INVALID_ARG;
    dlm::BoundaryArgs a{kl, entropy, batch, L_stride, window_len, cold_start, params->lambda,
                        params->L_min, params->smooth_w, params->norm_mode, block_len, score};
    return from_cuda(dlm::launch_boundary(a, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_revocable_step(const int32_t* argmax, const float* conf, const float* influence,
                              const float* drift, int32_t batch, int32_t blk, int32_t step,
                              const dlm_revocable_params* p, int32_t* tok, uint8_t* masked, uint8_t* seed,
                              int32_t* last_seed, int32_t* remasks, int32_t* last_tok, uint8_t* outcome,
                              int32_t* n_drafted, int32_t* n_revoked, int32_t* flipflops,
                              dlm_stream_t stream) {
    if (!p || batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    if (!isfinite(p->pi) || p->pi < 0.f || !isfinite(p->w_unc) || !isfinite(p->w_infl) ||
        !isfinite(p->w_drift) || isnan(p->tau_replace) || isnan(p->tau_draft))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!argmax || !conf || !tok || !masked || !seed || !last_seed || !remasks || !last_tok)
        return DLM_ERR_INVALID_ARG;
    dlm::RevocableArgs a{argmax, conf, influence, drift, batch, blk, step, p->tau_replace, p->tau_draft,
                         p->draft_budget, p->w_unc, p->w_infl, p->w_drift, p->pi, p->cooldown,
                         p->remask_budget, tok, masked, seed, last_seed, remasks, last_tok, outcome,
                         n_drafted, n_revoked, flipflops};
    return from_cuda(dlm::launch_revocable(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t dlm_cap_workspace_size(int32_t batch, int32_t p_max) {
    if (batch < 0 || p_max < 1 || p_max > DLM_MAX_BLK) return 0;
    return dlm::cap_workspace_bytes(batch, p_max);
}

dlm_status dlm_cap_select(const void* logits, dlm_dtype dtype, int64_t vocab, int64_t row_stride,
                          const int32_t* row_index, int64_t n_rows, const int32_t* argmax, const float* conf,
                          const float* lse, const uint8_t* masked, const int32_t* scope_len, int32_t batch,
                          int32_t blk, const dlm_cap_params* params, uint8_t* selected,
                          int32_t* n_selected, float* D_out, void* workspace, size_t ws_bytes,
                          uint32_t* dev_status, dlm_stream_t stream) {
    if (!dtype_ok(dtype)) return DLM_ERR_UNSUPPORTED;
    if (!params || batch < 0 || batch > DLM_MAX_BATCH || blk < 1 || blk > DLM_MAX_BLK || vocab < 1 ||
        row_stride < vocab || params->p_max < 1 || params->p_max > DLM_MAX_BLK ||
        (params->high_tier_unconditional != 0 && params->high_tier_unconditional != 1))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (n_rows < 1 || (!row_index && n_rows < (int64_t)batch * blk)) return DLM_ERR_INVALID_ARG;
    if (!logits || !argmax || !conf || !lse || !masked || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < dlm::cap_workspace_bytes(batch, params->p_max)) return DLM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DLM_ERR_ALIGNMENT;
    dlm::CapArgs a{};
    a.logits = logits;
    a.dtype = dtype;
    a.vocab = vocab;
    a.row_stride = row_stride;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.masked = masked;
    a.scope_len = scope_len;
    a.row_index = row_index;
    a.n_rows = n_rows;
    a.batch = batch;
    a.blk = blk;
    a.tau_low = params->tau_low;
    a.tau_high = params->tau_high;
    a.gamma = params->gamma;
    a.p_max = params->p_max;
    a.high_tier_unconditional = params->high_tier_unconditional;
    a.selected = selected;
    a.n_selected = n_selected;
    a.D_out = D_out;
    a.dev_status = dev_status;
    dlm::cap_carve(a, workspace);
    return from_cuda(dlm::launch_cap(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t dlm_dapd_workspace_size(int32_t batch, int32_t blk) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return 0;
    return dlm::dapd_workspace_bytes(batch, blk);
}

}  // extern "C"

namespace {

// Shared argument checks and set-up of the DAPD calls; selection outputs and
// conf are checked by the callers that need them.
dlm_status dapd_prepare(dlm::DapdArgs& a, const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                        int32_t n_heads, int64_t stride_b, int64_t stride_l, int64_t stride_h, int64_t stride_row,
                        int32_t block_start, int32_t blk, const uint8_t* masked, const dlm_dapd_params* params,
                        void* workspace, size_t ws_bytes, bool need_attn) {
    if (need_attn && !dtype_ok(dtype)) return DLM_ERR_UNSUPPORTED;
    if (!params || batch < 0 || batch > DLM_MAX_BATCH || blk < 1 || blk > DLM_MAX_BLK ||
        (params->order_mode != 0 && params->order_mode != 1) ||
        (params->preunmask_certain != 0 && params->preunmask_certain != 1) || !isfinite(params->tau_edge))
        return DLM_ERR_INVALID_ARG;
    if (need_attn && (n_layers < 1 || n_heads < 1 || (int64_t)n_layers * n_heads > (1 << 20) || block_start < 0 ||
                      stride_b < 0 || stride_l < 0 || stride_h < 0 || stride_row < blk))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (!masked || (need_attn && !attn)) return DLM_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < dlm::dapd_workspace_bytes(batch, blk)) return DLM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DLM_ERR_ALIGNMENT;
    a = dlm::DapdArgs{};
    if (need_attn) {
        const int esz = dtype_size(dtype);
        const char* first = static_cast<const char*>(attn) + ((int64_t)block_start * stride_row + block_start) * esz;
        if (!aligned16(first) || (stride_b * esz) % 16 || (stride_l * esz) % 16 || (stride_h * esz) % 16 ||
            (stride_row * esz) % 16)
            return DLM_ERR_ALIGNMENT;
        const double LH = (double)n_layers * (double)n_heads;
        const double unit = 2.0 * LH * 4294967296.0;        // 2 L H 2^32: s = I / unit
        const double t = floor((double)params->tau_edge * unit);  // exact: tau is fp32, unit < 2^53
        a.edge_thresh = t >= 9.2e18 ? 0x7fffffffffffffffLL : (t <= -9.2e18 ? -0x7fffffffffffffffLL - 1 : (long long)t);
        a.s_scale = (float)(1.0 / unit);
        a.attn = attn;
        a.dtype = dtype;
        a.n_layers = n_layers;
        a.n_heads = n_heads;
        a.sb = stride_b;
        a.sl = stride_l;
        a.sh = stride_h;
        a.sr = stride_row;
        a.block_start = block_start;
    }
    a.batch = batch;
    a.blk = blk;
    a.masked = masked;
    a.tau_edge = params->tau_edge;
    a.bulk_conf = params->bulk_conf;
    a.bulk_frac = params->bulk_frac;
    a.order_mode = params->order_mode;
    a.preunmask_certain = params->preunmask_certain;
    dlm::dapd_carve(a, workspace);
    return DLM_OK;
}

}  // namespace

extern "C" {

dlm_status dlm_attention_influence(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                                   int32_t n_heads, int64_t stride_b, int64_t stride_l, int64_t stride_h,
                                   int64_t stride_row, int32_t block_start, int32_t blk, const uint8_t* masked,
                                   float* influence, void* workspace, size_t ws_bytes, uint32_t* dev_status,
                                   dlm_stream_t stream) {
    const dlm_dapd_params prm = {0.f, 0.f, 0.f, 0, 0};
    dlm::DapdArgs a{};
    const dlm_status st = dapd_prepare(a, attn, dtype, batch, n_layers, n_heads, stride_b, stride_l, stride_h,
                                       stride_row, block_start, blk, masked, &prm, workspace, ws_bytes, true);
    if (st != DLM_OK || batch == 0) return st;
    if (!influence) return DLM_ERR_INVALID_ARG;
    a.dev_status = dev_status;
    return from_cuda(dlm::launch_attention_influence(a, sm_count(), influence, reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_dapd_graph_mis(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                              int32_t n_heads, int64_t stride_b, int64_t stride_l,
                              int64_t stride_h, int64_t stride_row, int32_t block_start,
                              int32_t blk, const uint8_t* masked, const float* conf,
                              const dlm_dapd_params* params, uint8_t* selected,
                              int32_t* n_selected, float* s_out, float* dtilde_out,
                              int32_t* deg_out, void* workspace, size_t ws_bytes,
                              uint32_t* dev_status, dlm_stream_t stream) {
    dlm::DapdArgs a{};
    const dlm_status st = dapd_prepare(a, attn, dtype, batch, n_layers, n_heads, stride_b, stride_l, stride_h,
                                       stride_row, block_start, blk, masked, params, workspace, ws_bytes, true);
    if (st != DLM_OK || batch == 0) return st;
    if (!conf || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    a.conf = conf;
    a.selected = selected;
    a.n_selected = n_selected;
    a.s_out = s_out;
    a.dtilde_out = dtilde_out;
    a.deg_out = deg_out;
    a.dev_status = dev_status;
    return from_cuda(dlm::launch_dapd(a, sm_count(), reinterpret_cast<cudaStream_t>(stream)));
}

dlm_status dlm_dapd_graph(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers, int32_t n_heads,
                          int64_t stride_b, int64_t stride_l, int64_t stride_h, int64_t stride_row,
                          int32_t block_start, int32_t blk, const uint8_t* masked, const dlm_dapd_params* params,
                          float* s_out, float* dtilde_out, int32_t* deg_out, void* workspace, size_t ws_bytes,
                          uint32_t* dev_status, dlm_stream_t stream) {
    dlm::DapdArgs a{};
    const dlm_status st = dapd_prepare(a, attn, dtype, batch, n_layers, n_heads, stride_b, stride_l, stride_h,
                                       stride_row, block_start, blk, masked, params, workspace, ws_bytes, true);
    if (st != DLM_OK || batch == 0) return st;
    a.s_out = s_out;
    a.dtilde_out = dtilde_out;
    a.deg_out = deg_out;
    a.dev_status = dev_status;
    // the selection rebuilds the graph from the sums; the graph kernel runs
    // only for the float outputs
    const bool graph_kernel = s_out || dtilde_out || deg_out;
    return from_cuda(dlm::launch_dapd_graph(a, sm_count(), reinterpret_cast<cudaStream_t>(stream), graph_kernel));
}

dlm_status dlm_dapd_select(const uint8_t* masked, const float* conf, int32_t batch, int32_t blk,
                           const dlm_dapd_params* params, uint8_t* selected, int32_t* n_selected,
                           void* workspace, size_t ws_bytes, dlm_stream_t stream) {
    dlm::DapdArgs a{};
    const dlm_status st = dapd_prepare(a, nullptr, DLM_F16, batch, 0, 0, 0, 0, 0, 0, 0, blk, masked, params,
                                       workspace, ws_bytes, false);
    if (st != DLM_OK || batch == 0) return st;
    if (!conf || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    a.conf = conf;
    a.selected = selected;
    a.n_selected = n_selected;
    a.thresh_from_ws = 1;
    return from_cuda(dlm::launch_dapd_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Folding pays where the rows are too few to fill the GPU (the row pass
// splits each row over a cluster) and the copied attention fits shared
// memory; with whole waves of rows the scattered attention reads cost the
// same DRAM time inside the row pass as in a pass of their own, and the
// separate pass beside the row pass is faster.
static bool attention_folds(int64_t n_rows, int split, dlm_dtype attn_dtype, int32_t n_layers, int32_t n_heads,
                            int32_t blk) {
    if (split < 2 || n_rows < 1) return false;
    dlm::RowAttn at{};
    at.attn = &at;  // any non-null pointer: only the shape decides
    at.esz = dtype_size(attn_dtype);
    at.n_layers = n_layers;
    at.n_heads = n_heads;
    at.blk = blk;
    return dlm::row_attn_smem(at) > 0;
}

int32_t dlm_row_stats_attention_folds(dlm_dtype dtype, int32_t batch, int32_t blk, int64_t vocab,
                                      dlm_dtype attn_dtype, int32_t n_layers, int32_t n_heads) {
    if (!dtype_ok(dtype) || !dtype_ok(attn_dtype) || n_layers < 1 || n_heads < 1 ||
        (int64_t)n_layers * n_heads > (1 << 20) || batch < 1 || blk < 1 || blk > DLM_MAX_BLK || vocab < 1 ||
        vocab > 0x7fffffffLL)
        return 0;
    const int64_t n_rows = (int64_t)batch * blk;
    return attention_folds(n_rows, row_split(dtype, n_rows, vocab), attn_dtype, n_layers, n_heads, blk) ? 1 : 0;
}

dlm_status dlm_row_stats_attention(const void* cur, const void* prev, dlm_dtype dtype, int32_t batch, int32_t blk,
                                   int64_t vocab, int64_t row_stride, int32_t* argmax, float* conf, float* lse,
                                   float* entropy, float* kl, float* lse_prev, const void* attn,
                                   dlm_dtype attn_dtype, int32_t n_layers, int32_t n_heads, int64_t stride_b,
                                   int64_t stride_l, int64_t stride_h, int64_t stride_row, int32_t block_start,
                                   const uint8_t* masked, const dlm_dapd_params* params, void* workspace,
                                   size_t ws_bytes, uint32_t* dev_status, dlm_stream_t stream) {
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    const int64_t n_rows = (int64_t)batch * blk;
    dlm::RowStatsArgs a{};
    dlm_status st = row_stats_prepare(a, cur, prev, dtype, n_rows, vocab, row_stride, nullptr);
    if (st != DLM_OK) return st;
    dlm::DapdArgs d{};
    st = dapd_prepare(d, attn, attn_dtype, batch, n_layers, n_heads, stride_b, stride_l, stride_h, stride_row,
                      block_start, blk, masked, params, workspace, ws_bytes, true);
    if (st != DLM_OK || n_rows == 0) return st;
    if (!argmax || !conf || !lse || !entropy) return DLM_ERR_INVALID_ARG;
    a.n_src = n_rows;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.entropy = entropy;
    a.kl = kl;
    a.lse_prev = lse_prev;
    a.dev_status = dev_status;
    d.dev_status = dev_status;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dlm::RowAttn& at = a.at;
    at.attn = attn;
    at.dtype = attn_dtype;
    at.esz = dtype_size(attn_dtype);
    at.n_layers = n_layers;
    at.n_heads = n_heads;
    at.sb = stride_b;
    at.sl = stride_l;
    at.sh = stride_h;
    at.sr = stride_row;
    at.block_start = block_start;
    at.blk = blk;
    at.vpr = (int)((int64_t)blk * at.esz / 16);
    at.masked = masked;
    at.mask4 = (blk % 4 == 0 && (reinterpret_cast<uintptr_t>(masked) & 3u) == 0) ? 1 : 0;
    at.bulk_frac = d.bulk_frac;
    at.edge_thresh = d.edge_thresh;
    at.s_scale = d.s_scale;
    at.A = d.A;
    at.hdr = d.hdr;
    if (attention_folds(n_rows, a.split, attn_dtype, n_layers, n_heads, blk))
        return from_cuda(dlm::launch_row_stats_attn(a, dtype, s));
    // not foldable: the row pass, then the attention pass, on the stream
    a.at = dlm::RowAttn{};
    const cudaError_t e = dlm::launch_row_stats(a, dtype, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(dlm::launch_dapd_graph(d, sm_count(), s, false));
}

}  // extern "C"
