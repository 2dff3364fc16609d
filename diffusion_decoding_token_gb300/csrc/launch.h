// launch.h -- internal kernel launchers of libdlm (host side, not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dlm.h"

namespace dlm {

// The DAPD attention sums folded into the row pass (dlm_row_stats_attention):
// the CTA of row b*blk + i (rank 0 of its cluster) copies row i of sequence
// b's attention block, for every layer and head, into shared memory while it
// streams the logits, then sums it into row i of the DAPD workspace's A.
struct RowAttn {
    const void* attn;          // null: no attention sums (plain row pass)
    int dtype, esz;
    int n_layers, n_heads;
    int64_t sb, sl, sh, sr;    // element strides
    int block_start, blk;
    int vpr;                   // 16-byte vectors per block row (blk * esz / 16)
    const uint8_t* masked;
    int mask4;                 // the mask rows are copied 4 bytes at a time (aligned, blk % 4 == 0)
    float bulk_frac;
    long long edge_thresh;
    float s_scale;
    long long* A;              // [batch][blk][blk] fixed-point sums (units 2^-32)
    long long* hdr;            // edge threshold, score scale bits
};

struct RowStatsArgs {
    const void* cur;
    const void* prev;
    int64_t n_rows, vocab, row_stride;
    const int32_t* row_index;
    int32_t* argmax;
    float* conf;
    float* lse;
    float* entropy;
    float* kl;
    float* lse_prev;
    uint32_t* dev_status;
    int split;  // CTAs per row (thread-block cluster size), 1..8
    void* partial;         // non-null: write each row's dlm_row_partial state instead of outputs
    int64_t vocab_offset;  // global position of the slice's first element
    int64_t row_base;      // first row of this grid (a tail grid after whole waves)
    int wait_prior;        // complete only after the previous grid on the stream
    int num_sms;
    int single_grid;       // no tail grid of half rows
    int64_t n_src;         // rows cur/prev hold: q >= n_src is skipped (0 = unchecked)
    int gather;            // outputs at r (the gathered order) instead of q
    RowAttn at;            // attention sums folded in (at.attn non-null; rows are b*blk + i)
};
cudaError_t launch_row_stats(const RowStatsArgs& a, int dtype, cudaStream_t s);
// the row pass with the attention sums folded in (a.at set); shared memory
// per CTA for it, or 0 when the attention cannot be folded in
size_t row_attn_smem(const RowAttn& at);
cudaError_t launch_row_stats_attn(const RowStatsArgs& a, int dtype, cudaStream_t s);
int row_stats_grids(const RowStatsArgs& a, int dtype);  // kernel launches launch_row_stats makes
// merge of dlm_row_partial states: a gives n_rows, row_index and the outputs
cudaError_t launch_row_merge(const RowStatsArgs& a, const void* partials, int n_shards, int64_t shard_stride,
                             bool prev, cudaStream_t s);
int row_stats_elems_per_vector(int dtype);
int row_stats_threads();

struct ThresholdArgs {
    const float* conf;
    const uint8_t* masked;
    int batch, blk;
    float tau;
    uint8_t* selected;
    int32_t* n_selected;
};
cudaError_t launch_threshold(const ThresholdArgs& a, cudaStream_t s);

struct RankSelectArgs {
    const float* conf;
    const uint8_t* masked;
    int batch, blk;
    int mode;  // 0: top-K, 1: factor decoding
    int k;
    float f;
    uint8_t* selected;
    int32_t* n_selected;
};
cudaError_t launch_rank_select(const RankSelectArgs& a, cudaStream_t s);

struct CertificateArgs {
    const float* conf;
    const uint8_t* selected;
    int batch, blk;
    uint8_t* certified;
};
cudaError_t launch_certificate(const CertificateArgs& a, cudaStream_t s);

struct RevocableArgs {
    const int32_t* argmax;
    const float* conf;
    const float* influence;
    const float* drift;
    int batch, blk, step;
    float tau_replace, tau_draft;
    int draft_budget;
    float w_unc, w_infl, w_drift, pi;
    int cooldown, remask_budget;
    int32_t* tok;
    uint8_t* masked;
    uint8_t* seed;
    int32_t* last_seed;
    int32_t* remasks;
    int32_t* last_tok;
    uint8_t* outcome;
    int32_t* n_drafted;
    int32_t* n_revoked;
    int32_t* flipflops;
};
cudaError_t launch_revocable(const RevocableArgs& a, cudaStream_t s);

struct BoundaryArgs {
    const float* kl;
    const float* entropy;
    int batch, L_window;     // L_window: row stride (the longest window)
    const int32_t* window_len;  // nullable: per-sequence window (<= L_window)
    const uint8_t* cold_start;
    float lambda;
    int L_min, smooth_w, norm_mode;
    int32_t* block_len;
    float* score;
};
cudaError_t launch_boundary(const BoundaryArgs& a, cudaStream_t s);

struct CapArgs {
    const void* logits;
    int dtype;
    int64_t vocab;  // a token outside [0, vocab) is never gathered
    int64_t row_stride;
    const int32_t* argmax;
    const float* conf;
    const float* lse;
    const uint8_t* masked;
    const int32_t* scope_len;
    const int32_t* row_index;  // [batch*blk] logit row of each block position (nullable)
    int64_t n_rows;            // rows the logits hold: others are never read
    int batch, blk;
    float tau_low, tau_high, gamma;
    int p_max, high_tier_unconditional;
    uint8_t* selected;
    int32_t* n_selected;
    float* D_out;
    uint32_t* dev_status;
    // workspace carve-up
    int32_t* pool;     // [batch][p_max] block positions in pool order
    int32_t* pool_n;   // [batch]
    uint32_t* adj;     // [batch][p_max][words] conflict bits over pool slots
    int words;         // ceil(p_max / 32)
};
size_t cap_workspace_bytes(int batch, int p_max);
void cap_carve(CapArgs& a, void* ws);
cudaError_t launch_cap(const CapArgs& a, cudaStream_t s);

struct DapdArgs {
    const void* attn;
    int dtype;
    int batch, n_layers, n_heads;
    int64_t sb, sl, sh, sr;  // element strides
    int block_start, blk;
    const uint8_t* masked;
    const float* conf;
    float tau_edge, bulk_conf, bulk_frac;
    int order_mode;
    int preunmask_certain;
    long long edge_thresh;   // floor(tau * 2 * L * H * 2^32): edge <=> 2LH 2^32 s > this
    float s_scale;           // 1 / (2 * L * H * 2^32)
    uint8_t* selected;
    int32_t* n_selected;
    float* s_out;
    float* dtilde_out;
    int32_t* deg_out;
    uint32_t* dev_status;
    // workspace carve-up
    long long* A;      // [batch][blk][blk] fixed-point sums (units 2^-32)
    long long* Dsum;   // [batch][blk]
    uint32_t* adj;     // [batch][blk][8]
    long long* hdr;    // [2]: edge threshold, score scale bits (written by the attention pass)
    int thresh_from_ws;  // the selection reads them from hdr (no attention arguments)
    int split;         // CTAs per cluster over the layer*head range
    int row_tile;      // rows per CTA
    // bulk-tensor (TMA) path: box = [box_cols x row_tile rows x box_heads]
    int box_cols, box_heads, head_groups, box_bytes;
    // >= 0: the first bulk-copy wait of the attention pass gives up after this
    // many clock cycles (non-blocking probes), a test of the timeout path;
    // < 0: every wait has the normal ~1 s limit
    long long first_wait_limit;
};
size_t dapd_workspace_bytes(int batch, int blk);
void dapd_carve(DapdArgs& a, void* ws);
cudaError_t launch_dapd(DapdArgs& a, int num_sms, cudaStream_t s);  // attention -> selection
// attention -> sums; with graph_kernel also the graph's float outputs (the
// selection rebuilds the graph from the sums itself)
cudaError_t launch_dapd_graph(DapdArgs& a, int num_sms, cudaStream_t s, bool graph_kernel);
cudaError_t launch_dapd_select(const DapdArgs& a, cudaStream_t s);  // (graph +) conf -> selection

// The fused row pass: after the rows of sequence b are all written, the CTA
// that wrote the last of them runs b's threshold, boundary and CAP rules
// (rules.cuh) with the arguments below; counter[b] counts finished rows and
// is reset to 0 by that CTA.  Rows are b*blk + i (no row index).
struct RowRules {
    unsigned* counter;  // [batch], zero before a call, left zero after it
    int blk;
    int thr, bnd, cap;  // which rules run (CAP reads the boundary's length when c.scope_len is set)
    ThresholdArgs t;
    BoundaryArgs d;
    CapArgs c;
};
cudaError_t launch_row_stats_rules(const RowStatsArgs& a, const RowRules& r, int dtype, cudaStream_t s);
// attention -> sums (every sequence) -> infl[b][j] = column sums over masked rows / (L H)
cudaError_t launch_attention_influence(DapdArgs& a, int num_sms, float* infl, cudaStream_t s);

}  // namespace dlm
