/*
 * dlm.h -- C ABI of the per-step unmask-decision library (libdlm.so).
 *
 * After every forward pass of a masked diffusion LM, the positions still
 * masked in the active block have a vocab-wide logit row each.  This library
 * turns those rows (and, for DAPD, the model's attention maps) into the set of
 * positions to unmask in this step.  Committing the tokens and updating the
 * mask stay with the caller; the token for a selected position is the argmax
 * returned by dlm_row_stats.
 *
 * Conventions shared by every entry point
 *  - Every data pointer is DEVICE memory owned by the caller.  The library
 *    never allocates, frees or synchronises; all work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream) and runs on the
 *    current CUDA device.
 *  - Argument errors are reported synchronously, before anything is launched:
 *    DLM_ERR_INVALID_ARG (null required pointer, negative or oversized size,
 *    bad parameter), DLM_ERR_ALIGNMENT (a base address or row stride that is
 *    not 16-byte aligned where the call says it must be), DLM_ERR_UNSUPPORTED
 *    (dtype not accepted by the call), DLM_ERR_WORKSPACE (workspace too
 *    small).  A failed launch returns DLM_ERR_CUDA.
 *  - Conditions found on the device never trap: they OR DLM_DEV_* bits into
 *    the caller's `dev_status` word (nullable: then they are not reported).
 *  - Positions are "block positions": sequence b, position i of its active
 *    block is row b*blk + i of every [batch][blk] array, and row b*blk + i of
 *    the logits.
 *  - Float decisions (threshold tests, orderings) are taken in fp32 on the
 *    values the caller passes; DAPD's graph decisions are exact (see there).
 *  - Sizes: 1 <= blk <= 256 for the selection calls; a batch of 0 is a no-op;
 *    CAP and DAPD take at most DLM_MAX_BATCH sequences per call (their grids
 *    hold up to 2048 CTAs per sequence), larger batches return
 *    DLM_ERR_INVALID_ARG.
 */
#ifndef DLM_H
#define DLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers */
typedef struct CUstream_st* dlm_stream_t;

typedef enum dlm_status {
    DLM_OK = 0,
    DLM_ERR_INVALID_ARG = 1,
    DLM_ERR_ALIGNMENT = 2,
    DLM_ERR_UNSUPPORTED = 3,
    DLM_ERR_WORKSPACE = 4,
    DLM_ERR_CUDA = 5
} dlm_status;

typedef enum dlm_dtype { DLM_F32 = 0, DLM_BF16 = 1, DLM_F16 = 2 } dlm_dtype;

/* device status bits (OR-ed into *dev_status by the kernels) */
#define DLM_DEV_NONFINITE 1u    /* a logit row held NaN or +inf, or only -inf   */
#define DLM_DEV_POOL_CLIPPED 2u /* a CAP pool had more than p_max candidates    */
#define DLM_DEV_TIMEOUT 4u      /* a kernel's bounded wait for its own copies gave
                                   up (~1 s); that call's outputs are unspecified */
#define DLM_DEV_BAD_INDEX 8u    /* a row index outside [0, rows) was skipped: that
                                   row was neither read nor written (row pass), or
                                   its pairs scored NaN (CAP) */

/* Maximum block size accepted by the selection calls. */
#define DLM_MAX_BLK 256
#define DLM_MAX_BATCH 1048575 /* 2^20 - 1: CAP / DAPD launch grids stay below 2^31 CTAs */

/* Human-readable name of a status code (static string, never NULL). */
const char* dlm_status_string(dlm_status s);

/* Library version: major*10000 + minor*100 + patch. */
int dlm_version(void);

/*
 * dlm_row_stats -- one fused streaming pass over each vocab-wide logit row.
 *
 * Defines (DepCap, "Methodology": I_k = KL(p_curr^k || p_prev^k),
 * H_k = H(p_curr^k), c_i = max_v p_i(v); Fast-dLLM review, "Method":
 * max-softmax confidence), with p = softmax(z) at temperature 1 and natural
 * logarithms:
 *   argmax[q]   = smallest v with z_v = max_v z_v (exact on stored values)
 *   conf[q]     = max_v p_v
 *   lse[q]      = log sum_v exp z_v
 *   entropy[q]  = -sum_v p_v log p_v
 *   kl[q]       = sum_v p_v (log p_v - log p'_v)   p' = softmax(prev row)
 *   lse_prev[q] = log sum_v exp z'_v
 *
 * cur, prev   : logit rows, element (q, v) at base + q*row_stride + v, dtype
 *               DLM_F32, DLM_BF16 or DLM_F16.  Base 16-byte aligned and
 *               row_stride*sizeof(dtype) a multiple of 16 (DLM_ERR_ALIGNMENT
 *               otherwise).  prev is nullable: then kl / lse_prev are not
 *               written.  -inf logits are allowed and carry probability 0.
 * n_rows      : number of rows to process (0 = nothing).
 * vocab       : row length V, 1 <= V <= row_stride, V < 2^31.
 * row_index   : nullable int32[n_rows]; row r processed is q = row_index[r]
 *               (else q = r).  Results are stored at index q, so the output
 *               arrays must hold max(q)+1 entries; entries of rows not
 *               processed are left unchanged.  An entry q < 0 is skipped (no
 *               read, no write) and sets DLM_DEV_BAD_INDEX; the upper bound
 *               is checked only by dlm_row_stats_ex (n_src_rows).
 * argmax      : int32 output (a row holding only NaN gets 0); conf, lse,
 *               entropy: float outputs (required).
 * kl, lse_prev: float outputs, nullable (ignored when prev is NULL).
 * dev_status  : nullable; DLM_DEV_NONFINITE is set for a row holding NaN or
 *               +inf (its outputs are then unspecified).
 */
dlm_status dlm_row_stats(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows,
                         int64_t vocab, int64_t row_stride, const int32_t* row_index,
                         int32_t* argmax, float* conf, float* lse, float* entropy, float* kl,
                         float* lse_prev, uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_row_stats_launches -- how many kernel launches dlm_row_stats_ex makes
 * for these sizes and flags (1, or 2 when the rows left over after whole
 * waves of the GPU run as half rows in a second grid that overlaps the first
 * one's last wave); 0 for no rows, -1 for arguments the call would reject.
 * Reads device attributes of the current device; launches nothing.
 */
int32_t dlm_row_stats_launches(dlm_dtype dtype, int32_t has_prev, int64_t n_rows, int64_t vocab,
                               uint32_t flags);

/*
 * dlm_row_stats_ex -- dlm_row_stats with a source-row bound and launch flags
 * (same definitions):
 *   n_src_rows            rows that cur and prev hold (0 = not checked).  With
 *                         row_index, an entry q >= n_src_rows is skipped like
 *                         a negative one (DLM_DEV_BAD_INDEX); without it,
 *                         n_rows > n_src_rows is DLM_ERR_INVALID_ARG.
 *   DLM_ROWS_SINGLE_GRID  never run the rows past whole waves as a second grid
 *                         of half rows.  The second grid fills the first one's
 *                         draining wave; when another kernel is meant to take
 *                         those slots (a lower-priority stream started with
 *                         the pass), one grid leaves them to it.
 *   DLM_ROWS_GATHER       store row r's results at index r instead of
 *                         q = row_index[r]: the outputs are [n_rows] arrays
 *                         of the gathered rows (e.g. a window of rows
 *                         cursor_b + k of a longer generation, in window
 *                         order).  A skipped row leaves its outputs unchanged.
 */
#define DLM_ROWS_SINGLE_GRID 1u
#define DLM_ROWS_GATHER 2u

dlm_status dlm_row_stats_ex(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows, int64_t vocab,
                            int64_t row_stride, const int32_t* row_index, int64_t n_src_rows, int32_t* argmax,
                            float* conf, float* lse, float* entropy, float* kl, float* lse_prev,
                            uint32_t* dev_status, uint32_t flags, dlm_stream_t stream);

/*
 * dlm_row_stats_partial / dlm_row_stats_merge -- dlm_row_stats over a row
 * whose vocabulary is split into slices (e.g. the vocab shards of a
 * tensor-parallel model, one per GPU).
 *
 * dlm_row_stats_partial reads one slice of every row -- element (q, v) at
 * cur + q*row_stride + v for 0 <= v < vocab, global position vocab_offset + v
 * -- and writes its partial state to partial[q].  dlm_row_stats_merge merges
 * the partial states of n_shards slices of the same rows (slice s of row q at
 * partials[s*shard_stride + q], merged in slice order) and writes exactly the
 * outputs dlm_row_stats writes for the whole row, with the same definitions
 * (argmax: smallest global position of the maximum).  Exchanging the 32-byte
 * states (an all-gather over the shards) is the only communication the split
 * needs.  Alignment, row_index and dtype rules are those of dlm_row_stats (the
 * slice's first element must be 16-byte aligned); a slice without a finite
 * maximum is allowed (it contributes nothing), and the merge raises
 * DLM_DEV_NONFINITE as dlm_row_stats does.  In the merge, a row index outside
 * [0, shard_stride) is skipped and sets DLM_DEV_BAD_INDEX.  has_prev in the merge says whether
 * the partial states were computed with prev (kl / lse_prev outputs).
 */
typedef struct dlm_row_partial {
    float mx;                /* maximum of the slice's logits (-inf clamped) */
    int32_t idx;             /* first global position of mx */
    float ref;               /* softmax reference of the sums below */
    float S, T, K;           /* sum 2^a, sum 2^a a, sum 2^a (z - z'); a = (z - ref) log2 e */
    float ref_prev, S_prev;  /* the previous row's reference and sum */
} dlm_row_partial;

dlm_status dlm_row_stats_partial(const void* cur, const void* prev, dlm_dtype dtype, int64_t n_rows,
                                 int64_t vocab, int64_t row_stride, const int32_t* row_index,
                                 int64_t vocab_offset, dlm_row_partial* partial, dlm_stream_t stream);

dlm_status dlm_row_stats_merge(const dlm_row_partial* partials, int32_t n_shards, int64_t shard_stride,
                               int64_t n_rows, const int32_t* row_index, int32_t has_prev, int32_t* argmax,
                               float* conf, float* lse, float* entropy, float* kl, float* lse_prev,
                               uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_select_threshold -- Fast-dLLM confidence-threshold decoding.
 *
 * Fast-dLLM review, "Method"; Fast-dLLM notes, "Key ideas" (safety valve):
 * selected[b][i] = masked[b][i] && conf[b][i] > tau; if that is empty for a
 * sequence with at least one masked position, the single masked position of
 * highest confidence is selected (ties to the lower position).
 *
 * conf [batch][blk] float, masked [batch][blk] uint8 (nonzero = masked),
 * selected [batch][blk] uint8 output (0/1), n_selected [batch] int32 output.
 */
dlm_status dlm_select_threshold(const float* conf, const uint8_t* masked, int32_t batch,
                                int32_t blk, float tau, uint8_t* selected, int32_t* n_selected,
                                dlm_stream_t stream);

/*
 * dlm_select_topk -- fixed top-K per step (the LLaDA default that Fast-dLLM
 * compares against; Fast-dLLM review, "Prior limitations": K tokens are
 * committed every step whatever their confidence).  Selects the min(k, masked)
 * masked positions of highest confidence, ties to the lower position.
 * Arrays as in dlm_select_threshold; k >= 0.
 */
dlm_status dlm_select_topk(const float* conf, const uint8_t* masked, int32_t batch, int32_t blk, int32_t k,
                           uint8_t* selected, int32_t* n_selected, dlm_stream_t stream);

/*
 * dlm_select_factor -- Fast-dLLM factor decoding (Fast-dLLM review,
 * "Method", appendix variant).  With c^(1) >= c^(2) >= ... the confidences of
 * the masked positions in decreasing order, the n* most confident positions
 * are selected, n* the largest n with (n + 1)(1 - c^(n)) < f (evaluated in
 * fp32; the qualifying n form a prefix).  If no n qualifies, the single most
 * confident masked position is selected (reading: the threshold rule's
 * progress guarantee).  Arrays as in dlm_select_threshold.
 */
dlm_status dlm_select_factor(const float* conf, const uint8_t* masked, int32_t batch, int32_t blk, float f,
                             uint8_t* selected, int32_t* n_selected, dlm_stream_t stream);

/*
 * dlm_parallel_certificate -- the Theorem-1 condition of the Fast-dLLM review
 * ("Key idea"): committing the n selected positions in parallel yields the
 * same tokens as committing them one at a time greedily when each has
 * confidence above 1 - 1/(n+1).  certified[b] = 1 when every selected position
 * of sequence b satisfies conf > 1 - 1/(n+1) in fp32 (an empty selection is
 * certified), else 0.  conf [batch][blk], selected [batch][blk] uint8,
 * certified [batch] uint8 output.
 */
dlm_status dlm_parallel_certificate(const float* conf, const uint8_t* selected, int32_t batch, int32_t blk,
                                    uint8_t* certified, dlm_stream_t stream);

/*
 * dlm_depcap_boundary -- DepGA-Block: length of the next block.
 *
 * DepCap, "Methodology" and "Technical Contribution": over a window of
 * L_window future positions with KL influence I_k and entropy H_k,
 * smooth both and normalise them within the window, form S_k = I~_k - lambda H~_k, stop
 * before the first S_k < 0 and clip the length to [L_min, L_window]; a cold
 * start uses L_min.  Readings of the unstated operators:
 *   smooth_w  : centred moving average of odd width (1 = none); at the
 *               window edges the neighbours that exist are averaged.
 *   norm_mode : 0 = divide by the window mean (floored at 1e-12),
 *               1 = rescale by window min/max to [0,1], 2 = none.
 *   length    = min(max(k*, L_min), L_window), k* = first k with S_k < 0
 *               (fp32 test) or L_window if none; cold start: min(L_min, L_window).
 * L_window = min(L_max, L_remain) is the caller's choice.
 *
 * kl, entropy : float [batch][L_window] (k-th future position of sequence b
 *               at b*L_window + k), 1 <= L_window <= 1024.
 * cold_start  : nullable uint8 [batch].
 * block_len   : int32 [batch] output.
 * score       : nullable float [batch][L_window] output (S_k).
 */
typedef struct dlm_depcap_params {
    float lambda;
    int32_t L_min;     /* >= 1 */
    int32_t smooth_w;  /* odd, 1..63 */
    int32_t norm_mode; /* 0, 1 or 2 */
} dlm_depcap_params;

dlm_status dlm_depcap_boundary(const float* kl, const float* entropy, int32_t batch,
                               int32_t L_window, const uint8_t* cold_start,
                               const dlm_depcap_params* params, int32_t* block_len,
                               float* score, dlm_stream_t stream);

/*
 * dlm_depcap_boundary_ragged -- dlm_depcap_boundary for a batch whose windows
 * differ in length: L_window = min(L_max, L_remain) is per sequence (DepCap,
 * "Methodology"), and sequences near the end of their generation have fewer
 * future positions than L_max.
 *
 * kl, entropy : float [batch][L_stride]; sequence b uses its first
 *               window_len[b] entries, exactly as dlm_depcap_boundary with
 *               L_window = window_len[b] would.  1 <= L_stride <= 1024.
 * window_len  : int32 [batch], required; values are clamped to [0, L_stride].
 *               A window of 0 gives block_len[b] = 0 (nothing left).
 * score       : nullable float [batch][L_stride]; entries at k >= window_len[b]
 *               are not written.
 * Other arguments and errors as dlm_depcap_boundary.
 */
dlm_status dlm_depcap_boundary_ragged(const float* kl, const float* entropy, int32_t batch, int32_t L_stride,
                                      const int32_t* window_len, const uint8_t* cold_start,
                                      const dlm_depcap_params* params, int32_t* block_len, float* score,
                                      dlm_stream_t stream);

/*
 * dlm_cap_select -- DepCap CAP-Decoding (conflict-aware parallel decoding).
 *
 * DepCap, "Methodology"; defaults in "Experiments" (tau_low 0.8, tau_high
 * 0.95, gamma -16).  Within the first scope_len[b] positions of the block:
 *   pool  = masked positions with conf >= tau_low, ordered by confidence
 *           (descending, ties to the lower position), at most p_max kept
 *           (DLM_DEV_POOL_CLIPPED when more qualified); the tau_high tier is
 *           the head of this order.
 *   D_ij  = log p_i(yhat_j) + log p_j(yhat_i),  log p_i(v) = z_i[v] - lse_i
 *   i, j conflict  <=>  D_ij > gamma
 *   greedy: scan the pool in order, keep a position iff it conflicts with no
 *   kept one.  high_tier_unconditional = 1 keeps every tier member first,
 *   then scans the rest.  Empty pool: the highest-confidence masked position
 *   of the scope (the page's fallback when nothing is safe to unmask).
 *
 * logits      : the current logit rows (as given to dlm_row_stats), stride
 *               row_stride elements; 16-byte alignment is not required
 *               (scattered 2-byte reads).
 * row_index   : nullable int32 [batch][blk]: position i of sequence b reads
 *               logit row row_index[b*blk + i] (NULL: row b*blk + i), so the
 *               block can be a window of a longer generation (rows
 *               cursor_b + k) without copying its rows.  A pool member whose
 *               row lies outside [0, n_rows) is not read: its pairs score NaN
 *               (no conflict) and DLM_DEV_BAD_INDEX is set.
 * n_rows      : number of rows the logits array holds, >= 1; without
 *               row_index it must be at least batch*blk.
 * argmax, conf, lse : [batch][blk] from dlm_row_stats.  A token outside
 *                     [0, vocab) is never read from the logits: its pairs
 *                     score NaN (no conflict) and DLM_DEV_NONFINITE is set.
 * masked      : uint8 [batch][blk].
 * scope_len   : nullable int32 [batch] (e.g. dlm_depcap_boundary's block_len);
 *               NULL = the whole block.
 * selected, n_selected : outputs as in dlm_select_threshold.
 * D_out       : nullable float [batch][blk][blk]; D_ij is written at [b][i][j]
 *               for every ordered pair of pool members; other entries are left
 *               unchanged.
 * workspace   : device scratch of at least dlm_cap_workspace_size(batch, p_max)
 *               bytes, 16-byte aligned, owned by the caller; its contents on
 *               entry do not matter.  Calls sharing a workspace must not
 *               overlap on the GPU.
 */
typedef struct dlm_cap_params {
    float tau_low;
    float tau_high;
    float gamma;
    int32_t p_max;                   /* 1..256 */
    int32_t high_tier_unconditional; /* 0 or 1 */
} dlm_cap_params;

size_t dlm_cap_workspace_size(int32_t batch, int32_t p_max);

dlm_status dlm_cap_select(const void* logits, dlm_dtype dtype, int64_t vocab, int64_t row_stride,
                          const int32_t* row_index, int64_t n_rows, const int32_t* argmax, const float* conf,
                          const float* lse,
                          const uint8_t* masked, const int32_t* scope_len, int32_t batch,
                          int32_t blk, const dlm_cap_params* params, uint8_t* selected,
                          int32_t* n_selected, float* D_out, void* workspace, size_t ws_bytes,
                          uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_row_stats_rules -- dlm_row_stats with the threshold, boundary and CAP
 * rules folded into the same launch.
 *
 * Computes exactly what these calls compute one after another on rows
 * b*blk + i (b < batch, i < blk): dlm_row_stats (no row index), then, for
 * the rules asked for in rules->rules, dlm_select_threshold(conf, masked,
 * tau), dlm_depcap_boundary(kl, entropy, L_window = blk, cold_start,
 * depcap) and dlm_cap_select(cur, no row index, argmax, conf, lse, masked,
 * scope = this call's block_len when cap_scope_from_boundary, else the
 * whole block; cap).  The rules of sequence b run in the CTA that writes the
 * last of b's rows (the one whose row completes b's count in the
 * workspace), so they overlap the rest of the row pass instead of following
 * it as separate launches; no CTA waits for another.  This is a library
 * arrangement with no counterpart on the pages (DepCap, "Methodology" and
 * the Fast-dLLM review, "Method", define the rules; dlm_row_stats,
 * dlm_select_threshold, dlm_depcap_boundary and dlm_cap_select cite them).
 *
 * cur, prev, dtype, vocab, row_stride : as dlm_row_stats (batch*blk rows;
 *                      prev is required for the boundary rule).
 * masked              : uint8 [batch][blk].
 * rules               : DLM_RULE_* bits and the rules' parameters (CAP:
 *                      p_max <= 64).
 * argmax .. lse_prev  : the row statistics, as dlm_row_stats ([batch*blk]).
 * thr_selected, thr_n_selected : threshold outputs (required with
 *                      DLM_RULE_THRESHOLD), as dlm_select_threshold.
 * block_len, score    : boundary outputs (block_len required with
 *                      DLM_RULE_BOUNDARY; score nullable [batch][blk]).
 * cap_selected, cap_n_selected : CAP outputs (required with DLM_RULE_CAP).
 * workspace           : dlm_row_stats_rules_workspace_size(batch) bytes,
 *                      16-byte aligned, ZERO before the first call (e.g.
 *                      one cudaMemsetAsync); every call leaves it zero.
 *                      Calls sharing a workspace must not overlap.
 * Sizes: 1 <= blk <= 256; batch*blk rows.
 */
#define DLM_RULE_THRESHOLD 1u
#define DLM_RULE_BOUNDARY 2u
#define DLM_RULE_CAP 4u

typedef struct dlm_step_rules {
    uint32_t rules;                  /* OR of DLM_RULE_* (at least one) */
    float tau;                       /* threshold rule */
    dlm_depcap_params depcap;        /* boundary rule */
    const uint8_t* cold_start;       /* boundary rule: nullable device [batch] */
    dlm_cap_params cap;              /* CAP rule: p_max 1..64 */
    int32_t cap_scope_from_boundary; /* 0 or 1 (needs DLM_RULE_BOUNDARY) */
} dlm_step_rules;

size_t dlm_row_stats_rules_workspace_size(int32_t batch);

dlm_status dlm_row_stats_rules(const void* cur, const void* prev, dlm_dtype dtype, int32_t batch, int32_t blk,
                               int64_t vocab, int64_t row_stride, const uint8_t* masked,
                               const dlm_step_rules* rules, int32_t* argmax, float* conf, float* lse,
                               float* entropy, float* kl, float* lse_prev, uint8_t* thr_selected,
                               int32_t* thr_n_selected, int32_t* block_len, float* score, uint8_t* cap_selected,
                               int32_t* cap_n_selected, void* workspace, size_t ws_bytes, uint32_t* dev_status,
                               dlm_stream_t stream);

/*
 * dlm_dapd_graph_mis -- DAPD: attention graph and Welsh-Powell selection.
 *
 * DAPD, "整体框架" and "关键设计 1-3".  V_t = masked positions of the block,
 * r = |V_t| / blk.
 *   r >= bulk_frac (fp32): a_ij = mean over the given layers and heads of
 *       attention[i][j]; s_ij = (a_ij + a_ji)/2; edge (i,j) <=> s_ij > tau_edge;
 *       d~_i = sum over j in V_t, j != i, of s_ij; key_i = d~_i * conf_i
 *       (order_mode 1: d~_i); scan V_t by key descending (ties to the lower
 *       position) keeping every node with no kept neighbour.
 *   r <  bulk_frac: select masked positions with conf > bulk_conf; if none,
 *       the highest-confidence masked one.
 * Which layers to average (the page uses roughly the last 30 %) is the
 * caller's choice: pass exactly those layers.  The per-pair sums are accumulated exactly in fixed point, so
 * the edge test and the key order are exact decisions when every attention
 * value is an f16 in [0, 256) and the sum over layers*heads of each entry
 * stays below 512 (true for softmax rows with layers*heads <= 511); other
 * inputs are summed with fp32-level accuracy.
 *
 * attn        : element (b, l, h, row, col) at
 *               attn + b*stride_b + l*stride_l + h*stride_h + row*stride_row + col
 *               (element strides); the block is rows and columns
 *               [block_start, block_start + blk).  dtype F16, BF16 or F32;
 *               the address of (b,l,h,block_start,block_start) and every
 *               stride must be 16-byte aligned.  Only masked rows are read.
 * masked, conf: [batch][blk].
 * selected, n_selected : outputs as in dlm_select_threshold.
 * s_out       : nullable float [batch][blk][blk]; s_ij for i, j in V_t.
 * dtilde_out  : nullable float [batch][blk]; d~_i for i in V_t.
 * deg_out     : nullable int32 [batch][blk]; number of tau-edges of i in V_t.
 *               (The three are written only for sequences on the graph path;
 *               other entries are left unchanged.)
 * workspace   : device scratch, at least dlm_dapd_workspace_size(batch, blk)
 *               bytes, 16-byte aligned; calls sharing it must not overlap.
 */
typedef struct dlm_dapd_params {
    float tau_edge;
    float bulk_conf;  /* 0.9 on the page */
    float bulk_frac;  /* 0.5 on the page */
    int32_t order_mode; /* 0: d~ * conf, 1: d~ (DAPD, 消融实验: the sort-key ablation) */
    int32_t preunmask_certain; /* 1: also select every masked position whose
                                  conf is exactly 1.0 in fp32 (DAPD, 关键设计 3,
                                  appendix remark: such a position can be
                                  unmasked at any time); the graph is unchanged */
} dlm_dapd_params;

size_t dlm_dapd_workspace_size(int32_t batch, int32_t blk);

dlm_status dlm_dapd_graph_mis(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                              int32_t n_heads, int64_t stride_b, int64_t stride_l,
                              int64_t stride_h, int64_t stride_row, int32_t block_start,
                              int32_t blk, const uint8_t* masked, const float* conf,
                              const dlm_dapd_params* params, uint8_t* selected,
                              int32_t* n_selected, float* s_out, float* dtilde_out,
                              int32_t* deg_out, void* workspace, size_t ws_bytes,
                              uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_dapd_graph_mis_noalloc -- dlm_dapd_graph_mis without a workspace.
 *
 * The pages have no counterpart to this call: it serves callers that cannot
 * allocate device memory, so cannot pass the DAPD workspace -- a serving
 * engine whose allocator reserved nearly all of HBM at start-up and hands out
 * nothing while decoding, a plug-in inside a framework that owns every
 * device allocation, a decode loop that must not pay cudaMalloc's implicit
 * device synchronisation.  It takes the arguments of dlm_dapd_graph_mis
 * except the workspace, gives the same results (it is that call with the
 * library's array as the workspace), and keeps the scratch -- the attention
 * pass's fixed-point sums, which the selection kernel reads back -- in one
 * array inside libdlm.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Limit: the array holds DLM_DAPD_NOALLOC_MAX_BYTES (8 MiB); a call whose
 * dlm_dapd_workspace_size(batch, blk) is larger returns DLM_ERR_WORKSPACE
 * before anything is launched (8 sequences of 256 positions need 4.3 MB and
 * fit; 16 of them do not).  The array exists on every GPU that loads the
 * library, until the process exits.
 * Set-up: the first call in a CUDA context looks up the array's device
 * address with that context's device current, and later calls reuse it (a
 * device reset starts a new context, whose first call looks it up again).
 * Make that first call on each device -- and the first after a reset --
 * before any stream capture.
 * Sharing: every call uses the same array and leaves its contents behind.
 * Nothing needs clearing between calls (a call writes every entry it reads
 * first), but calls that can overlap on the GPU -- other streams, other host
 * threads, concurrent graph branches -- race on the array and must be
 * ordered by the caller.
 */
#define DLM_DAPD_NOALLOC_MAX_BYTES (8u << 20)

dlm_status dlm_dapd_graph_mis_noalloc(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                                      int32_t n_heads, int64_t stride_b, int64_t stride_l, int64_t stride_h,
                                      int64_t stride_row, int32_t block_start, int32_t blk, const uint8_t* masked,
                                      const float* conf, const dlm_dapd_params* params, uint8_t* selected,
                                      int32_t* n_selected, float* s_out, float* dtilde_out, int32_t* deg_out,
                                      uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_dapd_graph / dlm_dapd_select -- dlm_dapd_graph_mis in two halves.
 *
 * The DAPD graph (a_ij, s_ij, tau-edges, d~, degrees) needs only the attention
 * and the mask, not the confidences, so it can be built on another stream
 * while dlm_row_stats reads the logits; the selection then needs conf.
 * dlm_dapd_graph takes the arguments of dlm_dapd_graph_mis except conf and the
 * selection outputs, and leaves in `workspace` what the selection needs: the
 * exact attention sums and the edge threshold (the selection rebuilds the
 * graph from the sums in its own launch); s_out / dtilde_out /
 * deg_out are written when given.
 * dlm_dapd_select reads that graph and conf and writes the selection exactly
 * as dlm_dapd_graph_mis does (late-phase sequences are decided from conf
 * alone).  The two calls must see the same batch, blk, masked, params and
 * workspace, and the caller orders them (same stream, or an event).
 */
dlm_status dlm_dapd_graph(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers, int32_t n_heads,
                          int64_t stride_b, int64_t stride_l, int64_t stride_h, int64_t stride_row,
                          int32_t block_start, int32_t blk, const uint8_t* masked, const dlm_dapd_params* params,
                          float* s_out, float* dtilde_out, int32_t* deg_out, void* workspace, size_t ws_bytes,
                          uint32_t* dev_status, dlm_stream_t stream);

dlm_status dlm_dapd_select(const uint8_t* masked, const float* conf, int32_t batch, int32_t blk,
                           const dlm_dapd_params* params, uint8_t* selected, int32_t* n_selected,
                           void* workspace, size_t ws_bytes, dlm_stream_t stream);

/*
 * dlm_row_stats_attention -- dlm_row_stats and dlm_dapd_graph in one pass.
 *
 * The pages give no such operation: it is the row statistics of the
 * Fast-dLLM review ("Method") and DepCap ("Methodology") over rows
 * b*blk + i, plus the DAPD attention sums of every masked row (DAPD,
 * "关键设计 1"), computed by the same CTAs.  Where the rows are too few to
 * fill the GPU (each row is split over a cluster of CTAs), the CTA holding
 * the start of row b*blk + i copies row i of sequence b's attention block,
 * for every layer and head, into shared memory while the cluster streams the
 * logits, then sums it exactly into the DAPD workspace: the scattered
 * attention reads wait under the logit stream instead of in a latency-bound
 * pass beside it.  With whole waves of rows the scattered reads cost the
 * same DRAM time either way and a separate attention pass beside the row
 * pass is faster, so the call then runs the row pass and the attention pass
 * one after the other on the stream (as it does when the attention is not
 * foldable: a block row that is not whole 16-byte vectors, or more copied
 * attention than fits 48 KB of shared memory).  Either way,
 * dlm_dapd_select(masked, conf, ...) on the workspace afterwards gives
 * exactly the selection dlm_dapd_graph followed by dlm_dapd_select gives.
 *
 * Arguments: those of dlm_row_stats_ex for n_rows = batch * blk rows with no
 * row index (row b*blk + i is position i of sequence b), then those of
 * dlm_dapd_graph (attention view, block, mask, params, workspace, status)
 * without the float outputs.  Layouts, alignment rules and errors are
 * theirs.  dlm_row_stats_attention_folds returns 1 when the call folds the
 * attention into the row pass for these shapes, 0 otherwise (including
 * invalid arguments); it launches nothing.
 */
int32_t dlm_row_stats_attention_folds(dlm_dtype dtype, int32_t batch, int32_t blk, int64_t vocab,
                                      dlm_dtype attn_dtype, int32_t n_layers, int32_t n_heads);

dlm_status dlm_row_stats_attention(const void* cur, const void* prev, dlm_dtype dtype, int32_t batch, int32_t blk,
                                   int64_t vocab, int64_t row_stride, int32_t* argmax, float* conf, float* lse,
                                   float* entropy, float* kl, float* lse_prev, const void* attn,
                                   dlm_dtype attn_dtype, int32_t n_layers, int32_t n_heads, int64_t stride_b,
                                   int64_t stride_l, int64_t stride_h, int64_t stride_row, int32_t block_start,
                                   const uint8_t* masked, const dlm_dapd_params* params, void* workspace,
                                   size_t ws_bytes, uint32_t* dev_status, dlm_stream_t stream);

/*
 * dlm_attention_influence -- downstream influence of every block position,
 * an input of dlm_revocable_step's seed score.
 *
 * COVER page, "Method": a seed's score combines its uncertainty, its
 * downstream influence and its cache drift; the page does not define
 * influence.  Reading: the attention position i receives from the positions
 * still to be decoded (the masked queries q of the block), averaged over the
 * given layers and heads:
 *   influence[b][i] = (1 / (L H)) sum_{q masked} sum_{l,h} attention[q][i]
 * for every position i of the block.  The sums are the DAPD attention pass's
 * exact fixed-point sums (dlm_dapd_graph_mis describes the exactness), taken
 * for every sequence whatever its masked fraction, then summed over the
 * masked rows exactly and rounded once to fp32.
 *
 * Arguments as dlm_dapd_graph_mis for attn, dtype, sizes, strides,
 * block_start, blk, masked and workspace (dlm_dapd_workspace_size bytes; the
 * call overwrites it); influence: float [batch][blk] output.
 */
dlm_status dlm_attention_influence(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                                   int32_t n_heads, int64_t stride_b, int64_t stride_l, int64_t stride_h,
                                   int64_t stride_row, int32_t block_start, int32_t blk, const uint8_t* masked,
                                   float* influence, void* workspace, size_t ws_bytes, uint32_t* dev_status,
                                   dlm_stream_t stream);

/*
 * dlm_revocable_step -- one state update of revocable parallel decoding
 * (COVER page: "Revocable Parallel Diffusion Decoding" for the step and its
 * state update, "Method" for the three revision outcomes, stability-aware
 * seed selection and the seed count |S_t| = ceil(sqrt(n_t) pi_t)).
 *
 * Per sequence b (one block of blk <= 256 positions), with yhat_i / c_i the
 * model's prediction and confidence at position i this step (for a seed:
 * its leave-one-out re-prediction), in this order:
 *  0. a sequence with no masked position at the start of the step has
 *     finished (the decode terminates when nothing is masked): nothing
 *     changes, outcome 0, counts 0.
 *  1. verify every seed (seed_i = 1 and decoded):
 *       KEEP    (2) if yhat_i == tok_i;
 *       REPLACE (3) if yhat_i != tok_i and c_i >= tau_replace: tok_i = yhat_i;
 *       REMASK  (4) otherwise: masked_i = 1, last_tok_i = tok_i, tok_i = -1,
 *                   remasks_i += 1.
 *  2. draft among the positions masked at the start of the step: those with
 *     c_i > tau_draft, most confident first (ties to the lower position), at
 *     most draft_budget of them (<= 0: no cap); if none qualifies, the single
 *     most confident one.  Drafted (1): tok_i = yhat_i, masked_i = 0; a
 *     drafted token equal to last_tok_i is a flip-flop (flipflops[b] += 1).
 *  3. choose the next step's seeds: eligible = decoded after 1-2, step -
 *     last_seed_i > cooldown, remasks_i < remask_budget.  With n eligible,
 *     k = min(n, ceil(sqrt(n) * pi)) (fp32); score_i = w_unc (1 - c_i) +
 *     w_infl infl_i - w_drift drift_i (fp32, each product and sum rounded,
 *     no fused multiply-add); the k best scores (ties to the lower position)
 *     get seed_i = 1 and last_seed_i = step, all others seed_i = 0.
 * Every comparison and the score are taken in fp32.
 *
 * Readings (the pages leave these open): KEEP / REPLACE / REMASK are decided
 * by the prediction matching the token and a confidence threshold; the
 * drafting rule is the confidence threshold with the top-1 fallback under an
 * optional budget; uncertainty is 1 - c_i, downstream influence and cache
 * drift are supplied by the caller (nullable: 0), the score is their linear
 * combination with weights w_*; the revision rate pi_t is the constant pi and
 * n_t the number of eligible positions.
 *
 * argmax, conf        : [batch][blk] int32 / float, this step's yhat, c.
 * influence, drift    : nullable float [batch][blk].
 * tok                 : int32 [batch][blk] in/out (-1 at masked positions).
 * masked, seed        : uint8 [batch][blk] in/out.
 * last_seed, remasks,
 * last_tok            : int32 [batch][blk] in/out state; start a decode with
 *                       last_seed = INT32_MIN / 2, remasks = 0, last_tok = -1.
 * outcome             : nullable uint8 [batch][blk] output (0 none, 1 drafted,
 *                       2 keep, 3 replace, 4 remask).
 * n_drafted, n_revoked: nullable int32 [batch] outputs (net growth of the
 *                       decoded set = drafted - revoked).
 * flipflops           : nullable int32 [batch], accumulated.
 * Errors: DLM_ERR_INVALID_ARG for a null required pointer, batch < 0,
 * blk outside [1, 256], pi or a weight not finite, pi < 0.
 */
typedef struct dlm_revocable_params {
    float tau_replace;     /* REPLACE threshold on c_i */
    float tau_draft;       /* drafting threshold (strict) */
    int32_t draft_budget;  /* <= 0: no cap */
    float w_unc, w_infl, w_drift;
    float pi;              /* seed rate: k = ceil(sqrt(n) * pi) */
    int32_t cooldown;      /* eligible iff step - last_seed > cooldown */
    int32_t remask_budget; /* eligible iff remasks < remask_budget */
} dlm_revocable_params;

dlm_status dlm_revocable_step(const int32_t* argmax, const float* conf, const float* influence, const float* drift,
                              int32_t batch, int32_t blk, int32_t step, const dlm_revocable_params* params,
                              int32_t* tok, uint8_t* masked, uint8_t* seed, int32_t* last_seed, int32_t* remasks,
                              int32_t* last_tok, uint8_t* outcome, int32_t* n_drafted, int32_t* n_revoked,
                              int32_t* flipflops, dlm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DLM_H */
