/*
 * dlm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement, in fp64, of what the per-step unmask
 * decision of a masked diffusion LM computes.  Only the test-suite, the
 * package smoke check and the CPU-baseline leg of the benchmark may load
 * this file; the product path never does.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (web pages on training-free parallel decoding):
 *  - "DepCap: Adaptive Block-Wise Parallel Decoding for Efficient Diffusion
 *    LM Inference", section Methodology: KL influence, entropy, the
 *    DepGA-Block score and boundary, CAP-Decoding pool, conflict score and
 *    greedy selection; section Experiments: default thresholds.
 *  - "Fast-dLLM: Training-Free Acceleration of Diffusion LLMs via KV Cache
 *    and Parallel Decoding" (review), section Method: max-softmax confidence,
 *    threshold decoding with a top-confidence fallback.
 *  - "DAPD: Dependency-Aware Parallel Decoding via Attention for Diffusion
 *    LLMs", sections 整体框架 and 关键设计 1-3: attention averaging, the
 *    symmetrised score, the tau-graph, the proxy degree, the Welsh-Powell
 *    greedy independent set and the late-phase confidence rule.
 *
 * Every decision that turns a float into an integer (a threshold test, an
 * ordering) is taken in the precision of the GPU kernel that mirrors it:
 * fp32 for confidence, score and conflict tests; the DAPD graph decisions
 * (edge test, key order) are exact in the kernel and are taken here in fp64.
 * Where the pages leave a step open, the reading taken is stated beside it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

int oracle_version(void) { return 1; }

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- storage decoding: exact widening of the stored value to fp64 ---- */

static double dec_bf16(uint16_t b) {
    /* bf16 is the top half of an IEEE binary32 */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dec_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 31;
    int man = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24); /* subnormal */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man + 1024), ex - 25);
    return sign ? -v : v;
}

static double load_elem(const void* base, int dtype, int64_t i) {
    switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_BF16: return dec_bf16(((const uint16_t*)base)[i]);
    default: return dec_f16(((const uint16_t*)base)[i]);
    }
}

/* ------------------------------------------------------------------------
 * Row statistics of one vocab-wide logit row (DepCap, Methodology: I_k is
 * KL(p_curr || p_prev), H_k the entropy of p_curr, c_i = max_v p_i(v);
 * Fast-dLLM, Method: max-softmax confidence).  Softmax temperature 1,
 * natural logarithms, argmax ties to the lowest vocab index.
 *
 * Straight from the definitions, three passes:
 *   m   = max_v z_v,            yhat = smallest v with z_v = m
 *   lse = m + log sum_v exp(z_v - m)
 *   p_v = exp(z_v - lse)
 *   conf = max_v p_v,  H = -sum_v p_v log p_v   (0 log 0 = 0)
 *   KL  = sum_v p_v (log p_v - log q_v),  q from the previous row
 * ------------------------------------------------------------------------ */
static void row_one(const void* cur, const void* prev, int dtype, int64_t vocab,
                    int64_t off, int32_t* argmax, double* conf, double* lse,
                    double* entropy, double* kl, double* lse_prev) {
    double m = -INFINITY;
    int64_t yhat = 0;
    for (int64_t v = 0; v < vocab; ++v) {
        double z = load_elem(cur, dtype, off + v);
        if (z > m) { m = z; yhat = v; }
    }
    double s = 0.0;
    for (int64_t v = 0; v < vocab; ++v) s += exp(load_elem(cur, dtype, off + v) - m);
    double L = m + log(s);

    double Lq = 0.0;
    if (prev) {
        double mq = -INFINITY;
        for (int64_t v = 0; v < vocab; ++v) {
            double z = load_elem(prev, dtype, off + v);
            if (z > mq) mq = z;
        }
        double sq = 0.0;
        for (int64_t v = 0; v < vocab; ++v) sq += exp(load_elem(prev, dtype, off + v) - mq);
        Lq = mq + log(sq);
    }

    double pmax = 0.0, h = 0.0, d = 0.0;
    for (int64_t v = 0; v < vocab; ++v) {
        double logp = load_elem(cur, dtype, off + v) - L;
        double p = exp(logp);
        if (p > pmax) pmax = p;
        if (p == 0.0) continue;
        h -= p * logp;
        if (prev) {
            double logq = load_elem(prev, dtype, off + v) - Lq;
            d += p * (logp - logq);
        }
    }
    *argmax = (int32_t)yhat;
    *conf = pmax;
    *lse = L;
    *entropy = h;
    if (prev) {
        if (kl) *kl = d;
        if (lse_prev) *lse_prev = Lq;
    }
}

/* Rows r = 0..n_rows-1 read row q = row_index[r] (or r) of cur/prev and
 * write their statistics at index q. */
void oracle_row_stats(const void* cur, const void* prev, int dtype, int64_t n_rows,
                      int64_t vocab, int64_t row_stride, const int32_t* row_index,
                      int32_t* argmax, double* conf, double* lse, double* entropy,
                      double* kl, double* lse_prev) {
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n_rows; ++r) {
        int64_t q = row_index ? row_index[r] : r;
        row_one(cur, prev, dtype, vocab, q * row_stride, argmax + q, conf + q, lse + q,
                entropy + q, kl ? kl + q : NULL, lse_prev ? lse_prev + q : NULL);
    }
}

/* Highest-confidence masked position among [0, n): ties to the lower index,
 * compared in fp32.  Returns -1 when nothing is masked. */
static int top_conf(const double* conf, const uint8_t* masked, int n) {
    int best = -1;
    float bc = 0.0f;
    for (int i = 0; i < n; ++i) {
        if (!masked[i]) continue;
        float c = (float)conf[i];
        if (best < 0 || c > bc) { best = i; bc = c; }
    }
    return best;
}

/* ------------------------------------------------------------------------
 * Fast-dLLM threshold decoding (Fast-dLLM review, Method; blog notes, Key
 * ideas): commit every masked position whose confidence exceeds tau; if
 * none does, commit the single highest-confidence masked position.
 * "Exceeds" is read as strict >.
 * ------------------------------------------------------------------------ */
void oracle_select_threshold(const double* conf, const uint8_t* masked, int batch, int blk,
                             float tau, uint8_t* selected, int32_t* n_selected) {
    for (int b = 0; b < batch; ++b) {
        const double* c = conf + (int64_t)b * blk;
        const uint8_t* mk = masked + (int64_t)b * blk;
        uint8_t* sel = selected + (int64_t)b * blk;
        int n = 0;
        for (int i = 0; i < blk; ++i) {
            sel[i] = (uint8_t)(mk[i] && (float)c[i] > tau);
            n += sel[i];
        }
        if (n == 0) {
            int t = top_conf(c, mk, blk);
            if (t >= 0) { sel[t] = 1; n = 1; }
        }
        n_selected[b] = n;
    }
}

/* ------------------------------------------------------------------------
 * DepGA-Block boundary (DepCap, Methodology and Technical Contribution).
 * I_k, H_k for the k-th future position; the unspecified smoothing and
 * local normalisation are read as a centred moving average of odd width w (edges average the
 * neighbours that exist) followed by a window-local normalisation:
 * norm_mode 0 divides by the window mean (floored at 1e-12), 1 rescales to
 * [0,1] by the window min and max, 2 leaves the values as they are.
 * S_k = I~_k - lambda H~_k; the boundary stops before the first S_k < 0
 * (fp32 sign test), the length is clipped to [L_min, L_window]
 * (min(max(k*, L_min), L_window)), and a cold start returns L_min.
 * ------------------------------------------------------------------------ */
static void smooth_norm(const double* x, int n, int w, int mode, double* out) {
    int h = w / 2;
    double* sm = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int k = 0; k < n; ++k) {
        int lo = k - h < 0 ? 0 : k - h;
        int hi = k + h > n - 1 ? n - 1 : k + h;
        double acc = 0.0;
        for (int j = lo; j <= hi; ++j) acc += x[j];
        sm[k] = acc / (double)(hi - lo + 1);
    }
    if (mode == 0) {
        double mean = 0.0;
        for (int k = 0; k < n; ++k) mean += sm[k];
        mean /= (double)n;
        if (mean < 1e-12) mean = 1e-12;
        for (int k = 0; k < n; ++k) out[k] = sm[k] / mean;
    } else if (mode == 1) {
        double mn = sm[0], mx = sm[0];
        for (int k = 1; k < n; ++k) {
            if (sm[k] < mn) mn = sm[k];
            if (sm[k] > mx) mx = sm[k];
        }
        for (int k = 0; k < n; ++k) out[k] = mx > mn ? (sm[k] - mn) / (mx - mn) : 0.0;
    } else {
        for (int k = 0; k < n; ++k) out[k] = sm[k];
    }
    free(sm);
}

void oracle_depcap_boundary(const double* kl, const double* entropy, int batch, int L_window,
                            const int32_t* window_len, const uint8_t* cold_start, float lambda,
                            int L_min, int smooth_w, int norm_mode, int32_t* block_len, double* score) {
    double* In = (double*)malloc(sizeof(double) * (size_t)L_window);
    double* Hn = (double*)malloc(sizeof(double) * (size_t)L_window);
    for (int b = 0; b < batch; ++b) {
        /* L_window = min(L_max, L_remain) per sequence when window_len is given;
         * the rows keep the stride L_window */
        int L = L_window;
        if (window_len) {
            L = window_len[b] < 0 ? 0 : window_len[b];
            if (L > L_window) L = L_window;
        }
        if (L == 0) {
            block_len[b] = 0;
            continue;
        }
        const double* I = kl + (int64_t)b * L_window;
        const double* H = entropy + (int64_t)b * L_window;
        smooth_norm(I, L, smooth_w, norm_mode, In);
        smooth_norm(H, L, smooth_w, norm_mode, Hn);
        int kstar = L;
        for (int k = 0; k < L; ++k) {
            double s = In[k] - (double)lambda * Hn[k];
            if (score) score[(int64_t)b * L_window + k] = s;
            if (kstar == L && (float)s < 0.0f) kstar = k;
        }
        int len = kstar < L_min ? L_min : kstar;
        if (len > L) len = L;
        if (cold_start && cold_start[b]) len = L_min < L ? L_min : L;
        block_len[b] = len;
    }
    free(In);
    free(Hn);
}

/* ------------------------------------------------------------------------
 * CAP-Decoding (DepCap, Methodology; defaults from Experiments and the
 * executive summary).  Inside the block the boundary rule chose (positions
 * [0, scope)):
 *   pool  = masked positions with c_i >= tau_low (fp32 test), ordered by
 *           confidence, ties to the lower position; at most p_max kept.
 *           The tau_high tier is the head of this order.
 *   D_ij  = log p_i(yhat_j) + log p_j(yhat_i), log p_i(v) = z_i[v] - lse_i
 *   conflict(i,j) <=> D_ij > gamma (fp32 test)
 *   greedy: scan the pool in order and keep i iff it conflicts with no
 *           kept j.  Variant high_tier_unconditional: every tier member is
 *           kept first, then the rest are scanned.
 *   no pool -> the highest-confidence masked position of the scope.
 * Outputs the selection, the pool (in order) and D over pool pairs
 * (D[i][j] at block positions; NaN elsewhere).  Returns 1 when the pool was
 * clipped at p_max.  Position i of sequence b reads logit row
 * row_index[b*blk + i] when row_index is given (the block as a window of a
 * longer generation), else row b*blk + i.
 * ------------------------------------------------------------------------ */
static int conf_before(const double* c, int a, int b) {
    float ca = (float)c[a], cb = (float)c[b];
    if (ca != cb) return ca > cb;
    return a < b;
}

int oracle_cap_select(const void* logits, int dtype, int64_t row_stride, const int32_t* row_index,
                      const int32_t* argmax, const double* conf, const double* lse,
                      const uint8_t* masked, const int32_t* scope_len, int batch, int blk,
                      float tau_low, float tau_high, float gamma, int p_max,
                      int high_tier_unconditional, uint8_t* selected, int32_t* n_selected,
                      double* D, int32_t* pool_out, int32_t* pool_n_out) {
    int clipped_any = 0;
    int b;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : clipped_any)
    for (b = 0; b < batch; ++b) {
        int64_t base = (int64_t)b * blk;
        const double* c = conf + base;
        const uint8_t* mk = masked + base;
        uint8_t* sel = selected + base;
        int scope = blk;
        if (scope_len && scope_len[b] < scope) scope = scope_len[b];
        if (scope < 0) scope = 0;
        int* pool = (int*)malloc(sizeof(int) * (size_t)blk);
        int n = 0;
        for (int i = 0; i < scope; ++i)
            if (mk[i] && (float)c[i] >= tau_low) pool[n++] = i;
        /* insertion sort by (conf desc, position asc) */
        for (int a = 1; a < n; ++a) {
            int x = pool[a], k = a - 1;
            while (k >= 0 && conf_before(c, x, pool[k])) { pool[k + 1] = pool[k]; --k; }
            pool[k + 1] = x;
        }
        if (n > p_max) { n = p_max; clipped_any = 1; }
        for (int i = 0; i < blk; ++i) sel[i] = 0;
        if (D)
            for (int64_t e = 0; e < (int64_t)blk * blk; ++e) D[(int64_t)b * blk * blk + e] = NAN;
        if (pool_out) {
            for (int k = 0; k < blk; ++k) pool_out[base + k] = k < n ? pool[k] : -1;
        }
        if (pool_n_out) pool_n_out[b] = n;

        if (n == 0) {
            int t = top_conf(c, mk, scope);
            if (t >= 0) sel[t] = 1;
            n_selected[b] = t >= 0 ? 1 : 0;
            free(pool);
            continue;
        }
        /* conflict matrix over pool slots */
        uint8_t* conf_mat = (uint8_t*)calloc((size_t)n * n, 1);
        for (int a = 0; a < n; ++a) {
            int i = pool[a];
            int64_t ri = (row_index ? (int64_t)row_index[base + i] : base + i) * row_stride;
            for (int e = 0; e < n; ++e) {
                if (e == a) continue;
                int j = pool[e];
                int64_t rj = (row_index ? (int64_t)row_index[base + j] : base + j) * row_stride;
                double lpi = load_elem(logits, dtype, ri + argmax[base + j]) - lse[base + i];
                double lpj = load_elem(logits, dtype, rj + argmax[base + i]) - lse[base + j];
                double d = lpi + lpj;
                if (D) D[(int64_t)b * blk * blk + (int64_t)i * blk + j] = d;
                conf_mat[(int64_t)a * n + e] = (uint8_t)((float)d > gamma);
            }
        }
        uint8_t* kept = (uint8_t*)calloc((size_t)n, 1);
        uint8_t* blocked = (uint8_t*)calloc((size_t)n, 1);
        if (high_tier_unconditional) {
            for (int a = 0; a < n; ++a)
                if ((float)c[pool[a]] >= tau_high) kept[a] = 1;
            for (int a = 0; a < n; ++a)
                if (kept[a])
                    for (int e = 0; e < n; ++e)
                        if (!kept[e] && conf_mat[(int64_t)a * n + e]) blocked[e] = 1;
        }
        for (int a = 0; a < n; ++a) {
            if (kept[a] || blocked[a]) continue;
            int ok = 1;
            for (int e = 0; e < n; ++e)
                if (kept[e] && conf_mat[(int64_t)a * n + e]) { ok = 0; break; }
            if (ok) kept[a] = 1;
        }
        int cnt = 0;
        for (int a = 0; a < n; ++a)
            if (kept[a]) { sel[pool[a]] = 1; ++cnt; }
        n_selected[b] = cnt;
        free(kept);
        free(blocked);
        free(conf_mat);
        free(pool);
    }
    return clipped_any;
}

/* ------------------------------------------------------------------------
 * DAPD step (DAPD, 整体框架 and 关键设计 1-3).
 *   V_t = masked positions of the block, r = |V_t| / blk.
 *   r < bulk_frac (fp32 test)  -> late phase: commit every masked position
 *       with c_i > bulk_conf; if none, the top-confidence one (a fallback
 *       borrowed from the Fast-dLLM and DepCap rules so progress is kept).
 *   otherwise:
 *       a_ij = mean over the given layers and heads of A[l][h][i][j]
 *       s_ij = (a_ij + a_ji) / 2,  edge (i,j) <=> s_ij > tau   (i != j)
 *       d~_i = sum over j in V_t, j != i of s_ij
 *       key_i = d~_i * c_i   (order_mode 1: key_i = d~_i)
 *       scan V_t by key descending (ties to the lower position) and keep a
 *       node iff none of its neighbours is already kept (Welsh-Powell greedy
 *       maximal independent set).
 * The attention element (b,l,h,row,col) is attn[b*sb + l*sl + h*sh +
 * row*sr + col]; the block occupies rows and columns
 * [block_start, block_start+blk).  Outputs s (NaN off V_t), d~, the edge
 * degree, and the path taken (0 graph, 1 late phase).
 * preunmask_certain (DAPD, 关键设计 3, appendix remark: a position whose
 * confidence is exactly 1.0 can be unmasked at any time): read as adding
 * every masked position with conf == 1.0 (fp32) to the selection of either
 * path; the graph itself is unchanged.
 * ------------------------------------------------------------------------ */
void oracle_dapd(const void* attn, int dtype, int batch, int n_layers, int n_heads,
                 int64_t sb, int64_t sl, int64_t sh, int64_t sr, int block_start, int blk,
                 const uint8_t* masked, const double* conf, float tau_edge, float bulk_conf,
                 float bulk_frac, int order_mode, int preunmask_certain, uint8_t* selected,
                 int32_t* n_selected, double* s_out, double* dtilde_out, int32_t* deg_out,
                 int32_t* path_out) {
    int b;
#pragma omp parallel for schedule(dynamic, 1)
    for (b = 0; b < batch; ++b) {
        int64_t base = (int64_t)b * blk;
        const uint8_t* mk = masked + base;
        const double* c = conf + base;
        uint8_t* sel = selected + base;
        int M = 0;
        for (int i = 0; i < blk; ++i) M += mk[i] ? 1 : 0;
        for (int i = 0; i < blk; ++i) sel[i] = 0;
        if (s_out)
            for (int64_t e = 0; e < (int64_t)blk * blk; ++e) s_out[(int64_t)b * blk * blk + e] = NAN;
        if (dtilde_out)
            for (int i = 0; i < blk; ++i) dtilde_out[base + i] = NAN;
        if (deg_out)
            for (int i = 0; i < blk; ++i) deg_out[base + i] = -1;

        if ((float)M < bulk_frac * (float)blk) {
            if (path_out) path_out[b] = 1;
            int n = 0;
            for (int i = 0; i < blk; ++i) {
                sel[i] = (uint8_t)(mk[i] && (float)c[i] > bulk_conf);
                n += sel[i];
            }
            if (n == 0) {
                int t = top_conf(c, mk, blk);
                if (t >= 0) { sel[t] = 1; n = 1; }
            }
            if (preunmask_certain)
                for (int i = 0; i < blk; ++i)
                    if (mk[i] && !sel[i] && (float)c[i] == 1.0f) { sel[i] = 1; ++n; }
            n_selected[b] = n;
            continue;
        }
        if (path_out) path_out[b] = 0;

        int* node = (int*)malloc(sizeof(int) * (size_t)M);
        int k = 0;
        for (int i = 0; i < blk; ++i)
            if (mk[i]) node[k++] = i;
        double* a = (double*)malloc(sizeof(double) * (size_t)M * M);
        double LH = (double)n_layers * (double)n_heads;
        for (int x = 0; x < M; ++x)
            for (int y = 0; y < M; ++y) {
                int64_t row = block_start + node[x], col = block_start + node[y];
                double acc = 0.0;
                for (int l = 0; l < n_layers; ++l)
                    for (int h = 0; h < n_heads; ++h)
                        acc += load_elem(attn, dtype, b * sb + l * sl + h * sh + row * sr + col);
                a[(int64_t)x * M + y] = acc / LH;
            }
        uint8_t* adj = (uint8_t*)calloc((size_t)M * M, 1);
        double* key = (double*)malloc(sizeof(double) * (size_t)M);
        for (int x = 0; x < M; ++x) {
            double dt = 0.0;
            int deg = 0;
            for (int y = 0; y < M; ++y) {
                double v = 0.5 * (a[(int64_t)x * M + y] + a[(int64_t)y * M + x]);
                if (s_out) s_out[(int64_t)b * blk * blk + (int64_t)node[x] * blk + node[y]] = v;
                if (y == x) continue;
                dt += v;
                if (v > (double)tau_edge) { adj[(int64_t)x * M + y] = 1; ++deg; }
            }
            if (dtilde_out) dtilde_out[base + node[x]] = dt;
            if (deg_out) deg_out[base + node[x]] = deg;
            key[x] = order_mode == 1 ? dt : dt * c[node[x]];
        }
        /* order: key descending, ties to the lower position */
        int* ord = (int*)malloc(sizeof(int) * (size_t)M);
        for (int x = 0; x < M; ++x) ord[x] = x;
        for (int p = 1; p < M; ++p) {
            int x = ord[p], q = p - 1;
            while (q >= 0 && (key[x] > key[ord[q]] || (key[x] == key[ord[q]] && x < ord[q]))) {
                ord[q + 1] = ord[q];
                --q;
            }
            ord[q + 1] = x;
        }
        uint8_t* kept = (uint8_t*)calloc((size_t)M, 1);
        int cnt = 0;
        for (int p = 0; p < M; ++p) {
            int x = ord[p];
            int ok = 1;
            for (int y = 0; y < M; ++y)
                if (kept[y] && adj[(int64_t)x * M + y]) { ok = 0; break; }
            if (ok) { kept[x] = 1; sel[node[x]] = 1; ++cnt; }
        }
        if (preunmask_certain)
            for (int i = 0; i < blk; ++i)
                if (mk[i] && !sel[i] && (float)c[i] == 1.0f) { sel[i] = 1; ++cnt; }
        n_selected[b] = cnt;
        free(kept);
        free(ord);
        free(key);
        free(adj);
        free(a);
        free(node);
    }
}

/* ------------------------------------------------------------------------
 * Downstream influence for the revocable rule's seed score (COVER page,
 * "Method": a seed's score combines its uncertainty, its downstream
 * influence and its cache drift; the page does not define influence).
 * Reading: the influence of block position i is the attention it receives
 * from the positions still to be decoded -- the masked queries q of the
 * block -- averaged over the given layers and heads:
 *   infl_i = (1 / (L H)) sum_{q masked} sum_{l, h} A[l][h][q][i]
 * for every position i of the block (masked or not).  Element (b,l,h,row,col)
 * of attn at b*sb + l*sl + h*sh + row*sr + col; the block is rows and
 * columns [block_start, block_start + blk).
 * ------------------------------------------------------------------------ */
void oracle_attention_influence(const void* attn, int dtype, int batch, int n_layers, int n_heads, int64_t sb,
                                int64_t sl, int64_t sh, int64_t sr, int block_start, int blk,
                                const uint8_t* masked, double* infl) {
    int b;
#pragma omp parallel for schedule(dynamic, 1)
    for (b = 0; b < batch; ++b) {
        const uint8_t* mk = masked + (int64_t)b * blk;
        double LH = (double)n_layers * (double)n_heads;
        for (int i = 0; i < blk; ++i) {
            double acc = 0.0;
            for (int q = 0; q < blk; ++q) {
                if (!mk[q]) continue;
                for (int l = 0; l < n_layers; ++l)
                    for (int h = 0; h < n_heads; ++h)
                        acc += load_elem(attn, dtype, b * sb + l * sl + h * sh + (int64_t)(block_start + q) * sr +
                                                          block_start + i);
            }
            infl[(int64_t)b * blk + i] = acc / LH;
        }
    }
}

/* Greedy maximal independent set over an explicit order (used by the tests
 * to evaluate alternative orders of near-tied keys): adj is n x n bytes,
 * order lists node ids; kept[x] = 1 for the nodes taken. */
void oracle_greedy_mis(int n, const uint8_t* adj, const int32_t* order, uint8_t* kept) {
    for (int x = 0; x < n; ++x) kept[x] = 0;
    for (int p = 0; p < n; ++p) {
        int x = order[p];
        int ok = 1;
        for (int y = 0; y < n; ++y)
            if (kept[y] && adj[(int64_t)x * n + y]) { ok = 0; break; }
        if (ok) kept[x] = 1;
    }
}

/* ------------------------------------------------------------------------
 * Confidence order of the masked positions of one block: (conf desc,
 * position asc), compared in fp32.  Returns the count m; order[0..m).
 * ------------------------------------------------------------------------ */
static int masked_by_conf(const double* c, const uint8_t* mk, int blk, int* order) {
    int m = 0;
    for (int i = 0; i < blk; ++i)
        if (mk[i]) order[m++] = i;
    for (int a = 1; a < m; ++a) {
        int x = order[a], k = a - 1;
        while (k >= 0 && conf_before(c, x, order[k])) { order[k + 1] = order[k]; --k; }
        order[k + 1] = x;
    }
    return m;
}

/* Fixed top-K per step (Fast-dLLM review, Prior limitations: LLaDA's default
 * commits K tokens per step whatever their confidence): the min(K, masked)
 * masked positions of highest confidence, ties to the lower position. */
void oracle_select_topk(const double* conf, const uint8_t* masked, int batch, int blk, int k,
                        uint8_t* selected, int32_t* n_selected) {
    int* order = (int*)malloc(sizeof(int) * (size_t)(blk > 0 ? blk : 1));
    for (int b = 0; b < batch; ++b) {
        const double* c = conf + (int64_t)b * blk;
        uint8_t* sel = selected + (int64_t)b * blk;
        int m = masked_by_conf(c, masked + (int64_t)b * blk, blk, order);
        int n = k < m ? k : m;
        for (int i = 0; i < blk; ++i) sel[i] = 0;
        for (int r = 0; r < n; ++r) sel[order[r]] = 1;
        n_selected[b] = n;
    }
    free(order);
}

/* Factor decoding (Fast-dLLM review, Method, appendix variant): with
 * c^(1) >= c^(2) >= ... the masked confidences in decreasing order, commit
 * the top n* positions, n* = the largest n with (n + 1)(1 - c^(n)) < f,
 * evaluated in fp32.  The left side grows with n, so the qualifying n form a
 * prefix.  If no n qualifies, the top position alone is committed (the
 * threshold rule's progress guarantee). */
void oracle_select_factor(const double* conf, const uint8_t* masked, int batch, int blk, float f,
                          uint8_t* selected, int32_t* n_selected) {
    int* order = (int*)malloc(sizeof(int) * (size_t)(blk > 0 ? blk : 1));
    for (int b = 0; b < batch; ++b) {
        const double* c = conf + (int64_t)b * blk;
        uint8_t* sel = selected + (int64_t)b * blk;
        int m = masked_by_conf(c, masked + (int64_t)b * blk, blk, order);
        int n = 0;
        for (int r = 0; r < m; ++r) {
            float cn = (float)c[order[r]];
            float lhs = (float)(r + 2) * (1.0f - cn);
            if (lhs < f) n = r + 1;
        }
        if (n == 0 && m > 0) n = 1;
        for (int i = 0; i < blk; ++i) sel[i] = 0;
        for (int r = 0; r < n; ++r) sel[order[r]] = 1;
        n_selected[b] = n;
    }
    free(order);
}

/* Theorem-1 certificate (Fast-dLLM review, Key idea): committing the n
 * selected positions in parallel gives the same tokens as committing them one
 * by one greedily when every one of them has confidence above 1 - 1/(n+1).
 * Tested in fp32; an empty selection is certified. */
void oracle_parallel_certificate(const double* conf, const uint8_t* selected, int batch, int blk,
                                 uint8_t* certified) {
    for (int b = 0; b < batch; ++b) {
        const double* c = conf + (int64_t)b * blk;
        const uint8_t* sel = selected + (int64_t)b * blk;
        int n = 0;
        for (int i = 0; i < blk; ++i) n += sel[i] ? 1 : 0;
        float bound = 1.0f - 1.0f / (float)(n + 1);
        int ok = 1;
        for (int i = 0; i < blk; ++i)
            if (sel[i] && !((float)c[i] > bound)) ok = 0;
        certified[b] = (uint8_t)ok;
    }
}

/* ------------------------------------------------------------------------
 * Revocable parallel decoding, one state update (COVER page: "Revocable
 * Parallel Diffusion Decoding" -- draft masked positions, verify the seeds,
 * remask some, net growth = drafted - revoked, stop when nothing is masked;
 * "Method" -- KEEP / REPLACE / REMASK, stability-aware seed selection from
 * uncertainty, downstream influence and cache drift, |S_t| = ceil(sqrt(n_t)
 * pi_t), recently selected positions and those at their remask budget
 * excluded).
 * Readings: KEEP iff the re-prediction equals the token; REPLACE iff it
 * differs and its confidence reaches tau_replace; REMASK otherwise.  Drafting
 * is the confidence threshold (strict) with the top-1 fallback, at most
 * draft_budget (<= 0: no cap).  score = w_unc (1 - c) + w_infl infl - w_drift
 * drift; pi_t = pi; n_t = number of eligible positions.  Every decision is
 * taken in fp32 (the score rounded after each operation).
 * ------------------------------------------------------------------------ */
static void sort_desc_f32(int* idx, const float* key, int n) {
    /* insertion sort: larger key first, ties to the lower index */
    for (int a = 1; a < n; ++a) {
        int v = idx[a];
        int p = a - 1;
        while (p >= 0 && (key[idx[p]] < key[v] || (key[idx[p]] == key[v] && idx[p] > v))) {
            idx[p + 1] = idx[p];
            --p;
        }
        idx[p + 1] = v;
    }
}

void oracle_revocable_step(const int32_t* argmax, const double* conf, const double* influence,
                           const double* drift, int batch, int blk, int step, float tau_replace,
                           float tau_draft, int draft_budget, float w_unc, float w_infl, float w_drift,
                           float pi, int cooldown, int remask_budget, int32_t* tok, uint8_t* masked,
                           uint8_t* seed, int32_t* last_seed, int32_t* remasks, int32_t* last_tok,
                           uint8_t* outcome, int32_t* n_drafted, int32_t* n_revoked, int32_t* flipflops) {
    int* idx = (int*)malloc(sizeof(int) * (size_t)blk);
    float* key = (float*)malloc(sizeof(float) * (size_t)blk);
    uint8_t* was_masked = (uint8_t*)malloc((size_t)blk);
    for (int b = 0; b < batch; ++b) {
        const int64_t o = (int64_t)b * blk;
        int m0 = 0;
        for (int i = 0; i < blk; ++i) {
            was_masked[i] = masked[o + i] ? 1 : 0;
            m0 += was_masked[i];
            outcome[o + i] = 0;
        }
        n_drafted[b] = 0;
        n_revoked[b] = 0;
        if (m0 == 0) continue; /* finished: nothing changes */

        /* 1. verification of the seeds */
        for (int i = 0; i < blk; ++i) {
            if (!seed[o + i] || was_masked[i]) continue;
            if (argmax[o + i] == tok[o + i]) {
                outcome[o + i] = 2;
            } else if ((float)conf[o + i] >= tau_replace) {
                outcome[o + i] = 3;
                tok[o + i] = argmax[o + i];
            } else {
                outcome[o + i] = 4;
                last_tok[o + i] = tok[o + i];
                tok[o + i] = -1;
                masked[o + i] = 1;
                remasks[o + i] += 1;
                n_revoked[b] += 1;
            }
        }

        /* 2. drafting over the positions masked at the start */
        int n = 0;
        for (int i = 0; i < blk; ++i) {
            key[i] = (float)conf[o + i];
            if (was_masked[i] && key[i] > tau_draft) idx[n++] = i;
        }
        if (n == 0) {
            for (int i = 0; i < blk; ++i)
                if (was_masked[i]) idx[n++] = i;
            sort_desc_f32(idx, key, n);
            n = 1;
        } else {
            sort_desc_f32(idx, key, n);
            if (draft_budget > 0 && n > draft_budget) n = draft_budget;
        }
        for (int r = 0; r < n; ++r) {
            int i = idx[r];
            outcome[o + i] = 1;
            tok[o + i] = argmax[o + i];
            masked[o + i] = 0;
            if (last_tok[o + i] == argmax[o + i] && flipflops) flipflops[b] += 1;
        }
        n_drafted[b] = n;

        /* 3. the next step's seeds */
        int ne = 0;
        for (int i = 0; i < blk; ++i) {
            seed[o + i] = 0;
            int eligible = !masked[o + i] && (step - last_seed[o + i] > cooldown) &&
                           remasks[o + i] < remask_budget;
            if (!eligible) continue;
            float unc = 1.0f - (float)conf[o + i];
            float a = w_unc * unc;
            float c = w_infl * (influence ? (float)influence[o + i] : 0.0f);
            float d = w_drift * (drift ? (float)drift[o + i] : 0.0f);
            float s = a + c;
            key[i] = s - d;
            idx[ne++] = i;
        }
        float kf = ceilf(sqrtf((float)ne) * pi);
        int k = kf < (float)ne ? (int)kf : ne;
        sort_desc_f32(idx, key, ne);
        for (int r = 0; r < k; ++r) {
            seed[o + idx[r]] = 1;
            last_seed[o + idx[r]] = step;
        }
    }
    free(idx);
    free(key);
    free(was_masked);
}
