// rules.cuh -- the per-sequence selection rules as block-level device
// functions: one CTA of kRuleThreads threads decides one sequence.  The rule
// kernels (select.cu, cap.cu) run one sequence per CTA; the fused row pass
// (row_stats.cu) runs them in the CTA that finishes a sequence's last row.
//
// Statistics a rule reads (conf, argmax, LSE, KL, entropy, a scope length)
// may have been written by other CTAs of the same launch, so they are loaded
// at L2 (ld.global.cg), never from a possibly stale L1 line.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace dlm {

constexpr int kRuleThreads = 256;  // >= DLM_MAX_BLK: one position per thread

template <typename T>
__device__ __forceinline__ T ld_l2(const T* p) {
    return __ldcg(p);
}

// ---- Fast-dLLM threshold --------------------------------------------------
// Fast-dLLM review, "Method"; Fast-dLLM notes, "Key ideas" (safety valve):
// keep masked positions with conf > tau, else the top-confidence masked one.
struct ThresholdSmem {
    float v[kRuleThreads / 32];
    int i[kRuleThreads / 32];
};

__device__ __forceinline__ void threshold_block(const ThresholdArgs& a, int b, ThresholdSmem& sm) {
    const int i = threadIdx.x;
    const bool valid = i < a.blk;
    const int64_t o = (int64_t)b * a.blk + i;
    const bool m = valid && a.masked[o] != 0;
    const float c = m ? ld_l2(a.conf + o) : 0.f;
    bool s = m && c > a.tau;
    int n = __syncthreads_count(s);
    const int any_m = __syncthreads_or(m);
    if (n == 0 && any_m) {
        float v = m ? c : -INFINITY;
        int idx = m ? i : 0x7fffffff;
        warp_argmax(v, idx);
        if ((i & 31) == 0) {
            sm.v[i >> 5] = v;
            sm.i[i >> 5] = idx;
        }
        __syncthreads();
        if (i < 32) {
            v = i < kRuleThreads / 32 ? sm.v[i] : -INFINITY;
            idx = i < kRuleThreads / 32 ? sm.i[i] : 0x7fffffff;
            warp_argmax(v, idx);
            if (i == 0) sm.i[0] = idx;
        }
        __syncthreads();
        s = (i == sm.i[0]);
        n = 1;
    }
    if (valid) a.selected[o] = s ? 1 : 0;
    if (i == 0) a.n_selected[b] = n;
}

// ---- DepGA-Block boundary -------------------------------------------------
// Block-wide sum and minimum in a fixed order (warp trees, then the warps in
// order), so results do not depend on timing.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(DLM_FULL_MASK, v, o);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) t += red[k];
    return t;
}

__device__ __forceinline__ float block_min(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(DLM_FULL_MASK, v, o));
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = red[0];
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) t = fminf(t, red[k]);
    return t;
}

template <int W>
struct BoundarySmem {
    float sI[W], sH[W], tI[W], tH[W];
    float red[kRuleThreads / 32];
};

// DepCap, "Methodology": S_k = I~_k - lambda H~_k over the window, stop before
// the first negative, clip to [L_min, L_window], cold start -> L_min.
// Smoothing: centred moving average of odd width, edge-truncated.
// Normalisation: 0 window mean, 1 min-max, 2 none.
// Ragged windows: with window_len, sequence b uses the first window_len[b]
// entries of its row (row stride L_window); an empty window gives length 0.
// W bounds the window (L_window <= W).
template <int W>
__device__ __forceinline__ void boundary_block(const BoundaryArgs& a, int b, BoundarySmem<W>& sm) {
    const int L = a.window_len ? min(max(a.window_len[b], 0), a.L_window) : a.L_window;
    const int64_t row = (int64_t)b * a.L_window;
    if (L == 0) {  // uniform over the CTA
        if (threadIdx.x == 0) a.block_len[b] = 0;
        return;
    }
    const float* I = a.kl + row;
    const float* H = a.entropy + row;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        sm.sI[k] = ld_l2(I + k);
        sm.sH[k] = ld_l2(H + k);
    }
    __syncthreads();
    const int h = a.smooth_w / 2;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        const int lo = max(0, k - h), hi = min(L - 1, k + h);
        float ai = 0.f, ah = 0.f;
        for (int j = lo; j <= hi; ++j) {
            ai += sm.sI[j];
            ah += sm.sH[j];
        }
        const float cnt = (float)(hi - lo + 1);
        sm.tI[k] = ai / cnt;
        sm.tH[k] = ah / cnt;
    }
    __syncthreads();
    float mulI = 1.f, addI = 0.f, mulH = 1.f, addH = 0.f;
    if (a.norm_mode == 0) {
        float pi = 0.f, ph = 0.f;
        for (int k = threadIdx.x; k < L; k += blockDim.x) {
            pi += sm.tI[k];
            ph += sm.tH[k];
        }
        const float mi = fmaxf(block_sum(pi, sm.red) / (float)L, 1e-12f);
        const float mh = fmaxf(block_sum(ph, sm.red) / (float)L, 1e-12f);
        mulI = 1.f / mi;
        mulH = 1.f / mh;
    } else if (a.norm_mode == 1) {
        float mni = INFINITY, mnh = INFINITY, mxi = -INFINITY, mxh = -INFINITY;
        for (int k = threadIdx.x; k < L; k += blockDim.x) {
            mni = fminf(mni, sm.tI[k]);
            mxi = fmaxf(mxi, sm.tI[k]);
            mnh = fminf(mnh, sm.tH[k]);
            mxh = fmaxf(mxh, sm.tH[k]);
        }
        mni = block_min(mni, sm.red);
        mnh = block_min(mnh, sm.red);
        mxi = -block_min(-mxi, sm.red);
        mxh = -block_min(-mxh, sm.red);
        mulI = mxi > mni ? 1.f / (mxi - mni) : 0.f;
        addI = -mni;
        mulH = mxh > mnh ? 1.f / (mxh - mnh) : 0.f;
        addH = -mnh;
    }
    float first = (float)L;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        float ni, nh;
        if (a.norm_mode == 0) {
            ni = sm.tI[k] * mulI;
            nh = sm.tH[k] * mulH;
        } else if (a.norm_mode == 1) {
            ni = (sm.tI[k] + addI) * mulI;
            nh = (sm.tH[k] + addH) * mulH;
        } else {
            ni = sm.tI[k];
            nh = sm.tH[k];
        }
        const float s = ni - a.lambda * nh;
        if (a.score) a.score[row + k] = s;
        if (s < 0.f) first = fminf(first, (float)k);
    }
    const float kstar = block_min(first, sm.red);
    if (threadIdx.x == 0) {
        int len = max((int)kstar, a.L_min);
        len = min(len, L);
        if (a.cold_start && a.cold_start[b]) len = min(a.L_min, L);
        a.block_len[b] = len;
    }
}

// ---- CAP-Decoding ---------------------------------------------------------
__device__ __forceinline__ float load_logit(const void* base, int dtype, int64_t i) {
    if (dtype == DLM_BF16) return __uint_as_float((uint32_t) static_cast<const uint16_t*>(base)[i] << 16);
    if (dtype == DLM_F16) return __half2float(static_cast<const __half*>(base)[i]);
    return static_cast<const float*>(base)[i];
}

// log p_i(token): the logit of `token` in row `row` minus the row's LSE.  A
// token outside the vocabulary (an argmax of a row that held only NaN) or a
// row outside the caller's logits is not read: the value is NaN (never a
// conflict) and the status word says so.
__device__ __forceinline__ float logp_at(const CapArgs& a, int row, int token, float lse) {
    if ((unsigned long long)(int64_t)row >= (unsigned long long)a.n_rows) {
        raise_status(a.dev_status, DLM_DEV_BAD_INDEX);
        return __int_as_float(0x7fc00000);
    }
    if ((unsigned)token >= (unsigned long long)a.vocab) {
        raise_status(a.dev_status, DLM_DEV_NONFINITE);
        return __int_as_float(0x7fc00000);
    }
    return load_logit(a.logits, a.dtype, (int64_t)row * a.row_stride + token) - lse;
}

// Logit row of block position t of sequence b (the caller's row_index, else
// b*blk + t; within int32 because batch*blk < 2^28).
__device__ __forceinline__ int row_of(const CapArgs& a, int b, int t) {
    const int64_t o = (int64_t)b * a.blk + t;
    return a.row_index ? a.row_index[o] : (int)o;
}

// The q-th unordered pair (i < j) of n items in row-major order (row i holds
// (i, i+1) .. (i, n-1)), in closed form: counted from the end, k = T-1-q falls
// in the block of the last r+1 rows with r(r+1)/2 <= k < (r+1)(r+2)/2.
__device__ __forceinline__ void pair_of(int q, int n, int& i, int& j) {
    const int T = n * (n - 1) / 2;
    const int k = T - 1 - q;
    int r = (int)((sqrtf(8.0f * (float)k + 1.0f) - 1.0f) * 0.5f);
    while ((r + 1) * (r + 2) / 2 <= k) ++r;  // correct a rounding of the root
    while (r * (r + 1) / 2 > k) --r;
    i = n - 2 - r;
    j = n - 1 - (k - r * (r + 1) / 2);
}

__device__ __forceinline__ int scope_of(const CapArgs& a, int b) {
    int sc = a.blk;
    if (a.scope_len) sc = min(sc, max(0, ld_l2(a.scope_len + b)));
    return sc;
}

// Pools of up to kCapBlockMaxPool candidates in one CTA: pool, conflict
// scores and greedy, with the pool, its rows / tokens / LSEs and the conflict
// bitmask in shared memory.  D is symmetric (the two log-probabilities are
// added in either order, and fp32 addition commutes), so each unordered pair
// is scored once and both bits are set.
constexpr int kCapBlockMaxPool = 64;
constexpr int kCapBlockWords = kCapBlockMaxPool / 32;
constexpr int kPairUnroll = 4;  // 64 * 63 / 2 pairs = 8 per thread at most

struct CapSmem {
    __align__(16) float c[kRuleThreads];
    __align__(4) unsigned char cand[kRuleThreads];
    int pool[kCapBlockMaxPool];
    int row[kCapBlockMaxPool];
    int y[kCapBlockMaxPool];
    float lse[kCapBlockMaxPool];
    uint32_t adj[kCapBlockMaxPool * kCapBlockWords];
    uint32_t kept[kCapBlockWords];
    unsigned char tier[kCapBlockMaxPool];
    float v[kRuleThreads / 32];
    int i[kRuleThreads / 32];
};

__device__ __forceinline__ void cap_block(const CapArgs& a, int b, CapSmem& sm) {
    const int t = threadIdx.x;
    const int scope = scope_of(a, b);
    const int64_t o = (int64_t)b * a.blk + t;
    uint8_t* sel = a.selected + (int64_t)b * a.blk;

    // 1. pool: masked in scope with conf >= tau_low, by (conf desc, position asc);
    // the token, LSE and logit row are loaded with the confidence (one round trip)
    const bool in = t < a.blk;
    const bool m = t < scope && a.masked[o] != 0;
    const float c = in ? ld_l2(a.conf + o) : 0.f;
    const int y = in ? ld_l2(a.argmax + o) : 0;
    const float l = in ? ld_l2(a.lse + o) : 0.f;
    const bool cand = m && c >= a.tau_low;
    const int row = cand ? row_of(a, b, t) : 0;
    sm.c[t] = c;
    sm.cand[t] = cand;
    if (t < kCapBlockMaxPool * kCapBlockWords) sm.adj[t] = 0u;
    const int n_cand = __syncthreads_count(cand);
    const int n = min(n_cand, a.p_max);
    if (cand) {
        const int rank = rank_desc(sm.c, sm.cand, (scope + 3) & ~3, c, t);
        if (rank < a.p_max) {
            sm.pool[rank] = t;
            sm.row[rank] = row;
            sm.y[rank] = y;
            sm.lse[rank] = l;
            sm.tier[rank] = a.high_tier_unconditional && c >= a.tau_high;
        }
    }
    if (t < a.blk) sel[t] = 0;
    if (t == 0 && n_cand > a.p_max) raise_status(a.dev_status, DLM_DEV_POOL_CLIPPED);
    __syncthreads();

    if (n == 0) {  // no candidate: the highest-confidence masked position of the scope
        float v = m ? c : -INFINITY;
        int idx = m ? t : 0x7fffffff;
        const int any_m = __syncthreads_or(m);
        warp_argmax(v, idx);
        if ((t & 31) == 0) {
            sm.v[t >> 5] = v;
            sm.i[t >> 5] = idx;
        }
        __syncthreads();
        if (t < 32) {
            v = t < kRuleThreads / 32 ? sm.v[t] : -INFINITY;
            idx = t < kRuleThreads / 32 ? sm.i[t] : 0x7fffffff;
            warp_argmax(v, idx);
            if (t == 0) {
                if (any_m) sel[idx] = 1;
                a.n_selected[b] = any_m ? 1 : 0;
            }
        }
        return;
    }

    // 2. conflicts: unordered pairs (i < j) of pool slots, kPairUnroll per
    // thread at a time with all their scattered logit loads issued together
    const int pairs = n * (n - 1) / 2;
    for (int q0 = t; q0 < pairs; q0 += kRuleThreads * kPairUnroll) {
        // an index past the last pair maps to the pair (0, 1), which exists
        // (pairs >= 1), and its result is dropped
        int pi[kPairUnroll], pj[kPairUnroll];
        float z1[kPairUnroll], z2[kPairUnroll];
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            pair_of(min(q0 + u * kRuleThreads, pairs - 1), n, pi[u], pj[u]);
        }
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            z1[u] = logp_at(a, sm.row[pi[u]], sm.y[pj[u]], sm.lse[pi[u]]);
            z2[u] = logp_at(a, sm.row[pj[u]], sm.y[pi[u]], sm.lse[pj[u]]);
        }
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            if (q0 + u * kRuleThreads >= pairs) break;
            const int i = pi[u], j = pj[u];
            const float d = z1[u] + z2[u];
            if (d > a.gamma) {
                atomicOr(&sm.adj[i * kCapBlockWords + (j >> 5)], 1u << (j & 31));
                atomicOr(&sm.adj[j * kCapBlockWords + (i >> 5)], 1u << (i & 31));
            }
            if (a.D_out) {
                a.D_out[((int64_t)b * a.blk + sm.pool[i]) * a.blk + sm.pool[j]] = d;
                a.D_out[((int64_t)b * a.blk + sm.pool[j]) * a.blk + sm.pool[i]] = d;
            }
        }
    }
    __syncthreads();

    // 3. greedy over the pool order
    const int W = (n + 31) >> 5;
    if (t < 32) {
        const uint32_t kept = greedy_scan_chunked(sm.adj, kCapBlockWords, sm.tier, n);  // slots are in pool order
        if (t < W) sm.kept[t] = kept;
    }
    __syncthreads();
    int mine = 0;
    if (t < n && ((sm.kept[t >> 5] >> (t & 31)) & 1u)) {
        sel[sm.pool[t]] = 1;
        mine = 1;
    }
    const int total = __syncthreads_count(mine);
    if (t == 0) a.n_selected[b] = total;
}

}  // namespace dlm
