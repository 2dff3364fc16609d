// cap.cu -- DepCap CAP-Decoding: confidence pool, pairwise conflict score,
// greedy conflict-free selection (DepCap, "Methodology"; defaults in
// "Experiments").
//
// Pools of up to 64 candidates: one fused launch (cap_fused_kernel below).
// Larger pools: three launches on the caller's stream:
//   cap_pool     one CTA per sequence: candidates (masked, conf >= tau_low)
//                ranked by (conf desc, position asc) with an all-pairs rank
//                count, clipped to p_max;
//   cap_conflict one warp per pool row: D_ij = log p_i(yhat_j) + log p_j(yhat_i)
//                from two scattered logit reads per pair, conflict bits packed
//                with a warp ballot (one 32-bit word per 32 partners);
//   cap_greedy   one CTA per sequence: the greedy scan over the pool order on
//                the shared-memory bitmask, or the top-confidence fallback.
// The pool order and the two bitmask passes live in the caller's workspace.
#include "common.cuh"
#include "launch.h"

namespace dlm {

namespace {

constexpr int kThreads = 256;
constexpr int kConflictWarps = 8;
constexpr int kMaxPoolWords = DLM_MAX_BLK / 32;  // p_max <= 256

__device__ __forceinline__ float load_logit(const void* base, int dtype, int64_t i) {
    if (dtype == DLM_BF16) return __uint_as_float((uint32_t) static_cast<const uint16_t*>(base)[i] << 16);
    if (dtype == DLM_F16) return __half2float(static_cast<const __half*>(base)[i]);
    return static_cast<const float*>(base)[i];
}

// log p_i(token): the logit of `token` in row `row` minus the row's LSE.  A
// token outside the vocabulary (an argmax of a row that held only NaN) is
// not read: the value is NaN (never a conflict) and the status word says so.
__device__ __forceinline__ float logp_at(const CapArgs& a, int64_t row, int token, float lse) {
    if ((unsigned)token >= (unsigned long long)a.vocab) {
        raise_status(a.dev_status, DLM_DEV_NONFINITE);
        return __int_as_float(0x7fc00000);
    }
    return load_logit(a.logits, a.dtype, row * a.row_stride + token) - lse;
}

__device__ __forceinline__ int scope_of(const CapArgs& a, int b) {
    int sc = a.blk;
    if (a.scope_len) sc = min(sc, max(0, a.scope_len[b]));
    return sc;
}

__global__ void __launch_bounds__(kThreads) cap_pool_kernel(CapArgs a) {
    __shared__ float s_c[kThreads];
    __shared__ int s_cand[kThreads];
    const int b = blockIdx.x, i = threadIdx.x;
    const int scope = scope_of(a, b);
    const int64_t o = (int64_t)b * a.blk + i;
    const bool cand = i < scope && a.masked[o] != 0 && a.conf[o] >= a.tau_low;
    s_c[i] = cand ? a.conf[o] : 0.f;
    s_cand[i] = cand;
    const int n = __syncthreads_count(cand);
    if (cand) {
        const float c = s_c[i];
        int rank = 0;
        for (int j = 0; j < scope; ++j) {
            if (!s_cand[j]) continue;
            const float cj = s_c[j];
            rank += (cj > c) || (cj == c && j < i);
        }
        if (rank < a.p_max) a.pool[(int64_t)b * a.p_max + rank] = i;
    }
    if (i == 0) {
        a.pool_n[b] = min(n, a.p_max);
        if (n > a.p_max) raise_status(a.dev_status, DLM_DEV_POOL_CLIPPED);
    }
}

__global__ void __launch_bounds__(kConflictWarps * 32) cap_conflict_kernel(CapArgs a) {
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = blockIdx.x * kConflictWarps + warp;
    const int n = a.pool_n[b];
    if (slot >= n) return;
    const int32_t* pool = a.pool + (int64_t)b * a.p_max;
    const int pi = pool[slot];
    const int64_t ri = (int64_t)b * a.blk + pi;
    const int yi = a.argmax[ri];
    const float li = a.lse[ri];
    uint32_t* adj = a.adj + ((int64_t)b * a.p_max + slot) * a.words;
    const int nw = (n + 31) >> 5;
    // every partner's scattered loads are issued before any is used (one
    // round trip for the row instead of one per 32 partners)
    float g[kMaxPoolWords];
#pragma unroll
    for (int c = 0; c < kMaxPoolWords; ++c) {
        const int e = c * 32 + lane;
        g[c] = __int_as_float(0x7fc00000);
        if (c < nw && e < n && e != slot) {
            const int pj = pool[e];
            const int64_t rj = (int64_t)b * a.blk + pj;
            g[c] = logp_at(a, ri, a.argmax[rj], li) + logp_at(a, rj, yi, a.lse[rj]);
        }
    }
#pragma unroll
    for (int c = 0; c < kMaxPoolWords; ++c) {
        if (c >= nw) break;
        const int e = c * 32 + lane;
        const bool conflict = g[c] > a.gamma;  // NaN (no partner) is never a conflict
        if (a.D_out && e < n && e != slot) a.D_out[((int64_t)b * a.blk + pi) * a.blk + pool[e]] = g[c];
        const uint32_t word = __ballot_sync(DLM_FULL_MASK, conflict);
        if (lane == 0) adj[c] = word;
    }
}

__global__ void __launch_bounds__(kThreads) cap_greedy_kernel(CapArgs a) {
    __shared__ uint32_t s_adj[DLM_MAX_BLK * (DLM_MAX_BLK / 32)];
    __shared__ uint32_t s_kept[DLM_MAX_BLK / 32];
    __shared__ unsigned char s_tier[DLM_MAX_BLK];
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    const int b = blockIdx.x, t = threadIdx.x;
    const int n = a.pool_n[b];
    const int scope = scope_of(a, b);
    uint8_t* sel = a.selected + (int64_t)b * a.blk;
    const int32_t* pool = a.pool + (int64_t)b * a.p_max;
    if (t < a.blk) sel[t] = 0;
    if (n == 0) {
        // no candidate: the highest-confidence masked position of the scope
        const int64_t o = (int64_t)b * a.blk + t;
        const bool m = t < scope && a.masked[o] != 0;
        float v = m ? a.conf[o] : -INFINITY;
        int idx = m ? t : 0x7fffffff;
        const int any_m = __syncthreads_or(m);
        warp_argmax(v, idx);
        if ((t & 31) == 0) {
            s_v[t >> 5] = v;
            s_i[t >> 5] = idx;
        }
        __syncthreads();
        if (t < 32) {
            v = t < kThreads / 32 ? s_v[t] : -INFINITY;
            idx = t < kThreads / 32 ? s_i[t] : 0x7fffffff;
            warp_argmax(v, idx);
            if (t == 0) {
                if (any_m) sel[idx] = 1;
                a.n_selected[b] = any_m ? 1 : 0;
            }
        }
        return;
    }
    const int W = (n + 31) >> 5;
    for (int k = t; k < n * W; k += blockDim.x) {
        const int s = k / W, w = k - s * W;
        s_adj[s * W + w] = a.adj[((int64_t)b * a.p_max + s) * a.words + w];
    }
    if (t < n) s_tier[t] = a.high_tier_unconditional && a.conf[(int64_t)b * a.blk + pool[t]] >= a.tau_high;
    __syncthreads();
    if (t < 32) {
        // lane w holds word w of the kept set; tier members are forced in when
        // the tier is unconditional (s_tier is all zero otherwise)
        const uint32_t kept = greedy_scan(s_adj, W, nullptr, s_tier, n, W);
        if (t < W) s_kept[t] = kept;
    }
    __syncthreads();
    int mine = 0;
    if (t < n && ((s_kept[t >> 5] >> (t & 31)) & 1u)) {
        sel[pool[t]] = 1;
        mine = 1;
    }
    const int total = __syncthreads_count(mine);
    if (t == 0) a.n_selected[b] = total;
}

// Small pools (p_max <= kFusedMaxPool): the three phases in one CTA per
// sequence, the pool, its tokens / LSEs and the conflict bitmask in shared
// memory.  D is symmetric (the two log-probabilities are added in either
// order, and fp32 addition commutes), so each unordered pair is scored once
// and both bits are set.
constexpr int kFusedMaxPool = 64;
constexpr int kFusedWords = kFusedMaxPool / 32;
constexpr int kPairUnroll = 4;  // 64 * 63 / 2 pairs = 8 per thread at most

__global__ void __launch_bounds__(kThreads) cap_fused_kernel(CapArgs a) {
    __shared__ float s_c[kThreads];
    __shared__ int s_cand[kThreads];
    __shared__ int s_pool[kFusedMaxPool];
    __shared__ int s_y[kFusedMaxPool];
    __shared__ float s_lse[kFusedMaxPool];
    __shared__ uint32_t s_adj[kFusedMaxPool * kFusedWords];
    __shared__ uint32_t s_kept[kFusedWords];
    __shared__ unsigned char s_tier[kFusedMaxPool];
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    const int b = blockIdx.x, t = threadIdx.x;
    const int scope = scope_of(a, b);
    const int64_t o = (int64_t)b * a.blk + t;
    uint8_t* sel = a.selected + (int64_t)b * a.blk;

    // 1. pool: masked in scope with conf >= tau_low, by (conf desc, position asc);
    // the token and LSE are loaded with the confidence (one round trip)
    const bool in = t < a.blk;
    const bool m = t < scope && a.masked[o] != 0;
    const float c = in ? a.conf[o] : 0.f;
    const int y = in ? a.argmax[o] : 0;
    const float l = in ? a.lse[o] : 0.f;
    const bool cand = m && c >= a.tau_low;
    s_c[t] = cand ? c : 0.f;
    s_cand[t] = cand;
    if (t < kFusedMaxPool * kFusedWords) s_adj[t] = 0u;
    const int n_cand = __syncthreads_count(cand);
    const int n = min(n_cand, a.p_max);
    if (cand) {
        int rank = 0;
        for (int j = 0; j < scope; ++j) {
            if (!s_cand[j]) continue;
            const float cj = s_c[j];
            rank += (cj > c) || (cj == c && j < t);
        }
        if (rank < a.p_max) {
            s_pool[rank] = t;
            s_y[rank] = y;
            s_lse[rank] = l;
            s_tier[rank] = a.high_tier_unconditional && c >= a.tau_high;
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
            s_v[t >> 5] = v;
            s_i[t >> 5] = idx;
        }
        __syncthreads();
        if (t < 32) {
            v = t < kThreads / 32 ? s_v[t] : -INFINITY;
            idx = t < kThreads / 32 ? s_i[t] : 0x7fffffff;
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
    for (int q0 = t; q0 < pairs; q0 += kThreads * kPairUnroll) {
        // an index past the last pair maps to the pair (0, 1), which exists
        // (pairs >= 1), and its result is dropped
        int pi[kPairUnroll], pj[kPairUnroll];
        float z1[kPairUnroll], z2[kPairUnroll];
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            const int q = min(q0 + u * kThreads, pairs - 1);
            // row i holds the pairs (i, i+1 .. n-1); find i with start(i) <= q
            int i = 0, start = 0;
            while (start + (n - 1 - i) <= q) {
                start += n - 1 - i;
                ++i;
            }
            pi[u] = i;
            pj[u] = i + 1 + (q - start);
        }
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            const int64_t ri = (int64_t)b * a.blk + s_pool[pi[u]];
            const int64_t rj = (int64_t)b * a.blk + s_pool[pj[u]];
            z1[u] = logp_at(a, ri, s_y[pj[u]], s_lse[pi[u]]);
            z2[u] = logp_at(a, rj, s_y[pi[u]], s_lse[pj[u]]);
        }
#pragma unroll
        for (int u = 0; u < kPairUnroll; ++u) {
            if (q0 + u * kThreads >= pairs) break;
            const int i = pi[u], j = pj[u];
            const float d = z1[u] + z2[u];
            if (d > a.gamma) {
                atomicOr(&s_adj[i * kFusedWords + (j >> 5)], 1u << (j & 31));
                atomicOr(&s_adj[j * kFusedWords + (i >> 5)], 1u << (i & 31));
            }
            if (a.D_out) {
                a.D_out[((int64_t)b * a.blk + s_pool[i]) * a.blk + s_pool[j]] = d;
                a.D_out[((int64_t)b * a.blk + s_pool[j]) * a.blk + s_pool[i]] = d;
            }
        }
    }
    __syncthreads();

    // 3. greedy over the pool order
    const int W = (n + 31) >> 5;
    if (t < 32) {
        const uint32_t kept = greedy_scan(s_adj, kFusedWords, nullptr, s_tier, n, W);
        if (t < W) s_kept[t] = kept;
    }
    __syncthreads();
    int mine = 0;
    if (t < n && ((s_kept[t >> 5] >> (t & 31)) & 1u)) {
        sel[s_pool[t]] = 1;
        mine = 1;
    }
    const int total = __syncthreads_count(mine);
    if (t == 0) a.n_selected[b] = total;
}

}  // namespace

size_t cap_workspace_bytes(int batch, int p_max) {
    const size_t words = (size_t)((p_max + 31) / 32);
    size_t pool = ((size_t)batch * p_max * 4 + 255) & ~(size_t)255;
    size_t pn = ((size_t)batch * 4 + 255) & ~(size_t)255;
    size_t adj = (size_t)batch * p_max * words * 4;
    return pool + pn + adj;
}

void cap_carve(CapArgs& a, void* ws) {
    char* p = static_cast<char*>(ws);
    a.words = (a.p_max + 31) / 32;
    a.pool = reinterpret_cast<int32_t*>(p);
    p += ((size_t)a.batch * a.p_max * 4 + 255) & ~(size_t)255;
    a.pool_n = reinterpret_cast<int32_t*>(p);
    p += ((size_t)a.batch * 4 + 255) & ~(size_t)255;
    a.adj = reinterpret_cast<uint32_t*>(p);
}

cudaError_t launch_cap(const CapArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kThreads);
    if (a.p_max <= kFusedMaxPool) return cudaLaunchKernelEx(&cfg, cap_fused_kernel, a);
    cudaError_t e = cudaLaunchKernelEx(&cfg, cap_pool_kernel, a);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)((a.p_max + kConflictWarps - 1) / kConflictWarps), (unsigned)a.batch);
    cfg.blockDim = dim3(kConflictWarps * 32);
    e = cudaLaunchKernelEx(&cfg, cap_conflict_kernel, a);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kThreads);
    return cudaLaunchKernelEx(&cfg, cap_greedy_kernel, a);
}

}  // namespace dlm
