// cap.cu -- DepCap CAP-Decoding: confidence pool, pairwise conflict score,
// greedy conflict-free selection (DepCap, "Methodology"; defaults in
// "Experiments").
//
// One launch per call:
//   pools of up to 64 candidates: cap_fused_kernel, one CTA per sequence;
//   larger pools: cap_cluster_kernel, a thread-block cluster per sequence.
// Both rank the candidates (masked, conf >= tau_low) by (conf desc, position
// asc) with an all-pairs count, clip to p_max, score every unordered pool
// pair once (D_ij = log p_i(yhat_j) + log p_j(yhat_i), two scattered logit
// reads from the rows the caller's row_index names), keep the conflict bits
// in shared memory and run the greedy scan over the pool order, or the
// top-confidence fallback on an empty pool.  The
// caller's workspace is validated but not used by these kernels (their
// scratch is shared memory); it stays in the interface as the scratch of any
// later variant that needs global memory.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "rules.cuh"

namespace cg = cooperative_groups;

namespace dlm {

namespace {

constexpr int kThreads = kRuleThreads;
constexpr int kMaxPoolWords = DLM_MAX_BLK / 32;  // p_max <= 256
constexpr int kFusedMaxPool = kCapBlockMaxPool;

// Small pools (p_max <= kFusedMaxPool): pool, conflict scores and greedy in
// one CTA per sequence (rules.cuh: cap_block).
__global__ void __launch_bounds__(kThreads) cap_fused_kernel(CapArgs a) {
    __shared__ CapSmem sm;
    cap_block(a, blockIdx.x, sm);
}

// Large pools (p_max > kFusedMaxPool): one thread-block cluster of kCapCluster
// CTAs per sequence.  Every CTA ranks the pool (cheap, redundant), the CTAs
// split the unordered pairs between them and set the conflict bits with
// atomics in the leader CTA's shared bitmask (distributed shared memory), and
// the leader runs the greedy scan: one launch instead of three, and the
// scattered logit loads spread over kCapCluster x 256 threads.
constexpr int kCapCluster = 8;
constexpr int kClusterPairUnroll = 8;

__global__ void __launch_bounds__(kThreads) cap_cluster_kernel(CapArgs a) {
    __shared__ __align__(16) float s_c[kThreads];
    __shared__ __align__(4) unsigned char s_cand[kThreads];
    __shared__ int s_pool[DLM_MAX_BLK];
    __shared__ int s_row[DLM_MAX_BLK];
    __shared__ int s_y[DLM_MAX_BLK];
    __shared__ float s_lse[DLM_MAX_BLK];
    __shared__ uint32_t s_adj[DLM_MAX_BLK * kMaxPoolWords];
    __shared__ uint32_t s_kept[kMaxPoolWords];
    __shared__ unsigned char s_tier[DLM_MAX_BLK];
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int b = blockIdx.x / kCapCluster;
    const int t = threadIdx.x;
    const int scope = scope_of(a, b);
    const int64_t o = (int64_t)b * a.blk + t;

    // 1. the pool, in every CTA of the cluster
    const bool in = t < a.blk;
    const bool m = t < scope && a.masked[o] != 0;
    const float c = in ? a.conf[o] : 0.f;
    const int y = in ? a.argmax[o] : 0;
    const float l = in ? a.lse[o] : 0.f;
    const bool cand = m && c >= a.tau_low;
    const int row = cand ? row_of(a, b, t) : 0;
    s_c[t] = c;
    s_cand[t] = cand;
    for (int k = t; k < DLM_MAX_BLK * kMaxPoolWords; k += kThreads) s_adj[k] = 0u;
    const int n_cand = __syncthreads_count(cand);
    const int n = min(n_cand, a.p_max);
    if (cand) {
        const int rank = rank_desc(s_c, s_cand, (scope + 3) & ~3, c, t);
        if (rank < a.p_max) {
            s_pool[rank] = t;
            s_row[rank] = row;
            s_y[rank] = y;
            s_lse[rank] = l;
            s_tier[rank] = a.high_tier_unconditional && c >= a.tau_high;
        }
    }
    cluster.sync();  // pools ranked and the leader's bitmask zeroed, cluster-wide

    // 2. the pairs, split over the cluster; bits land in the leader's bitmask
    uint32_t* adj0 = cluster.map_shared_rank(s_adj, 0);
    const int pairs = n * (n - 1) / 2;
    const int stride = kThreads * kCapCluster;
    for (int q0 = crank * kThreads + t; q0 < pairs; q0 += stride * kClusterPairUnroll) {
        int pi[kClusterPairUnroll], pj[kClusterPairUnroll];
        float dv[kClusterPairUnroll];
#pragma unroll
        for (int u = 0; u < kClusterPairUnroll; ++u) {
            // an index past the last pair maps to the pair (0, 1), which
            // exists (pairs >= 1); its result is dropped
            pair_of(min(q0 + u * stride, pairs - 1), n, pi[u], pj[u]);
        }
#pragma unroll
        for (int u = 0; u < kClusterPairUnroll; ++u) {
            dv[u] = logp_at(a, s_row[pi[u]], s_y[pj[u]], s_lse[pi[u]]) +
                    logp_at(a, s_row[pj[u]], s_y[pi[u]], s_lse[pj[u]]);
        }
#pragma unroll
        for (int u = 0; u < kClusterPairUnroll; ++u) {
            if (q0 + u * stride >= pairs) break;
            const int i = pi[u], j = pj[u];
            if (dv[u] > a.gamma) {
                atomicOr(adj0 + i * kMaxPoolWords + (j >> 5), 1u << (j & 31));
                atomicOr(adj0 + j * kMaxPoolWords + (i >> 5), 1u << (i & 31));
            }
            if (a.D_out) {
                a.D_out[((int64_t)b * a.blk + s_pool[i]) * a.blk + s_pool[j]] = dv[u];
                a.D_out[((int64_t)b * a.blk + s_pool[j]) * a.blk + s_pool[i]] = dv[u];
            }
        }
    }
    cluster.sync();  // every conflict bit is in the leader's bitmask
    if (crank != 0) return;

    // 3. the leader: greedy scan, or the fallback when the pool is empty
    uint8_t* sel = a.selected + (int64_t)b * a.blk;
    if (in) sel[t] = 0;
    if (t == 0 && n_cand > a.p_max) raise_status(a.dev_status, DLM_DEV_POOL_CLIPPED);
    __syncthreads();
    if (n == 0) {
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
    const int W = (n + 31) >> 5;
    if (t < 32) {
        const uint32_t kept = greedy_scan_chunked(s_adj, kMaxPoolWords, s_tier, n);  // slots are in pool order
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCapCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(a.batch * kCapCluster));
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cap_cluster_kernel, a);
}

}  // namespace dlm
