// select.cu -- Fast-dLLM threshold selection, the DepGA-Block boundary, the
// fixed top-K and factor-decoding rules and the Theorem-1 certificate.
//
// All are per-sequence decisions over at most a few hundred values, so each
// sequence is one CTA working out of registers and shared memory; the cost is
// launch latency, not bandwidth.
#include "common.cuh"
#include "launch.h"

namespace dlm {

namespace {

constexpr int kSelThreads = 256;  // >= DLM_MAX_BLK: one position per thread

// Fast-dLLM review, "Method"; Fast-dLLM notes, "Key ideas" (safety valve):
// keep masked positions with conf > tau, else the top-confidence masked one.
__global__ void __launch_bounds__(kSelThreads) threshold_kernel(ThresholdArgs a) {
    __shared__ float s_v[kSelThreads / 32];
    __shared__ int s_i[kSelThreads / 32];
    const int b = blockIdx.x, i = threadIdx.x;
    const bool valid = i < a.blk;
    const int64_t o = (int64_t)b * a.blk + i;
    const bool m = valid && a.masked[o] != 0;
    const float c = m ? a.conf[o] : 0.f;
    bool s = m && c > a.tau;
    int n = __syncthreads_count(s);
    const int any_m = __syncthreads_or(m);
    if (n == 0 && any_m) {
        float v = m ? c : -INFINITY;
        int idx = m ? i : 0x7fffffff;
        warp_argmax(v, idx);
        if ((i & 31) == 0) {
            s_v[i >> 5] = v;
            s_i[i >> 5] = idx;
        }
        __syncthreads();
        if (i < 32) {
            v = i < kSelThreads / 32 ? s_v[i] : -INFINITY;
            idx = i < kSelThreads / 32 ? s_i[i] : 0x7fffffff;
            warp_argmax(v, idx);
            if (i == 0) s_i[0] = idx;
        }
        __syncthreads();
        s = (i == s_i[0]);
        n = 1;
    }
    if (valid) a.selected[o] = s ? 1 : 0;
    if (i == 0) a.n_selected[b] = n;
}

// Block-wide sum in a fixed order (thread-strided partial sums, then a tree).
__device__ float block_sum(float v, float* red) {
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

__device__ float block_min(float v, float* red) {
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

constexpr int kBndThreads = 256;
constexpr int kMaxWindow = 1024;

// DepCap, "Methodology": S_k = I~_k - lambda H~_k over the window, stop before
// the first negative, clip to [L_min, L_window], cold start -> L_min.
// Smoothing: centred moving average of odd width, edge-truncated.
// Normalisation: 0 window mean, 1 min-max, 2 none.
// Ragged windows: with window_len, sequence b uses the first window_len[b]
// entries of its row (row stride L_window); an empty window gives length 0.
__global__ void __launch_bounds__(kBndThreads) boundary_kernel(BoundaryArgs a) {
    __shared__ float sI[kMaxWindow], sH[kMaxWindow], tI[kMaxWindow], tH[kMaxWindow];
    __shared__ float red[kBndThreads / 32];
    const int b = blockIdx.x;
    const int L = a.window_len ? min(max(a.window_len[b], 0), a.L_window) : a.L_window;
    const int64_t row = (int64_t)b * a.L_window;
    if (L == 0) {  // uniform over the CTA
        if (threadIdx.x == 0) a.block_len[b] = 0;
        return;
    }
    const float* I = a.kl + row;
    const float* H = a.entropy + row;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        sI[k] = I[k];
        sH[k] = H[k];
    }
    __syncthreads();
    const int h = a.smooth_w / 2;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        const int lo = max(0, k - h), hi = min(L - 1, k + h);
        float ai = 0.f, ah = 0.f;
        for (int j = lo; j <= hi; ++j) {
            ai += sI[j];
            ah += sH[j];
        }
        const float cnt = (float)(hi - lo + 1);
        tI[k] = ai / cnt;
        tH[k] = ah / cnt;
    }
    __syncthreads();
    float mulI = 1.f, addI = 0.f, mulH = 1.f, addH = 0.f;
    if (a.norm_mode == 0) {
        float pi = 0.f, ph = 0.f;
        for (int k = threadIdx.x; k < L; k += blockDim.x) {
            pi += tI[k];
            ph += tH[k];
        }
        const float mi = fmaxf(block_sum(pi, red) / (float)L, 1e-12f);
        const float mh = fmaxf(block_sum(ph, red) / (float)L, 1e-12f);
        mulI = 1.f / mi;
        mulH = 1.f / mh;
    } else if (a.norm_mode == 1) {
        float mni = INFINITY, mnh = INFINITY, mxi = -INFINITY, mxh = -INFINITY;
        for (int k = threadIdx.x; k < L; k += blockDim.x) {
            mni = fminf(mni, tI[k]);
            mxi = fmaxf(mxi, tI[k]);
            mnh = fminf(mnh, tH[k]);
            mxh = fmaxf(mxh, tH[k]);
        }
        mni = block_min(mni, red);
        mnh = block_min(mnh, red);
        mxi = -block_min(-mxi, red);
        mxh = -block_min(-mxh, red);
        mulI = mxi > mni ? 1.f / (mxi - mni) : 0.f;
        addI = -mni;
        mulH = mxh > mnh ? 1.f / (mxh - mnh) : 0.f;
        addH = -mnh;
    }
    float first = (float)L;
    for (int k = threadIdx.x; k < L; k += blockDim.x) {
        float ni, nh;
        if (a.norm_mode == 0) {
            ni = tI[k] * mulI;
            nh = tH[k] * mulH;
        } else if (a.norm_mode == 1) {
            ni = (tI[k] + addI) * mulI;
            nh = (tH[k] + addH) * mulH;
        } else {
            ni = tI[k];
            nh = tH[k];
        }
        const float s = ni - a.lambda * nh;
        if (a.score) a.score[row + k] = s;
        if (s < 0.f) first = fminf(first, (float)k);
    }
    const float kstar = block_min(first, red);
    if (threadIdx.x == 0) {
        int len = max((int)kstar, a.L_min);
        len = min(len, L);
        if (a.cold_start && a.cold_start[b]) len = min(a.L_min, L);
        a.block_len[b] = len;
    }
}

// Fixed top-K (Fast-dLLM review, Prior limitations: LLaDA's default commits
// K tokens per step whatever their confidence) and factor decoding (Fast-dLLM
// review, Method, appendix variant: the largest n with (n+1)(1 - c^(n)) < f,
// the top position alone when no n qualifies).  mode 0 = top-K, 1 = factor.
__global__ void __launch_bounds__(kSelThreads) rank_select_kernel(RankSelectArgs a) {
    __shared__ __align__(16) float s_c[kSelThreads];
    __shared__ __align__(4) unsigned char s_m[kSelThreads];
    const int b = blockIdx.x, i = threadIdx.x;
    const bool valid = i < a.blk;
    const int64_t o = (int64_t)b * a.blk + i;
    const bool m = valid && a.masked[o] != 0;
    s_c[i] = m ? a.conf[o] : 0.f;
    s_m[i] = m;
    const int M = __syncthreads_count(m);
    // rank in (conf desc, position asc) order among the masked positions
    const int r = m ? rank_desc(s_c, s_m, (a.blk + 3) & ~3, s_c[i], i) : 0x7fffffff;
    int n;
    if (a.mode == 0) {
        n = min(a.k, M);
    } else {
        const bool ok = m && __fmul_rn((float)(r + 2), __fsub_rn(1.0f, s_c[i])) < a.f;
        n = __syncthreads_count(ok);  // the qualifying n form a prefix of the order
        if (n == 0 && M > 0) n = 1;
    }
    if (valid) a.selected[o] = (m && r < n) ? 1 : 0;
    if (i == 0) a.n_selected[b] = n;
}

// Theorem-1 certificate (Fast-dLLM review, Key idea): every one of the n
// selected positions has confidence above 1 - 1/(n+1); an empty selection is
// certified.
__global__ void __launch_bounds__(kSelThreads) certificate_kernel(CertificateArgs a) {
    const int b = blockIdx.x, i = threadIdx.x;
    const bool valid = i < a.blk;
    const int64_t o = (int64_t)b * a.blk + i;
    const bool s = valid && a.selected[o] != 0;
    const int n = __syncthreads_count(s);
    const float bound = __fsub_rn(1.0f, __fdiv_rn(1.0f, (float)(n + 1)));
    const bool bad = s && !(a.conf[o] > bound);
    const int any_bad = __syncthreads_or(bad);
    if (i == 0) a.certified[b] = any_bad ? 0 : 1;
}

}  // namespace

cudaError_t launch_threshold(const ThresholdArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, threshold_kernel, a);
}

cudaError_t launch_rank_select(const RankSelectArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, rank_select_kernel, a);
}

cudaError_t launch_certificate(const CertificateArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, certificate_kernel, a);
}

cudaError_t launch_boundary(const BoundaryArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kBndThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, boundary_kernel, a);
}

}  // namespace dlm
