// select.cu -- Fast-dLLM threshold selection, the DepGA-Block boundary, the
// fixed top-K and factor-decoding rules and the Theorem-1 certificate.
//
// All are per-sequence decisions over at most a few hundred values, so each
// sequence is one CTA working out of registers and shared memory; the cost is
// launch latency, not bandwidth.
#include "common.cuh"
#include "launch.h"
#include "rules.cuh"

namespace dlm {

namespace {

constexpr int kSelThreads = kRuleThreads;  // >= DLM_MAX_BLK: one position per thread
constexpr int kBndThreads = kRuleThreads;
constexpr int kMaxWindow = 1024;

// Fast-dLLM threshold rule, one CTA per sequence (rules.cuh: threshold_block).
__global__ void __launch_bounds__(kSelThreads) threshold_kernel(ThresholdArgs a) {
    __shared__ ThresholdSmem sm;
    threshold_block(a, blockIdx.x, sm);
}

// DepGA-Block boundary, one CTA per sequence (rules.cuh: boundary_block).
__global__ void __launch_bounds__(kBndThreads) boundary_kernel(BoundaryArgs a) {
    __shared__ BoundarySmem<kMaxWindow> sm;
    boundary_block<kMaxWindow>(a, blockIdx.x, sm);
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
