// revocable.cu -- one state update of revocable parallel decoding (COVER
// page: "Revocable Parallel Diffusion Decoding"; "Method": KEEP / REPLACE /
// REMASK outcomes, stability-aware seed selection, seed count
// ceil(sqrt(n) pi)).
//
// One CTA per sequence, one thread per block position (blk <= 256); the
// state lives in registers for the step and the two rankings (drafting by
// confidence, next seeds by score) count dominating keys in shared memory.
// The work is a few hundred values per sequence: launch latency bounds it.
#include "common.cuh"
#include "launch.h"

namespace dlm {

namespace {

constexpr int kRevThreads = 256;  // >= DLM_MAX_BLK

__global__ void __launch_bounds__(kRevThreads) revocable_kernel(RevocableArgs a) {
    __shared__ __align__(16) float s_key[kRevThreads];
    __shared__ __align__(4) unsigned char s_flag[kRevThreads];
    __shared__ float s_v[kRevThreads / 32];
    __shared__ int s_i[kRevThreads / 32];
    const int b = blockIdx.x, i = threadIdx.x;
    const bool valid = i < a.blk;
    const int64_t o = (int64_t)b * a.blk + i;
    const bool m0 = valid && a.masked[o] != 0;
    if (__syncthreads_count(m0) == 0) {  // finished sequence: nothing changes
        if (valid && a.outcome) a.outcome[o] = 0;
        if (i == 0) {
            if (a.n_drafted) a.n_drafted[b] = 0;
            if (a.n_revoked) a.n_revoked[b] = 0;
        }
        return;
    }
    int tok = valid ? a.tok[o] : -1;
    const int am = valid ? a.argmax[o] : 0;
    const float c = valid ? a.conf[o] : 0.f;
    int remasks = valid ? a.remasks[o] : 0;
    int last_tok = valid ? a.last_tok[o] : -1;
    int last_seed = valid ? a.last_seed[o] : 0;
    bool msk = m0;
    int out = 0;

    // 1. verification of the seeds
    if (valid && a.seed[o] != 0 && !m0) {
        if (am == tok) {
            out = 2;
        } else if (c >= a.tau_replace) {
            out = 3;
            tok = am;
        } else {
            out = 4;
            last_tok = tok;
            tok = -1;
            msk = true;
            remasks += 1;
        }
    }
    const int n_revoked = __syncthreads_count(out == 4);

    // 2. drafting over the positions masked at the start of the step
    const bool cand = m0 && c > a.tau_draft;
    s_key[i] = c;
    s_flag[i] = cand ? 1 : 0;
    const int n_cand = __syncthreads_count(cand);
    bool drafted;
    int n_drafted;
    if (n_cand > 0) {
        n_drafted = a.draft_budget > 0 ? min(n_cand, a.draft_budget) : n_cand;
        drafted = cand && rank_desc(s_key, s_flag, (a.blk + 3) & ~3, s_key[i], i) < n_drafted;
    } else {  // nothing clears the threshold: the most confident masked position
        float v = m0 ? c : -INFINITY;
        int idx = m0 ? i : 0x7fffffff;
        warp_argmax(v, idx);
        if ((i & 31) == 0) {
            s_v[i >> 5] = v;
            s_i[i >> 5] = idx;
        }
        __syncthreads();
        if (i < 32) {
            v = i < kRevThreads / 32 ? s_v[i] : -INFINITY;
            idx = i < kRevThreads / 32 ? s_i[i] : 0x7fffffff;
            warp_argmax(v, idx);
            if (i == 0) s_i[0] = idx;
        }
        __syncthreads();
        drafted = (i == s_i[0]);
        n_drafted = 1;
    }
    if (drafted) {
        out = 1;
        tok = am;
        msk = false;
    }
    const int n_flip = __syncthreads_count(drafted && last_tok == am);

    // 3. the next step's seeds
    const bool elig = valid && !msk && (a.step - last_seed > a.cooldown) && remasks < a.remask_budget;
    float score = 0.f;
    if (elig) {
        const float infl = a.influence ? a.influence[o] : 0.f;
        const float drift = a.drift ? a.drift[o] : 0.f;
        const float t_unc = __fmul_rn(a.w_unc, __fsub_rn(1.0f, c));
        const float t_infl = __fmul_rn(a.w_infl, infl);
        const float t_drift = __fmul_rn(a.w_drift, drift);
        score = __fsub_rn(__fadd_rn(t_unc, t_infl), t_drift);
    }
    __syncthreads();  // the drafting ranks are done with s_key / s_flag
    s_key[i] = score;
    s_flag[i] = elig ? 1 : 0;
    const int n_elig = __syncthreads_count(elig);
    const float kf = ceilf(__fmul_rn(__fsqrt_rn((float)n_elig), a.pi));
    const int k = kf < (float)n_elig ? (int)kf : n_elig;
    const bool seed_next = elig && rank_desc(s_key, s_flag, (a.blk + 3) & ~3, s_key[i], i) < k;
    if (seed_next) last_seed = a.step;

    if (valid) {
        a.tok[o] = tok;
        a.masked[o] = msk ? 1 : 0;
        a.seed[o] = seed_next ? 1 : 0;
        a.last_seed[o] = last_seed;
        a.remasks[o] = remasks;
        a.last_tok[o] = last_tok;
        if (a.outcome) a.outcome[o] = (uint8_t)out;
    }
    if (i == 0) {
        if (a.n_drafted) a.n_drafted[b] = n_drafted;
        if (a.n_revoked) a.n_revoked[b] = n_revoked;
        if (a.flipflops) a.flipflops[b] += n_flip;
    }
}

}  // namespace

cudaError_t launch_revocable(const RevocableArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kRevThreads);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, revocable_kernel, a);
}

}  // namespace dlm
