// row_stats.cu -- fused streaming pass over vocab-wide logit rows.
//
// Per row (DepCap "Methodology": I_k = KL(p_curr || p_prev), H_k = H(p_curr),
// c = max_v p(v); Fast-dLLM review "Method": max-softmax confidence) one pass
// over the current row and, optionally, the previous step's row produces
// argmax, confidence, log-sum-exp, entropy, KL(cur || prev) and the previous
// row's log-sum-exp.
//
// Design (HBM-bound, ~1 flop per byte):
//  * one CTA (or a cluster of `split` CTAs when there are too few rows to
//    fill 152 SMs) streams a row with coalesced 16-byte loads that bypass L1;
//  * each thread keeps an online softmax state relative to a lazily moved
//    reference (moved only when a value exceeds it by more than kRebase, so
//    the common path has no rescale), in base-2 units so every element costs
//    a subtract, a multiply and one ex2 on the SFU; the arithmetic is done on
//    packed f32x2;
//  * the exact maximum is tracked per 8-element vector and the argmax position
//    is recovered at the end by re-reading the winning vector, ties to the
//    lowest index everywhere;
//  * partial states merge through warp shuffles, shared memory and, for split
//    rows, distributed shared memory inside the cluster; the merge order is
//    fixed, so results are deterministic;
//  * row_stats_attn_kernel (few-row launches) also computes the DAPD
//    attention sums of its row: the runs are copied into shared memory with
//    asynchronous copies before the logits stream and summed afterwards
//    (attn_sum.cuh), so their latency hides under the row.
// Every quantity is independent of the reference r:
//   S = sum 2^{a_v}, a_v = (z_v - r) log2 e,  T = sum 2^{a_v} a_v,
//   K = sum 2^{a_v} (z_v - z'_v):
//   lse = r + ln S, conf = exp(max z - r) / S, H = ln S - ln2 T/S,
//   KL = K/S - (r - r') - (ln S - ln S').
#include <cooperative_groups.h>

#include <cstddef>

#include "attn_sum.cuh"
#include "common.cuh"
#include "launch.h"
#include "rules.cuh"

namespace cg = cooperative_groups;

namespace dlm {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr float kRebase = 8.0f;    // e^8 of headroom before the reference moves
constexpr float kFloorLog2 = -256.0f;
constexpr float kClampLo = -1e30f;                 // lower clamp of bf16 / f32 logits
constexpr unsigned short kClampBf16 = 0xf14a;        // -1e30 rounded to bf16
constexpr float kDegenerate = -1e29f;              // a row whose max is below this held only -inf

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// partial state of a slice of one row
struct Part {
    float mx;   // exact max of the (clamped) stored values
    int idx;    // first position holding mx
    float ref;  // softmax reference
    float S, T, K;
    float refp, Sp;
};

static_assert(sizeof(Part) == sizeof(dlm_row_partial), "Part mirrors dlm_row_partial");
static_assert(offsetof(Part, idx) == offsetof(dlm_row_partial, idx) &&
                  offsetof(Part, S) == offsetof(dlm_row_partial, S) &&
                  offsetof(Part, refp) == offsetof(dlm_row_partial, ref_prev) &&
                  offsetof(Part, Sp) == offsetof(dlm_row_partial, S_prev),
              "Part mirrors dlm_row_partial");

__device__ __forceinline__ void part_empty(Part& p) {
    p.mx = -INFINITY;
    p.idx = 0x7fffffff;
    p.ref = -FLT_MAX;
    p.S = p.T = p.K = 0.f;
    p.refp = -FLT_MAX;
    p.Sp = 0.f;
}

__device__ __forceinline__ void part_merge(Part& a, const Part& b) {
    if (b.mx > a.mx || (b.mx == a.mx && b.idx < a.idx)) {
        a.mx = b.mx;
        a.idx = b.idx;
    }
    float r = fmaxf(a.ref, b.ref);
    float da = fmaxf((a.ref - r) * kLog2e, kFloorLog2);
    float db = fmaxf((b.ref - r) * kLog2e, kFloorLog2);
    float ea = ex2(da), eb = ex2(db);
    a.T = ea * fmaf(da, a.S, a.T) + eb * fmaf(db, b.S, b.T);
    a.S = ea * a.S + eb * b.S;
    a.K = ea * a.K + eb * b.K;
    a.ref = r;
    float rp = fmaxf(a.refp, b.refp);
    float dpa = fmaxf((a.refp - rp) * kLog2e, kFloorLog2);
    float dpb = fmaxf((b.refp - rp) * kLog2e, kFloorLog2);
    a.Sp = ex2(dpa) * a.Sp + ex2(dpb) * b.Sp;
    a.refp = rp;
}

__device__ __forceinline__ Part part_shfl(const Part& p, int o) {
    Part q;
    q.mx = __shfl_xor_sync(DLM_FULL_MASK, p.mx, o);
    q.idx = __shfl_xor_sync(DLM_FULL_MASK, p.idx, o);
    q.ref = __shfl_xor_sync(DLM_FULL_MASK, p.ref, o);
    q.S = __shfl_xor_sync(DLM_FULL_MASK, p.S, o);
    q.T = __shfl_xor_sync(DLM_FULL_MASK, p.T, o);
    q.K = __shfl_xor_sync(DLM_FULL_MASK, p.K, o);
    q.refp = __shfl_xor_sync(DLM_FULL_MASK, p.refp, o);
    q.Sp = __shfl_xor_sync(DLM_FULL_MASK, p.Sp, o);
    return q;
}

__device__ __forceinline__ void warp_merge(Part& p) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        Part q = part_shfl(p, o);
        // combine in a fixed (lower lane first) order so every lane agrees
        if (threadIdx.x & o) {
            Part lo = q;
            part_merge(lo, p);
            p = lo;
        } else {
            part_merge(p, q);
        }
    }
}

// ---- storage formats --------------------------------------------------
// A 16-byte vector is unpacked into NP packed pairs of fp32 and its max.
// Values are clamped from below (NaN is kept) so that -inf logits become a
// large finite negative number: its exponential is exactly 0 and its product
// with the base-2 scaling stays finite, so 0 * (z - r) terms stay 0.  The
// clamp is -1e30 for bf16/f32 storage and the f16 minimum for f16.
template <int DT>
struct Fmt;

template <>
struct Fmt<DLM_BF16> {
    static constexpr int EPV = 8;
    static constexpr int ESZ = 2;
    static __device__ __forceinline__ float scalar(const void* base, int64_t i) {
        uint32_t b = static_cast<const uint16_t*>(base)[i];
        return max_nan(__uint_as_float(b << 16), __uint_as_float((uint32_t)kClampBf16 << 16));
    }
    static __device__ __forceinline__ float unpack(uint4 w, f2 (&z)[4]) {
        const __nv_bfloat162 lo = __halves2bfloat162(__ushort_as_bfloat16(kClampBf16), __ushort_as_bfloat16(kClampBf16));
        uint32_t r[4] = {w.x, w.y, w.z, w.w};
        __nv_bfloat162 m;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&r[k]);
            h = __hmax2_nan(h, lo);
            m = k ? __hmax2(m, h) : h;
            r[k] = *reinterpret_cast<uint32_t*>(&h);
            z[k] = bf16x2_to_f2(r[k]);
        }
        return fmaxf(__low2float(m), __high2float(m));
    }
};

template <>
struct Fmt<DLM_F16> {
    static constexpr int EPV = 8;
    static constexpr int ESZ = 2;
    static __device__ __forceinline__ float scalar(const void* base, int64_t i) {
        return max_nan(__half2float(static_cast<const __half*>(base)[i]), -65504.f);
    }
    static __device__ __forceinline__ float unpack(uint4 w, f2 (&z)[4]) {
        const __half2 lo = __halves2half2(__ushort_as_half(0xfbff), __ushort_as_half(0xfbff));
        uint32_t r[4] = {w.x, w.y, w.z, w.w};
        __half2 m;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = *reinterpret_cast<__half2*>(&r[k]);
            h = __hmax2_nan(h, lo);
            m = k ? __hmax2(m, h) : h;
            r[k] = *reinterpret_cast<uint32_t*>(&h);
            z[k] = f16x2_to_f2(r[k]);
        }
        return fmaxf(__low2float(m), __high2float(m));
    }
};

template <>
struct Fmt<DLM_F32> {
    static constexpr int EPV = 4;
    static constexpr int ESZ = 4;
    static __device__ __forceinline__ float scalar(const void* base, int64_t i) {
        return max_nan(static_cast<const float*>(base)[i], kClampLo);
    }
    static __device__ __forceinline__ float unpack(uint4 w, f2 (&z)[2]) {
        float a = max_nan(__uint_as_float(w.x), kClampLo);
        float b = max_nan(__uint_as_float(w.y), kClampLo);
        float c = max_nan(__uint_as_float(w.z), kClampLo);
        float d = max_nan(__uint_as_float(w.w), kClampLo);
        z[0] = pack2(a, b);
        z[1] = pack2(c, d);
        return fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
};

// per-thread accumulator
struct Acc {
    float mx;
    int bv;     // vector holding mx (first), or -1 when it came from the tail
    int bidx;   // position when it came from the tail
    float ref;
    f2 S, T, K;
    float refp;
    f2 Sp;
};

__device__ __forceinline__ void rebase(Acc& a, float nref) {
    float d = fmaxf((a.ref - nref) * kLog2e, kFloorLog2);
    float al = ex2(d);
    f2 d2 = pack2(d, d), al2 = pack2(al, al);
    a.T = mul2(al2, fma2(d2, a.S, a.T));
    a.S = mul2(al2, a.S);
    a.K = mul2(al2, a.K);
    a.ref = nref;
}

__device__ __forceinline__ void rebase_p(Acc& a, float nref) {
    float d = fmaxf((a.refp - nref) * kLog2e, kFloorLog2);
    float al = ex2(d);
    a.Sp = mul2(pack2(al, al), a.Sp);
    a.refp = nref;
}

template <int NP, bool PREV>
__device__ __forceinline__ void accum(Acc& a, const f2 (&z)[NP], const f2 (&zp)[NP]) {
    // x = (z - r) log2 e: the subtraction is exact for nearby values, so x
    // carries one rounding whatever the magnitude of r
    const f2 l2e = pack2(kLog2e, kLog2e);
    const f2 r = pack2(a.ref, a.ref);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        f2 x = mul2(sub2(z[p], r), l2e);
        f2 e = ex2x2(x);
        a.S = add2(a.S, e);
        a.T = fma2(e, x, a.T);
        if (PREV) a.K = fma2(e, sub2(z[p], zp[p]), a.K);
    }
    if (PREV) {
        const f2 rp = pack2(a.refp, a.refp);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            f2 x = mul2(sub2(zp[p], rp), l2e);
            a.Sp = add2(a.Sp, ex2x2(x));
        }
    }
}

template <int DT, bool PREV>
__device__ __forceinline__ void process_vec(Acc& a, uint4 cw, uint4 pw, int v) {
    constexpr int NP = Fmt<DT>::EPV / 2;
    f2 z[NP], zp[NP];
    float vmax = Fmt<DT>::unpack(cw, z);
    float vmaxp = 0.f;
    if (PREV) vmaxp = Fmt<DT>::unpack(pw, zp);
    if (vmax > a.mx) {
        a.mx = vmax;
        a.bv = v;
    }
    if (vmax > a.ref + kRebase) rebase(a, vmax);
    if (PREV && vmaxp > a.refp + kRebase) rebase_p(a, vmaxp);
    accum<NP, PREV>(a, z, zp);
}

template <bool PREV>
__device__ __forceinline__ void process_scalar(Acc& a, float z, float zp, int pos) {
    if (z > a.mx) {
        a.mx = z;
        a.bv = -1;
        a.bidx = pos;
    }
    if (z > a.ref + kRebase) rebase(a, z);
    if (PREV && zp > a.refp + kRebase) rebase_p(a, zp);
    // scalar form of accum (keeps the pair layout: only the low lane is used)
    float x = (z - a.ref) * kLog2e;
    float e = ex2(x);
    a.S = add2(a.S, pack2(e, 0.f));
    a.T = fma2(pack2(e, 0.f), pack2(x, 0.f), a.T);
    if (PREV) {
        a.K = fma2(pack2(e, 0.f), pack2(z - zp, 0.f), a.K);
        float xp = (zp - a.refp) * kLog2e;
        a.Sp = add2(a.Sp, pack2(ex2(xp), 0.f));
    }
}

// The outputs of a row from its merged state (one thread).
template <bool PREV>
__device__ __forceinline__ void write_outputs(const RowStatsArgs& args, const Part& p, int64_t q) {
    const float lnS = logf(p.S);
    const float lse = p.ref + lnS;
    // a row of NaN only has no maximum: position 0 (the status flags the row)
    args.argmax[q] = p.idx != 0x7fffffff ? p.idx : 0;
    args.lse[q] = lse;
    // max p = e^{max - ref} / S: max - ref is exact (nearby values) and in
    // [0, kRebase], so no cancellation against ln S
    args.conf[q] = expf(p.mx - p.ref) / p.S;
    args.entropy[q] = lnS - kLn2 * (p.T / p.S);
    bool ok = isfinite(p.S) && p.S > 0.f && isfinite(p.T) && isfinite(p.mx) && p.mx > kDegenerate;
    if (PREV) {
        const float lnSp = logf(p.Sp);
        if (args.kl) args.kl[q] = p.K / p.S - (p.ref - p.refp) - (lnS - lnSp);
        if (args.lse_prev) args.lse_prev[q] = p.refp + lnSp;
        ok = ok && isfinite(p.Sp) && p.Sp > 0.f && isfinite(p.K);
    }
    if (!ok) raise_status(args.dev_status, DLM_DEV_NONFINITE);
}

// The rules the CTA that finishes a sequence's last row runs (fused row
// pass); one shared-memory area serves them in turn.
union RuleSmem {
    ThresholdSmem t;
    BoundarySmem<DLM_MAX_BLK> d;
    CapSmem c;
};

__device__ __forceinline__ void run_rules(const RowRules& rr, int b, RuleSmem& sm) {
    if (rr.thr) threshold_block(rr.t, b, sm.t);
    __syncthreads();
    if (rr.bnd) boundary_block<DLM_MAX_BLK>(rr.d, b, sm.d);
    __syncthreads();  // the block length is visible to CAP's scope
    if (rr.cap) cap_block(rr.c, b, sm.c);
}

// shared memory of the folded attention: the copied runs, the sequence's
// mask flags, then the partials of the sums
__host__ __device__ __forceinline__ size_t attn_buf_bytes(const RowAttn& at) {
    return ((size_t)at.n_layers * at.n_heads * at.vpr * 16 + 15) & ~(size_t)15;
}
__host__ __device__ __forceinline__ size_t attn_red_offset(const RowAttn& at) {
    return attn_buf_bytes(at) + (((size_t)at.blk + 15) & ~(size_t)15);
}

// The DAPD attention sums folded into the row pass.  Row r = b*blk + i: the
// CTA copies row i of sequence b's attention block for every (layer, head)
// -- L*H runs of blk contiguous values -- into shared memory with
// asynchronous 16-byte copies issued before it streams the logits, so the
// scattered reads wait under the stream instead of after it.
__device__ __forceinline__ void attn_prefetch(const RowAttn& at, int64_t r, unsigned char* buf) {
    const int b = (int)(r / at.blk), i = (int)(r - (int64_t)b * at.blk);
    const char* base = static_cast<const char*>(at.attn) +
                       ((int64_t)b * at.sb + (int64_t)(at.block_start + i) * at.sr + at.block_start) * at.esz;
    const int LH = at.n_layers * at.n_heads, nq = LH * at.vpr;
    for (int q = threadIdx.x; q < nq; q += kThreads) {
        const int s = q / at.vpr, cv = q - s * at.vpr;
        const int l = s / at.n_heads, h = s - l * at.n_heads;
        cp_async16(buf + (size_t)q * 16, base + ((int64_t)l * at.sl + (int64_t)h * at.sh) * at.esz + cv * 16);
    }
    if (at.mask4 && (int)threadIdx.x < at.blk / 4)  // the sequence's mask flags, 4 at a time
        cp_async4(buf + attn_buf_bytes(at) + threadIdx.x * 4, at.masked + (int64_t)b * at.blk + threadIdx.x * 4);
}

// Thread t sums column vector t % vpr of the runs t / vpr, t / vpr + per, ...
// (exact hi / lo split); the partials meet in `red` (component-major) and
// thread j < blk adds column j's and stores A[b][i][j] in fixed point.
template <int AT>
__device__ __forceinline__ void attn_row_sums_typed(const RowAttn& at, int b, int i, const unsigned char* buf,
                                                    float* red) {
    constexpr int EPV = AFmt<AT>::EPV;
    constexpr int NP = EPV / 2;
    const int t = threadIdx.x, vpr = at.vpr, per = kThreads / vpr;
    const int LH = at.n_layers * at.n_heads;
    const int g = t / vpr, cv = t - g * vpr;
    f2 H[NP], L[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) H[p] = L[p] = pack2(0.f, 0.f);
    if (g < per) {
        for (int s = g; s < LH; s += per) {
            const uint4 w = *reinterpret_cast<const uint4*>(buf + ((size_t)s * vpr + cv) * 16);
            f2 x[NP];
            AFmt<AT>::to_f2(w, x);
            split_acc<NP>(x, H, L);
        }
    }
    if ((32 % vpr) == 0) {
        // lanes l, l + vpr, l + 2 vpr, ... of a warp hold the same column
        // vector: shuffles add them, then lane cv < vpr of each warp leaves the
        // warp's partial and thread j adds the warps' (kWarps terms)
        for (int off = vpr; off < 32; off <<= 1) {
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                float h0, h1, l0, l1;
                unpack2(H[p], h0, h1);
                unpack2(L[p], l0, l1);
                h0 += __shfl_xor_sync(DLM_FULL_MASK, h0, off);
                h1 += __shfl_xor_sync(DLM_FULL_MASK, h1, off);
                l0 += __shfl_xor_sync(DLM_FULL_MASK, l0, off);
                l1 += __shfl_xor_sync(DLM_FULL_MASK, l1, off);
                H[p] = pack2(h0, h1);
                L[p] = pack2(l0, l1);
            }
        }
        const int lane = t & 31, warp = t >> 5;
        if (lane < vpr) {
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                float h0, h1, l0, l1;
                unpack2(H[p], h0, h1);
                unpack2(L[p], l0, l1);
                float* o = red + (size_t)(warp * vpr + lane) * (2 * EPV);
                o[4 * p + 0] = h0;
                o[4 * p + 1] = h1;
                o[4 * p + 2] = l0;
                o[4 * p + 3] = l1;
            }
        }
        __syncthreads();
        if (t < at.blk) {
            const int cj = t / EPV, e = t - cj * EPV, p = e >> 1, c = e & 1;
            float hi = 0.f, lo = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* o = red + (size_t)(w * vpr + cj) * (2 * EPV);
                hi += o[4 * p + c];
                lo += o[4 * p + 2 + c];
            }
            at.A[((int64_t)b * at.blk + i) * at.blk + t] = attn_fixed(hi, lo);
        }
        return;
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        float h0, h1, l0, l1;
        unpack2(H[p], h0, h1);
        unpack2(L[p], l0, l1);
        red[(4 * p + 0) * kThreads + t] = h0;
        red[(4 * p + 1) * kThreads + t] = h1;
        red[(4 * p + 2) * kThreads + t] = l0;
        red[(4 * p + 3) * kThreads + t] = l1;
    }
    __syncthreads();
    if (t < at.blk) {
        const int cj = t / EPV, e = t - cj * EPV, p = e >> 1, c = e & 1;
        float hi = 0.f, lo = 0.f;
        for (int gg = 0; gg < per; ++gg) {
            hi += red[(4 * p + c) * kThreads + gg * vpr + cj];
            lo += red[(4 * p + 2 + c) * kThreads + gg * vpr + cj];
        }
        at.A[((int64_t)b * at.blk + i) * at.blk + t] = attn_fixed(hi, lo);
    }
}

// Every thread of the row's CTA (rank 0 of its cluster) calls it after the row
// is streamed.  Rows of late-phase sequences (fewer than bulk_frac * blk
// masked positions: no graph) and unmasked rows store nothing.
__device__ __forceinline__ void attn_row_sums(const RowAttn& at, int64_t r, const unsigned char* buf, float* red) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    const int b = (int)(r / at.blk), i = (int)(r - (int64_t)b * at.blk);
    const int t = threadIdx.x;
    const uint8_t* mk = at.mask4 ? buf + attn_buf_bytes(at) : at.masked + (int64_t)b * at.blk;
    __syncthreads();  // every thread's copies have landed
    const bool m = t < at.blk && mk[t] != 0;
    const int M = __syncthreads_count(m);
    if ((float)M < at.bulk_frac * (float)at.blk) return;
    if (!mk[i]) return;
    switch (at.dtype) {
    case DLM_F16: attn_row_sums_typed<DLM_F16>(at, b, i, buf, red); break;
    case DLM_BF16: attn_row_sums_typed<DLM_BF16>(at, b, i, buf, red); break;
    default: attn_row_sums_typed<DLM_F32>(at, b, i, buf, red); break;
    }
}


template <int DT, bool PREV, bool RULES, bool ATTN = false>
__device__ __forceinline__ void row_stats_body(const RowStatsArgs& args, const RowRules* rules) {
    constexpr int EPV = Fmt<DT>::EPV;
    constexpr int ESZ = Fmt<DT>::ESZ;
    __shared__ Part s_warp[kWarps];
    __shared__ Part s_cta;

    const int split = args.split;
    // a kernel launched after this one with programmatic serialization may
    // start as this grid's last wave drains (it does not read our results)
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t r = args.row_base + blockIdx.x / split;
    const int rank = blockIdx.x - (int)((blockIdx.x / split) * split);
    const int64_t q = args.row_index ? (int64_t)args.row_index[r] : r;
    if (q < 0 || (args.n_src > 0 && q >= args.n_src)) {
        // a row index outside the caller's rows: nothing is read or written
        // (every CTA of a cluster sees the same q, so none waits at a barrier)
        if (rank == 0 && threadIdx.x == 0) raise_status(args.dev_status, DLM_DEV_BAD_INDEX);
        if (args.wait_prior && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    extern __shared__ __align__(16) unsigned char s_attn[];  // folded attention (ATTN only)
    if constexpr (ATTN) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {  // for the DAPD selection
            args.at.hdr[0] = args.at.edge_thresh;
            args.at.hdr[1] = (long long)(uint32_t)__float_as_int(args.at.s_scale);
        }
        if (rank == 0) attn_prefetch(args.at, r, s_attn);
    }
    const char* cur_row = static_cast<const char*>(args.cur) + q * args.row_stride * ESZ;
    const char* prev_row = PREV ? static_cast<const char*>(args.prev) + q * args.row_stride * ESZ : nullptr;
    const uint4* cv = reinterpret_cast<const uint4*>(cur_row);
    const uint4* pv = reinterpret_cast<const uint4*>(prev_row);

    const int nvec = (int)(args.vocab / EPV);
    const int chunk = (nvec + split - 1) / split;
    const int v0 = rank * chunk;
    const int v1 = min(nvec, v0 + chunk);

    Acc a;
    a.mx = -INFINITY;
    a.bv = -1;
    a.bidx = 0x7fffffff;
    a.ref = -FLT_MAX;
    a.S = a.T = a.K = pack2(0.f, 0.f);
    a.refp = -FLT_MAX;
    a.Sp = pack2(0.f, 0.f);

    int v = v0 + threadIdx.x;
    for (; v + (kUnroll - 1) * kThreads < v1; v += kUnroll * kThreads) {
        uint4 c[kUnroll], p[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            c[u] = ld_stream(cv + v + u * kThreads);
            if (PREV) p[u] = ld_stream(pv + v + u * kThreads);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) process_vec<DT, PREV>(a, c[u], PREV ? p[u] : c[u], v + u * kThreads);
    }
    for (; v < v1; v += kThreads) {
        uint4 c = ld_stream(cv + v);
        uint4 p = PREV ? ld_stream(pv + v) : c;
        process_vec<DT, PREV>(a, c, p, v);
    }
    // ragged tail (vocab not a multiple of the vector width): last CTA of the row
    if (rank == split - 1) {
        const int64_t t0 = (int64_t)nvec * EPV;
        for (int64_t i = t0 + threadIdx.x; i < args.vocab; i += kThreads) {
            float z = Fmt<DT>::scalar(cur_row, i);
            float zp = PREV ? Fmt<DT>::scalar(prev_row, i) : 0.f;
            process_scalar<PREV>(a, z, zp, (int)i);
        }
    }

    Part p;
    p.mx = a.mx;
    p.idx = a.bidx;
    if (a.bv >= 0) {
        // recover the first position of the maximum inside the winning vector
        constexpr int NP = EPV / 2;
        f2 z[NP];
        Fmt<DT>::unpack(ld_stream(cv + a.bv), z);
        int k = EPV;
#pragma unroll
        for (int j = NP - 1; j >= 0; --j) {
            float x, y;
            unpack2(z[j], x, y);
            if (y == a.mx) k = 2 * j + 1;
            if (x == a.mx) k = 2 * j;
        }
        p.idx = a.bv * EPV + k;
    }
    p.ref = a.ref;
    p.S = hsum2(a.S);
    p.T = hsum2(a.T);
    p.K = hsum2(a.K);
    p.refp = a.refp;
    p.Sp = hsum2(a.Sp);

    warp_merge(p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) s_warp[warp] = p;
    __syncthreads();
    if (warp == 0) {
        if (lane < kWarps)
            p = s_warp[lane];
        else
            part_empty(p);
        warp_merge(p);
        if (lane == 0) s_cta = p;
    }
    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0 && warp == 0) {
            if (lane < split) {
                Part* rp = cluster.map_shared_rank(&s_cta, lane);
                p = *rp;
            } else {
                part_empty(p);
            }
            warp_merge(p);
        }
        cluster.sync();
    }
    if constexpr (ATTN) {
        if (rank == 0)
            attn_row_sums(args.at, args.row_base + blockIdx.x / split, s_attn,
                          reinterpret_cast<float*>(s_attn + attn_red_offset(args.at)));
    }
    // a tail launch overlapping the previous grid completes only after it, so
    // whatever follows on the stream sees both grids' results
    if (args.wait_prior && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (!RULES) {
        if (rank != 0 || threadIdx.x != 0) return;
        // where this row's results go, recomputed here so that nothing extra is
        // live across the streaming loop: q (default) or r (gathered outputs)
        const int64_t r_out = args.row_base + blockIdx.x / split;
        const int64_t out = (args.gather || !args.row_index) ? r_out : (int64_t)args.row_index[r_out];
        if (args.partial) {  // a slice of the row: its state, positions made global
            if (p.idx != 0x7fffffff) p.idx += (int)args.vocab_offset;
            static_cast<Part*>(args.partial)[out] = p;
            return;
        }
        write_outputs<PREV>(args, p, out);
    } else {
        // fused rules: rows are b*blk + i.  The row's outputs are published
        // (fence, then the count); the CTA whose row completes sequence b's
        // count reads the other rows' outputs at L2 and runs b's rules.  No
        // CTA waits for another.
        __shared__ int s_seq;
        __shared__ RuleSmem s_rules;
        if (rank != 0) return;
        if (threadIdx.x == 0) {
            const int64_t out = args.row_base + blockIdx.x / split;
            write_outputs<PREV>(args, p, out);
            __threadfence();
            const int b = (int)(out / rules->blk);
            const unsigned done = atomicAdd(rules->counter + b, 1u) + 1u;
            s_seq = done == (unsigned)rules->blk ? b : -1;
        }
        __syncthreads();
        const int b = s_seq;
        if (b < 0) return;
        __threadfence();
        if (threadIdx.x == 0) rules->counter[b] = 0u;  // zero again for the next call
        run_rules(*rules, b, s_rules);
    }
}

template <int DT, bool PREV>
__global__ void __launch_bounds__(kThreads, 4) row_stats_kernel(RowStatsArgs args) {  // 4 CTAs per SM
    row_stats_body<DT, PREV, false>(args, nullptr);
}

// The row pass with the DAPD attention sums folded in (dynamic shared memory:
// the copied attention runs, the mask flags and the partials of their sums).
// Launched only for rows split over clusters (a grid well inside one wave),
// so it takes the registers of 2 CTAs per SM rather than 4.
template <int DT, bool PREV>
__global__ void __launch_bounds__(kThreads, 2) row_stats_attn_kernel(RowStatsArgs args) {
    row_stats_body<DT, PREV, false, true>(args, nullptr);
}

// The row pass with the fused rules epilogue (few-row launches; no occupancy
// floor, the epilogue's shared memory and registers come on top of the pass's).
template <int DT, bool PREV>
__global__ void __launch_bounds__(kThreads) row_stats_rules_kernel(RowStatsArgs args, RowRules rules) {
    row_stats_body<DT, PREV, true>(args, &rules);
}

// Merge the partial states of n_shards slices of each row (slice order fixed)
// and write the row's outputs.  One thread per row.
template <bool PREV>
__global__ void __launch_bounds__(256) row_merge_kernel(RowStatsArgs args, const Part* parts, int n_shards,
                                                        int64_t shard_stride) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= args.n_rows) return;
    const int64_t q = args.row_index ? (int64_t)args.row_index[r] : r;
    if (q < 0 || (shard_stride > 0 && q >= shard_stride)) {
        raise_status(args.dev_status, DLM_DEV_BAD_INDEX);
        return;
    }
    Part p = parts[q];
    for (int sh = 1; sh < n_shards; ++sh) part_merge(p, parts[(int64_t)sh * shard_stride + q]);
    write_outputs<PREV>(args, p, q);
}

// Rows left over after whole waves run as half rows (clusters of 2 CTAs) in
// a second grid that starts, by programmatic serialization, while the first
// grid's last wave drains: the tail of the pass is made of half-length CTAs.
// Measured on 2048 rows x 152064: 200.8 -> 196.7 us (splits of 3 or 4, or a
// longer tail, were slower: the cluster merge costs more than they save).
constexpr int kTailSplit = 2;

template <int DT, bool PREV, bool RULES = false, bool ATTN = false>
int64_t tail_rows(const RowStatsArgs& a) {
    if (a.split != 1 || a.num_sms <= 0 || a.partial || a.single_grid) return 0;
    int per_sm = 0;
    cudaError_t e;
    if constexpr (RULES)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_stats_rules_kernel<DT, PREV>, kThreads, 0);
    else if constexpr (ATTN)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_stats_attn_kernel<DT, PREV>, kThreads,
                                                          row_attn_smem(a.at));
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_stats_kernel<DT, PREV>, kThreads, 0);
    if (e != cudaSuccess || per_sm <= 0) return 0;
    const int64_t slots = (int64_t)a.num_sms * per_sm;
    const int64_t nvec = a.vocab / Fmt<DT>::EPV;
    if (a.n_rows <= slots || nvec / kTailSplit < 2LL * kThreads) return 0;
    return a.n_rows % slots;
}

template <int DT, bool PREV, bool RULES = false, bool ATTN = false>
cudaError_t launch_grid(const RowStatsArgs& a, bool programmatic, cudaStream_t s, const RowRules* rules = nullptr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.n_rows * a.split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = ATTN ? row_attn_smem(a.at) : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (a.split > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = a.split;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (programmatic) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    if constexpr (RULES)
        return cudaLaunchKernelEx(&cfg, row_stats_rules_kernel<DT, PREV>, a, *rules);
    else if constexpr (ATTN)
        return cudaLaunchKernelEx(&cfg, row_stats_attn_kernel<DT, PREV>, a);
    else
        return cudaLaunchKernelEx(&cfg, row_stats_kernel<DT, PREV>, a);
}

template <int DT, bool PREV, bool RULES = false, bool ATTN = false>
cudaError_t launch_typed(const RowStatsArgs& a, cudaStream_t s, const RowRules* rules = nullptr) {
    const int64_t tail = tail_rows<DT, PREV, RULES, ATTN>(a);
    if (tail == 0) return launch_grid<DT, PREV, RULES, ATTN>(a, false, s, rules);
    RowStatsArgs head = a;
    head.n_rows = a.n_rows - tail;
    cudaError_t e = launch_grid<DT, PREV, RULES, ATTN>(head, false, s, rules);
    if (e != cudaSuccess) return e;
    RowStatsArgs rest = a;
    rest.row_base = a.n_rows - tail;
    rest.n_rows = tail;
    rest.split = kTailSplit;
    rest.wait_prior = 1;
    return launch_grid<DT, PREV, RULES, ATTN>(rest, true, s, rules);
}

template <int DT, bool PREV>
int grids_typed(const RowStatsArgs& a) {
    return tail_rows<DT, PREV>(a) > 0 ? 2 : 1;
}

}  // namespace

int row_stats_elems_per_vector(int dtype) { return dtype == DLM_F32 ? 4 : 8; }

int row_stats_grids(const RowStatsArgs& a, int dtype) {
    const bool prev = a.prev != nullptr;
    switch (dtype) {
    case DLM_BF16: return prev ? grids_typed<DLM_BF16, true>(a) : grids_typed<DLM_BF16, false>(a);
    case DLM_F16: return prev ? grids_typed<DLM_F16, true>(a) : grids_typed<DLM_F16, false>(a);
    default: return prev ? grids_typed<DLM_F32, true>(a) : grids_typed<DLM_F32, false>(a);
    }
}

cudaError_t launch_row_merge(const RowStatsArgs& a, const void* partials, int n_shards, int64_t shard_stride,
                             bool prev, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.n_rows + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    const Part* parts = static_cast<const Part*>(partials);
    return prev ? cudaLaunchKernelEx(&cfg, row_merge_kernel<true>, a, parts, n_shards, shard_stride)
                : cudaLaunchKernelEx(&cfg, row_merge_kernel<false>, a, parts, n_shards, shard_stride);
}

cudaError_t launch_row_stats(const RowStatsArgs& a, int dtype, cudaStream_t s) {
    const bool prev = a.prev != nullptr;
    switch (dtype) {
    case DLM_BF16: return prev ? launch_typed<DLM_BF16, true>(a, s) : launch_typed<DLM_BF16, false>(a, s);
    case DLM_F16: return prev ? launch_typed<DLM_F16, true>(a, s) : launch_typed<DLM_F16, false>(a, s);
    default: return prev ? launch_typed<DLM_F32, true>(a, s) : launch_typed<DLM_F32, false>(a, s);
    }
}

int row_stats_threads() { return kThreads; }

// The shared memory the folded attention needs, or 0 when a block row is not
// whole 16-byte vectors or it would not fit the default 48 KB.
size_t row_attn_smem(const RowAttn& at) {
    if (!at.attn || at.esz <= 0 || ((int64_t)at.blk * at.esz) % 16 != 0) return 0;
    const int epv = 16 / at.esz;
    RowAttn t = at;
    t.vpr = at.blk / epv;
    const size_t bytes = attn_red_offset(t) + (size_t)kThreads * 2 * epv * sizeof(float);
    return bytes <= 48 * 1024 ? bytes : 0;
}

cudaError_t launch_row_stats_attn(const RowStatsArgs& a, int dtype, cudaStream_t s) {
    if (row_attn_smem(a.at) == 0) return cudaErrorInvalidValue;
    const bool prev = a.prev != nullptr;
    switch (dtype) {
    case DLM_BF16:
        return prev ? launch_typed<DLM_BF16, true, false, true>(a, s) : launch_typed<DLM_BF16, false, false, true>(a, s);
    case DLM_F16:
        return prev ? launch_typed<DLM_F16, true, false, true>(a, s) : launch_typed<DLM_F16, false, false, true>(a, s);
    default:
        return prev ? launch_typed<DLM_F32, true, false, true>(a, s) : launch_typed<DLM_F32, false, false, true>(a, s);
    }
}

cudaError_t launch_row_stats_rules(const RowStatsArgs& a, const RowRules& r, int dtype, cudaStream_t s) {
    const bool prev = a.prev != nullptr;
    switch (dtype) {
    case DLM_BF16:
        return prev ? launch_typed<DLM_BF16, true, true>(a, s, &r) : launch_typed<DLM_BF16, false, true>(a, s, &r);
    case DLM_F16:
        return prev ? launch_typed<DLM_F16, true, true>(a, s, &r) : launch_typed<DLM_F16, false, true>(a, s, &r);
    default:
        return prev ? launch_typed<DLM_F32, true, true>(a, s, &r) : launch_typed<DLM_F32, false, true>(a, s, &r);
    }
}

}  // namespace dlm
