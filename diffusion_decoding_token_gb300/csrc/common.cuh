// common.cuh -- device helpers shared by the libdlm kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "dlm.h"

#define DLM_FULL_MASK 0xffffffffu

namespace dlm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the SFU (PTX ex2.approx, flush-to-zero): relative error ~2^-22.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// NaN-propagating max (PTX max.NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// ---- packed fp32x2 arithmetic (sm_100+ f32x2 forms) --------------------
struct f2 {
    uint64_t v;
};

__device__ __forceinline__ f2 pack2(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void unpack2(f2 r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r.v));
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return d;
}
__device__ __forceinline__ f2 ex2x2(f2 a) {
    float x, y;
    unpack2(a, x, y);
    return pack2(ex2(x), ex2(y));
}
__device__ __forceinline__ float hsum2(f2 a) {
    float x, y;
    unpack2(a, x, y);
    return x + y;
}

// ---- 16-bit storage -> fp32 (exact widening) ----------------------------
// bf16 pair in one 32-bit word: element 0 in the low half.
__device__ __forceinline__ f2 bf16x2_to_f2(uint32_t w) {
    return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ f2 f16x2_to_f2(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    return pack2(f.x, f.y);
}

// ---- reductions -----------------------------------------------------------
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(DLM_FULL_MASK, v, o);
    return v;
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(DLM_FULL_MASK, v, o);
    return v;
}

// (value, index) arg-max with ties to the lower index; NaN never wins.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
    bool take = (v2 > v) || (v2 == v && i2 < i) || (v != v && v2 == v2);
    if (take) {
        v = v2;
        i = i2;
    }
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float v2 = __shfl_xor_sync(DLM_FULL_MASK, v, o);
        int i2 = __shfl_xor_sync(DLM_FULL_MASK, i, o);
        argmax_merge(v, i, v2, i2);
    }
}

// Rank of slot i (key ki) among the flagged slots of shared-memory arrays in
// (key descending, slot ascending) order: the number of flagged slots j with
// key_j > ki, or key_j == ki and j < i.  n is a multiple of 4, key is 16-byte
// and flag 4-byte aligned; every thread reads the same vectors at a time
// (broadcast) and the count has no branches.
__device__ __forceinline__ int rank_desc(const float* key, const unsigned char* flag, int n, float ki, int i) {
    const float4* k4 = reinterpret_cast<const float4*>(key);
    const uchar4* f4 = reinterpret_cast<const uchar4*>(flag);
    int r = 0;
#pragma unroll 4
    for (int q = 0; q < n / 4; ++q) {
        const float4 v = k4[q];
        const uchar4 f = f4[q];
        const int j = 4 * q;
        r += (f.x != 0) & ((v.x > ki) | ((v.x == ki) & (j < i)));
        r += (f.y != 0) & ((v.y > ki) | ((v.y == ki) & (j + 1 < i)));
        r += (f.z != 0) & ((v.z > ki) | ((v.z == ki) & (j + 2 < i)));
        r += (f.w != 0) & ((v.w > ki) | ((v.w == ki) & (j + 3 < i)));
    }
    return r;
}

__device__ __forceinline__ void raise_status(uint32_t* st, uint32_t bits) {
    if (st) atomicOr(st, bits);
}

}  // namespace dlm

// ---- mbarrier / bulk tensor copy (TMA) helpers ---------------------------
namespace dlm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// asynchronous global -> shared copies (completed by cp.async.wait_all)
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of a barrier phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same bound with non-blocking tests only, so a short limit expires on
// time even while the phase is about to complete (try_wait may suspend the
// thread until it does).
__device__ __forceinline__ bool mbar_wait_bounded_probe(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}
// Wait for a barrier phase with a time limit (clock cycles); false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}
// 5-d tiled bulk tensor load into this CTA's shared memory, completing on bar.
__device__ __forceinline__ void tma_load_5d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2,
                                            int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

// Greedy scan by one warp over nodes 0..n-1 in order, the adjacency given in
// ORDER coordinates (bit k of word w of row r: node 32w+k is a neighbour of
// node r): keep a node iff it is forced or has no kept earlier neighbour.
// The nodes go 32 at a time: lane l takes node 32c+l, tests it against the
// kept nodes of earlier chunks in parallel, and the chunk's own order is then
// resolved in rounds of ballots.  Returns word c of the kept set (order
// coordinates) in lane c.
__device__ __forceinline__ uint32_t greedy_scan_chunked(const uint32_t* adj_ord, int row_words,
                                                        const unsigned char* force_keep, int n) {
    const int lane = threadIdx.x & 31;
    uint32_t kept_words = 0;  // lane c: kept set of chunk c
    const int chunks = (n + 31) >> 5;
    for (int c = 0; c < chunks; ++c) {
        const int r = c * 32 + lane;
        const bool valid = r < n;
        const uint32_t* row = adj_ord + (size_t)min(r, n - 1) * row_words;  // a real row for every lane
        bool blocked = false;
        for (int w = 0; w < c; ++w) {
            const uint32_t kw = __shfl_sync(DLM_FULL_MASK, kept_words, w);
            blocked |= valid && (row[w] & kw) != 0u;
        }
        const uint32_t intra = valid ? (row[c] & ((1u << lane) - 1u)) : 0u;  // earlier nodes of this chunk
        const bool forced = valid && force_keep != nullptr && force_keep[r];
        // candidate: valid and (forced, or not blocked by an earlier chunk)
        const uint32_t cand = __ballot_sync(DLM_FULL_MASK, valid && (forced || !blocked));
        // the chunk in rounds: a candidate is kept once it is forced or every
        // earlier in-chunk neighbour is decided and none of them is kept, and
        // dropped once one of them is kept; the first undecided candidate is
        // always decided, so this ends (in a few rounds on sparse graphs)
        uint32_t und = cand, kc = 0u;
        while (und) {
            const bool u = (und >> lane) & 1u;
            const uint32_t km = __ballot_sync(DLM_FULL_MASK, u && (forced || (intra & (und | kc)) == 0u));
            const uint32_t dm = __ballot_sync(DLM_FULL_MASK, u && !forced && (intra & kc) != 0u);
            kc |= km;
            und &= ~(km | dm);
        }
        if (lane == c) kept_words = kc;
    }
    return kept_words;
}

}  // namespace dlm
