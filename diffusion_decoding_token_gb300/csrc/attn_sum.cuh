// attn_sum.cuh -- the exact attention sums of DAPD (DAPD, "关键设计 1"):
// a_ij summed over layers and heads.  Each value x in [0, 256) is split as
// hi = (x + 256) - 256 (a multiple of 2^-15) and lo = x - hi (a multiple of
// 2^-24 for f16 input, |lo| <= 2^-16); hi and lo are summed separately in
// fp32.  Both sums stay exactly representable (for totals below 512), so any
// order of additions gives the same result, stored as a 64-bit fixed-point
// number in units of 2^-32.  Shared by the attention pass (dapd.cu) and the
// row pass that folds the sums in (row_stats.cu).
#pragma once

#include "common.cuh"

namespace dlm {
namespace {

template <int DT>
struct AFmt;
template <>
struct AFmt<DLM_F16> {
    static constexpr int EPV = 8;
    static constexpr int ESZ = 2;
    static __device__ __forceinline__ void to_f2(uint4 w, f2 (&x)[4]) {
        x[0] = f16x2_to_f2(w.x);
        x[1] = f16x2_to_f2(w.y);
        x[2] = f16x2_to_f2(w.z);
        x[3] = f16x2_to_f2(w.w);
    }
    static __device__ __forceinline__ float scalar(const void* p) { return __half2float(*static_cast<const __half*>(p)); }
};
template <>
struct AFmt<DLM_BF16> {
    static constexpr int EPV = 8;
    static constexpr int ESZ = 2;
    static __device__ __forceinline__ void to_f2(uint4 w, f2 (&x)[4]) {
        x[0] = bf16x2_to_f2(w.x);
        x[1] = bf16x2_to_f2(w.y);
        x[2] = bf16x2_to_f2(w.z);
        x[3] = bf16x2_to_f2(w.w);
    }
    static __device__ __forceinline__ float scalar(const void* p) {
        return __uint_as_float((uint32_t) * static_cast<const uint16_t*>(p) << 16);
    }
};
template <>
struct AFmt<DLM_F32> {
    static constexpr int EPV = 4;
    static constexpr int ESZ = 4;
    static __device__ __forceinline__ void to_f2(uint4 w, f2 (&x)[2]) {
        x[0] = pack2(__uint_as_float(w.x), __uint_as_float(w.y));
        x[1] = pack2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
    static __device__ __forceinline__ float scalar(const void* p) { return *static_cast<const float*>(p); }
};

// exact split accumulate: x = hi + lo, hi multiple of 2^-15 when 0 <= x < 256
template <int NP>
__device__ __forceinline__ void split_acc(const f2 (&x)[NP], f2 (&H)[NP], f2 (&L)[NP]) {
    const f2 c = pack2(256.f, 256.f);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        f2 hi = sub2(add2(x[p], c), c);
        f2 lo = sub2(x[p], hi);
        H[p] = add2(H[p], hi);
        L[p] = add2(L[p], lo);
    }
}

// the fixed-point value (units of 2^-32) of a pair of exact hi / lo sums
__device__ __forceinline__ long long attn_fixed(float hi, float lo) {
    return __float2ll_rn(hi * 32768.f) * 131072LL + __float2ll_rn(lo * 4294967296.f);
}

}  // namespace
}  // namespace dlm
