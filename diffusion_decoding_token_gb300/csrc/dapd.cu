// dapd.cu -- DAPD: attention -> tau-graph -> Welsh-Powell greedy independent
// set, with the late-phase confidence rule (DAPD, "整体框架", "关键设计 1-3").
//
// Two launches on the caller's stream:
//   attention    the HBM-bound part: for every masked row i of the block and
//                every column j, the sum over the given layers and heads of
//                attention[i][j] (dapd_accum_tma_kernel: bulk tensor copies
//                into a shared-memory ring; dapd_accum_kernel: 16-byte register
//                loads, for views a tensor map cannot describe).  Grid =
//                sequences x row tiles x split, the split CTAs of one tile
//                forming a thread-block cluster that divides the layer*head
//                range and merges through distributed shared memory.  The sums
//                are exact: each value x is split as hi = (x + 256) - 256 (a
//                multiple of 2^-15) and lo = x - hi (a multiple of 2^-24 for
//                f16 input, |lo| <= 2^-16), hi and lo are summed separately in
//                fp32 -- both sums stay exactly representable for f16 values in
//                [0, 256) whose total stays below 512 -- and the pair is stored
//                as a 64-bit fixed-point number in units of 2^-32.
//   decide       per sequence, the graph and the selection: one warp per
//                masked row builds I_ij = A_ij + A_ji (= 2 L H 2^32 s_ij), the
//                edge test I_ij > floor(2 L H 2^32 tau) (exact), the adjacency
//                words by ballot and the row sum D_i (= 2 L H 2^32 d~_i) in
//                shared memory (dapd_decide_kernel: one CTA, blocks of up to 64;
//                dapd_decide_cluster_kernel: a cluster of 32-row CTAs writing
//                into the leader's shared memory); then the 50% switch, and
//                either the late-phase rule or the exact ordering of
//                key_i = d~_i conf_i (128-bit sortable keys) and the greedy
//                scan over the adjacency bitmask.
// dapd_graph_kernel writes the graph's float outputs for a separate
// dlm_dapd_graph call that asks for them.
#include <cooperative_groups.h>
#include <cuda.h>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "attn_sum.cuh"
#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace dlm {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxWords = DLM_MAX_BLK / 32;
constexpr int kSliceUnroll = 8;

// The 50% switch of sequence b (every thread of the CTA calls it): fewer than
// bulk_frac * blk masked positions left -> the late-phase confidence rule.
__device__ __forceinline__ bool late_phase(const DapdArgs& a, int b) {
    const bool m = threadIdx.x < (unsigned)a.blk && a.masked[(int64_t)b * a.blk + threadIdx.x] != 0;
    const int M = __syncthreads_count(m);
    return (float)M < a.bulk_frac * (float)a.blk;
}

__device__ __forceinline__ uint4 ld_nc(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) dapd_accum_kernel(DapdArgs a) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // for a later dlm_dapd_select
        a.hdr[0] = a.edge_thresh;
        a.hdr[1] = (long long)__float_as_int(a.s_scale);
    }
    constexpr int EPV = AFmt<DT>::EPV;
    constexpr int ESZ = AFmt<DT>::ESZ;
    constexpr int NP = EPV / 2;
    // per thread: NP pairs of (H, L) -> 2*EPV floats
    __shared__ __align__(16) float s_red[kThreads * 2 * EPV];
    __shared__ int s_rows[kThreads];
    __shared__ int s_nm;

    const int split = a.split;
    const int g = blockIdx.x % split;
    const int tb = blockIdx.x / split;
    const int tiles = (a.blk + a.row_tile - 1) / a.row_tile;
    const int tile = tb % tiles;
    const int b = tb / tiles;
    if (late_phase(a, b)) return;  // the whole cluster takes the same branch

    const int r0 = tile * a.row_tile, r1 = min(a.blk, r0 + a.row_tile);
    {
        // compact the masked rows of the tile, in order (ballot prefix sums)
        __shared__ int s_wcount[kThreads / 32];
        const int r = r0 + (int)threadIdx.x;
        const bool mr = r < r1 && a.masked[(int64_t)b * a.blk + r] != 0;
        const unsigned bal = __ballot_sync(DLM_FULL_MASK, mr);
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        if (lane == 0) s_wcount[wid] = __popc(bal);
        __syncthreads();
        int off = 0;
        for (int k = 0; k < wid; ++k) off += s_wcount[k];
        if (mr) s_rows[off + __popc(bal & ((1u << lane) - 1u))] = r;
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int k = 0; k < kThreads / 32; ++k) tot += s_wcount[k];
            s_nm = tot;
        }
    }
    __syncthreads();
    const int nm = s_nm;
    const int vpr = (a.blk + EPV - 1) / EPV;  // vectors per row
    const int Q = nm * vpr;                   // slots per slice (<= kThreads by construction)
    const int LH = a.n_layers * a.n_heads;
    const int chunk = (LH + split - 1) / split;
    const int s0 = g * chunk, s1 = min(LH, s0 + chunk);
    const int G2 = Q > 0 ? max(1, kThreads / Q) : 1;  // slice groups inside the CTA
    const int t = threadIdx.x;
    const bool active = Q > 0 && t < G2 * Q;
    const int slot = active ? t % Q : 0;
    const int grp = active ? t / Q : 0;
    const int row = active ? s_rows[slot / vpr] : 0;
    const int vec = slot % vpr;
    const int col0 = vec * EPV;
    const bool full = col0 + EPV <= a.blk;

    f2 H[NP], L[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) H[p] = L[p] = pack2(0.f, 0.f);

    if (active) {
        const char* base = static_cast<const char*>(a.attn) +
                           ((int64_t)b * a.sb + (int64_t)(a.block_start + row) * a.sr + a.block_start + col0) * ESZ;
        // walk the (layer, head) slices s0+grp, s0+grp+G2, ... with running
        // element offsets instead of a division per load
        const int nh = a.n_heads;
        int s = s0 + grp;
        int h = s % nh;
        int64_t off = (int64_t)(s / nh) * a.sl + (int64_t)h * a.sh;
        const int dh = G2 % nh;
        const int64_t doff = (int64_t)(G2 / nh) * a.sl + (int64_t)dh * a.sh;
        const int64_t wrap = a.sl - (int64_t)nh * a.sh;
        auto next = [&]() {
            off += doff;
            h += dh;
            if (h >= nh) {
                h -= nh;
                off += wrap;
            }
        };
        if (full) {
            for (; s + (kSliceUnroll - 1) * G2 < s1; s += kSliceUnroll * G2) {
                uint4 w[kSliceUnroll];
#pragma unroll
                for (int u = 0; u < kSliceUnroll; ++u) {
                    w[u] = ld_nc(base + off * ESZ);
                    next();
                }
#pragma unroll
                for (int u = 0; u < kSliceUnroll; ++u) {
                    f2 x[NP];
                    AFmt<DT>::to_f2(w[u], x);
                    split_acc<NP>(x, H, L);
                }
            }
            for (; s < s1; s += G2) {
                f2 x[NP];
                AFmt<DT>::to_f2(ld_nc(base + off * ESZ), x);
                next();
                split_acc<NP>(x, H, L);
            }
        } else {
            // ragged last vector of the row: element loads of the valid columns
            for (; s < s1; s += G2) {
                const char* p = base + off * ESZ;
                next();
                float v[EPV];
#pragma unroll
                for (int k = 0; k < EPV; ++k) v[k] = (col0 + k < a.blk) ? AFmt<DT>::scalar(p + k * ESZ) : 0.f;
                f2 x[NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) x[q] = pack2(v[2 * q], v[2 * q + 1]);
                split_acc<NP>(x, H, L);
            }
        }
    }

    // merge the slice groups of this CTA in group order, then the CTAs of the
    // cluster in rank order.  Partial sums are stored component-major,
    // s_red[k * kThreads + thread], so stores and loads are bank-conflict free,
    // and each rank's values are loaded into registers before they are added.
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        float h0, h1, l0, l1;
        unpack2(H[p], h0, h1);
        unpack2(L[p], l0, l1);
        s_red[(4 * p + 0) * kThreads + t] = h0;
        s_red[(4 * p + 1) * kThreads + t] = h1;
        s_red[(4 * p + 2) * kThreads + t] = l0;
        s_red[(4 * p + 3) * kThreads + t] = l1;
    }
    __syncthreads();
    float acc[2 * EPV];
#pragma unroll
    for (int k = 0; k < 2 * EPV; ++k) acc[k] = s_red[k * kThreads + t];
    if (active && grp == 0) {
        for (int gg = 1; gg < G2; ++gg) {
            const int src = gg * Q + slot;
#pragma unroll
            for (int k = 0; k < 2 * EPV; ++k) acc[k] += s_red[k * kThreads + src];
        }
    }
    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        __syncthreads();
        if (active && grp == 0) {
#pragma unroll
            for (int k = 0; k < 2 * EPV; ++k) s_red[k * kThreads + t] = acc[k];
        }
        cluster.sync();
        if (g == 0 && active && grp == 0) {
            for (int r = 1; r < split; ++r) {
                const float* o = cluster.map_shared_rank(s_red, r);
                float v[2 * EPV];
#pragma unroll
                for (int k = 0; k < 2 * EPV; ++k) v[k] = o[k * kThreads + t];
#pragma unroll
                for (int k = 0; k < 2 * EPV; ++k) acc[k] += v[k];
            }
        }
        cluster.sync();
    }
    if (g != 0 || !active || grp != 0) return;
    long long* A = a.A + ((int64_t)b * a.blk + row) * a.blk;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int col = col0 + 2 * p + k;
            if (col < a.blk) {
                const float hi = acc[4 * p + k], lo = acc[4 * p + 2 + k];
                A[col] = attn_fixed(hi, lo);
            }
        }
    }
}

constexpr int kStages = 3;                       // bulk-copy ring depth
constexpr int kBoxBytes = 32768;                 // target bytes per bulk tensor copy
constexpr long long kWaitLimit = 2000000000LL;   // ~1 s at 2 GHz

// The same sums as dapd_accum_kernel, with the attention staged by the TMA
// engine: one thread issues bulk tensor copies of [box_heads x rows x
// box_cols] boxes (about 32 KB) into a kStages-deep shared-memory ring, so a
// CTA keeps up to 96 KB in flight without spending registers on it; every
// thread then sums its (row, 8-column vector) slots over the heads of each box.
// Rows of the tile that are not masked are loaded but never stored.
template <int DT>
__global__ void __launch_bounds__(kThreads) dapd_accum_tma_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                  DapdArgs a) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // for a later dlm_dapd_select
        a.hdr[0] = a.edge_thresh;
        a.hdr[1] = (long long)__float_as_int(a.s_scale);
    }
    constexpr int EPV = AFmt<DT>::EPV;
    constexpr int ESZ = AFmt<DT>::ESZ;
    constexpr int NP = EPV / 2;
    // the ring holds the boxes while streaming; once the stream is done the
    // same bytes hold the per-thread partial sums for the merges
    extern __shared__ __align__(128) unsigned char s_ring[];
    float* const s_red = reinterpret_cast<float*>(s_ring);
    __shared__ __align__(8) uint64_t s_full[kStages];
    __shared__ int s_timed_out;  // read by the cluster's rank 0 before it stores the sums

    const int split = a.split;
    const int g = blockIdx.x % split;
    const int tb = blockIdx.x / split;
    const int tiles = (a.blk + a.row_tile - 1) / a.row_tile;
    const int tile = tb % tiles;
    const int b = tb / tiles;
    if (late_phase(a, b)) return;  // the whole cluster takes the same branch

    const int RB = a.row_tile, CB = a.box_cols, HB = a.box_heads;
    const int r0 = tile * RB;
    const int vpr = CB / EPV;
    const int Q = RB * vpr;
    const int G2 = max(1, min(HB, kThreads / Q));
    const int t = threadIdx.x;
    const bool active = t < G2 * Q;
    const int slot = active ? t % Q : 0;
    const int grp = active ? t / Q : 0;
    const int rr = slot / vpr, cv = slot % vpr;
    const int nbox = a.n_layers * a.head_groups;
    const int chunk = (nbox + split - 1) / split;
    const int j0 = g * chunk;
    const int n = max(0, min(nbox, j0 + chunk) - j0);
    const int stage_stride = (a.box_bytes + 127) & ~127;  // 128-byte aligned ring slots

    if (t == 0) {
        for (int k = 0; k < kStages; ++k) mbar_init(&s_full[k], 1);
        mbar_init_fence();
    }
    __syncthreads();
    auto issue = [&](int j, int stage) {
        const int bj = j0 + j;
        const int l = bj / a.head_groups, hg = bj - l * a.head_groups;
        mbar_expect_tx(&s_full[stage], (uint32_t)a.box_bytes);
        tma_load_5d(s_ring + (size_t)stage * stage_stride, &tmap, &s_full[stage], a.block_start,
                    a.block_start + r0, hg * HB, l, b);
    };
    if (t == 0)
        for (int k = 0; k < min(kStages, n); ++k) issue(k, k);

    f2 H[NP], L[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) H[p] = L[p] = pack2(0.f, 0.f);
    int timed_out = 0, j_stop = n;
    for (int j = 0; j < n; ++j) {
        const int stage = j % kStages;
        const uint32_t parity = (uint32_t)((j / kStages) & 1);
        const int late = (j == 0 && a.first_wait_limit >= 0)
                             ? !mbar_wait_bounded_probe(&s_full[stage], parity, a.first_wait_limit)
                             : !mbar_wait_bounded(&s_full[stage], parity, kWaitLimit);
        if (__syncthreads_or(late)) {
            timed_out = 1;
            j_stop = j;
            break;
        }
        if (active) {
            const unsigned char* box = s_ring + (size_t)stage * stage_stride;
            for (int hh = grp; hh < HB; hh += G2) {
                const uint4 w = *reinterpret_cast<const uint4*>(box + ((size_t)(hh * RB + rr) * CB + cv * EPV) * ESZ);
                f2 x[NP];
                AFmt<DT>::to_f2(w, x);
                split_acc<NP>(x, H, L);
            }
        }
        __syncthreads();  // the stage is free again
        if (t == 0 && j + kStages < n) issue(j + kStages, stage);
    }
    if (timed_out) {
        // wait (with the full limit) for the copies already issued to land
        // before the shared memory they target is reused, then report; the
        // sums of this tile are not stored
        if (t == 0) {
            for (int j = j_stop; j < min(n, j_stop + kStages); ++j)
                mbar_wait_bounded(&s_full[j % kStages], (uint32_t)((j / kStages) & 1), kWaitLimit);
            raise_status(a.dev_status, DLM_DEV_TIMEOUT);
        }
    }
    if (t == 0) s_timed_out = timed_out;
    __syncthreads();  // every read of the ring is done before it is reused

    // partial sums, component-major: s_red[k * kThreads + thread], so stores
    // and loads are bank-conflict free; merged by group, then by cluster rank
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        float h0, h1, l0, l1;
        unpack2(H[p], h0, h1);
        unpack2(L[p], l0, l1);
        s_red[(4 * p + 0) * kThreads + t] = h0;
        s_red[(4 * p + 1) * kThreads + t] = h1;
        s_red[(4 * p + 2) * kThreads + t] = l0;
        s_red[(4 * p + 3) * kThreads + t] = l1;
    }
    __syncthreads();
    float acc[2 * EPV];
#pragma unroll
    for (int k = 0; k < 2 * EPV; ++k) acc[k] = s_red[k * kThreads + t];
    if (active && grp == 0) {
        for (int gg = 1; gg < G2; ++gg) {
            const int src = gg * Q + slot;
#pragma unroll
            for (int k = 0; k < 2 * EPV; ++k) acc[k] += s_red[k * kThreads + src];
        }
    }
    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        __syncthreads();
        if (active && grp == 0) {
#pragma unroll
            for (int k = 0; k < 2 * EPV; ++k) s_red[k * kThreads + t] = acc[k];
        }
        cluster.sync();
        if (g == 0)  // a rank that gave up waiting leaves the tile's sums incomplete: none is stored
            for (int r = 1; r < split; ++r) timed_out |= *cluster.map_shared_rank(&s_timed_out, r);
        if (g == 0 && active && grp == 0) {
            for (int r = 1; r < split; ++r) {
                const float* o = cluster.map_shared_rank(s_red, r);
                float v[2 * EPV];
#pragma unroll
                for (int k = 0; k < 2 * EPV; ++k) v[k] = o[k * kThreads + t];
#pragma unroll
                for (int k = 0; k < 2 * EPV; ++k) acc[k] += v[k];
            }
        }
        cluster.sync();
    }
    const int row = r0 + rr;
    if (g != 0 || !active || grp != 0 || timed_out || row >= a.blk) return;
    if (!a.masked[(int64_t)b * a.blk + row]) return;
    long long* A = a.A + ((int64_t)b * a.blk + row) * a.blk;
    const int col0 = cv * EPV;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int col = col0 + 2 * p + k;
            if (col < a.blk) {
                const float hi = acc[4 * p + k], lo = acc[4 * p + 2 + k];
                A[col] = attn_fixed(hi, lo);
            }
        }
    }
}

// One warp builds node i's graph row from the fixed-point sums A of sequence
// b: the symmetrised score against every masked j, the tau-edges as a
// bitmask (words of 32 neighbours, kMaxWords per row) and the proxy degree D
// (sum over masked j != i); optional float outputs.  adj_row / D_out may point
// to global or shared memory.
// Ai is row i of A (global or shared memory); with col_T, A_ji comes from a
// shared-memory copy of the block's columns from col0 on, col_ld words per row
// j: col_T[j * col_ld + (i - col0)], else from A in global memory.
constexpr int kColStride = 33;  // padded: a warp's column reads hit distinct bank pairs



struct RowLoad {
    long long Iv[kMaxWords];  // I_ij for the lane's column j of each word
    bool in[kMaxWords];       // j is masked
};

// the row's loads (one round trip), issued before any decision
__device__ __forceinline__ void graph_row_load(const DapdArgs& a, int b, int i, const long long* Ai,
                                               const long long* col_T, int col_ld, int col0, const uint8_t* mk,
                                               RowLoad& L) {
    const int lane = threadIdx.x & 31;
    const long long* A = a.A + (int64_t)b * a.blk * a.blk;
    const int nw = (a.blk + 31) >> 5;
#pragma unroll
    for (int c = 0; c < kMaxWords; ++c) {
        const int j = c * 32 + lane;
        L.in[c] = c < nw && j < a.blk && mk[j];
        const long long Aji = !L.in[c] ? 0 : (col_T ? col_T[j * col_ld + (i - col0)] : A[(int64_t)j * a.blk + i]);
        L.Iv[c] = L.in[c] ? Ai[j] + Aji : 0;
    }
}

__device__ __forceinline__ void graph_row_finish(const DapdArgs& a, int b, int i, long long thresh, float scale,
                                                 const RowLoad& L, uint32_t* adj_row, long long* D_out) {
    const int lane = threadIdx.x & 31;
    long long D = 0;
    int deg = 0;
    const int nw = (a.blk + 31) >> 5;
#pragma unroll
    for (int c = 0; c < kMaxWords; ++c) {
        if (c >= nw) break;
        const int j = c * 32 + lane;
        bool edge = false;
        if (L.in[c]) {
            const long long I = L.Iv[c];
            if (a.s_out) a.s_out[((int64_t)b * a.blk + i) * a.blk + j] = __ll2float_rn(I) * scale;
            if (j != i) {
                D += I;
                edge = I > thresh;
                deg += edge;
            }
        }
        const uint32_t w = __ballot_sync(DLM_FULL_MASK, edge);
        if (lane == 0) adj_row[c] = w;
    }
    D = warp_sum_ll(D);
    deg = warp_sum_i(deg);
    if (lane == 0) {
        *D_out = D;
        if (a.dtilde_out) a.dtilde_out[(int64_t)b * a.blk + i] = __ll2float_rn(D) * scale;
        if (a.deg_out) a.deg_out[(int64_t)b * a.blk + i] = deg;
    }
}

__device__ __forceinline__ void graph_row(const DapdArgs& a, int b, int i, long long thresh, float scale,
                                          uint32_t* adj_row, long long* D_out) {
    RowLoad L;
    graph_row_load(a, b, i, a.A + ((int64_t)b * a.blk + i) * a.blk, nullptr, 0, 0, a.masked + (int64_t)b * a.blk, L);
    graph_row_finish(a, b, i, thresh, scale, L, adj_row, D_out);
}

__global__ void __launch_bounds__(kThreads) dapd_graph_kernel(DapdArgs a) {
    const int b = blockIdx.y;
    if (late_phase(a, b)) return;
    const int warp = threadIdx.x >> 5;
    const int i = blockIdx.x * (kThreads / 32) + warp;
    if (i >= a.blk) return;
    if (!a.masked[(int64_t)b * a.blk + i]) return;
    graph_row(a, b, i, a.edge_thresh, a.s_scale, a.adj + ((int64_t)b * a.blk + i) * kMaxWords,
              a.Dsum + (int64_t)b * a.blk + i);
}

// Sortable exact key.  key = D * c (order_mode 0) or D (order_mode 1), with D
// an integer of at most 51 bits and c an fp32 confidence: the product has at
// most 75 significant bits.  It is written as sign, an 11-bit biased binary
// exponent and the 127 bits below the leading one of the normalised 128-bit
// mantissa, of which the top 115 are kept (bits below those are zero for
// every such product).  Two unsigned 64-bit words then compare exactly like
// the keys: (hi, lo) larger <=> key larger.  Zero keys sit between the
// negatives and the positives; unused slots are (0, 0).
struct SortKey {
    unsigned long long hi, lo;
};

__device__ __forceinline__ SortKey make_sort_key(long long D, float c, int order_mode) {
    int sign = D > 0 ? 1 : (D < 0 ? -1 : 0);
    const unsigned long long mag = D < 0 ? (unsigned long long)(-D) : (unsigned long long)D;
    unsigned long long mhi = 0, mlo = mag;
    int e = 0;
    if (order_mode == 0) {
        const uint32_t u = __float_as_uint(c);
        const int ce = (u >> 23) & 0xff;
        uint32_t cm = u & 0x7fffff;
        if (!(c > 0.f) || ce == 0xff) sign = 0;  // zero, negative, NaN or inf confidence: key 0
        if (ce != 0) cm |= 0x800000u;
        e = ce == 0 ? -149 : ce - 150;
        mlo = mag * (unsigned long long)cm;
        mhi = __umul64hi(mag, (unsigned long long)cm);
    }
    SortKey k;
    if (sign == 0 || (mhi == 0 && mlo == 0)) {
        k.hi = 1ULL << 63;
        k.lo = 0;
        return k;
    }
    // normalise: leading one to bit 127
    const int lz = mhi ? __clzll(mhi) : 64 + __clzll(mlo);
    if (lz >= 64) {
        mhi = mlo << (lz - 64);
        mlo = 0;
    } else if (lz > 0) {
        mhi = (mhi << lz) | (mlo >> (64 - lz));
        mlo <<= lz;
    }
    const unsigned long long ex = (unsigned long long)(e - lz + 512) & 0x7ffULL;  // biased exponent
    // fraction bits 126..76 -> 51 bits, 75..12 -> 64 bits
    const unsigned long long f1 = (mhi << 1) >> 13;
    const unsigned long long f2 = (mhi << 52) | (mlo >> 12);
    unsigned long long hi = (ex << 51) | f1, lo = f2;
    if (sign > 0) {
        hi |= 1ULL << 63;
    } else {  // mirror below zero: 2^127 - magnitude
        hi = (0x8000000000000000ULL - hi) - (lo != 0 ? 1 : 0);
        lo = ~lo + 1;
    }
    k.hi = hi;
    k.lo = lo;
    return k;
}

// a goes before b: larger key first, then the lower position
__device__ __forceinline__ bool key_before(unsigned long long ah, unsigned long long al, int ai, unsigned long long bh,
                                           unsigned long long bl, int bi) {
    if (ah != bh) return ah > bh;
    if (al != bl) return al > bl;
    return ai < bi;
}

// Greedy scan over the nodes order[0..n) of the symmetric tau-graph, with
// adjacency rows in node coordinates (bit k of word w of row v: node 32w + k
// is a neighbour of v): keep a node iff no neighbour earlier in the order is
// kept.  The nodes go 32 at a time.  intra[r] holds, for the node at order
// position r, which earlier nodes of its chunk are neighbours (bit k: the node
// at position (r & ~31) + k).  One warp runs the scan: lane l takes the node at
// position 32c + l, drops it when an earlier chunk's kept node is a neighbour
// (the union of the kept nodes' rows, word w in lane w), and the chunk is
// resolved in rounds of ballots: a node whose earlier in-chunk neighbours are
// all decided is kept if none of them was kept, dropped otherwise (the first
// undecided node is always decided, so a chunk takes at most 32 rounds and
// sparse graphs a few).  Leaves the kept set (node coordinates) in
// s_kept[0..kMaxWords).
__device__ __forceinline__ void greedy_scan_sym(const uint32_t* adj, const int* order, const uint32_t* intra_in,
                                                int n, int nw, uint32_t* s_kept) {
    const int lane = threadIdx.x & 31;
    uint32_t blocked_w = 0u, kept_w = 0u;  // lane w: word w of the kept nodes' neighbours / of the kept set
    for (int c0 = 0; c0 < n; c0 += 32) {
        const bool valid = c0 + lane < n;
        const int v = valid ? order[c0 + lane] : 0;
        const uint32_t vb = 1u << (v & 31);
        const uint32_t bw = __shfl_sync(DLM_FULL_MASK, blocked_w, v >> 5);
        const uint32_t cand = __ballot_sync(DLM_FULL_MASK, valid && (bw & vb) == 0u);
        const uint32_t intra = valid ? intra_in[c0 + lane] : 0u;
        uint32_t und = cand, kept = 0u;
        while (und) {
            const bool u = (und >> lane) & 1u;
            const uint32_t km = __ballot_sync(DLM_FULL_MASK, u && (intra & (und | kept)) == 0u);
            const uint32_t dm = __ballot_sync(DLM_FULL_MASK, u && (intra & kept) != 0u);
            kept |= km;
            und &= ~(km | dm);
        }
        const bool mine = (kept >> lane) & 1u;
        for (int w = 0; w < nw; ++w) {
            const uint32_t nb = __reduce_or_sync(DLM_FULL_MASK, mine ? adj[v * kMaxWords + w] : 0u);
            const uint32_t kb = __reduce_or_sync(DLM_FULL_MASK, (mine && (v >> 5) == w) ? vb : 0u);
            if (lane == w) {
                blocked_w |= nb;
                kept_w |= kb;
            }
        }
    }
    if (lane < kMaxWords) s_kept[lane] = kept_w;
}

// The selection of sequence b (DAPD, key designs 2-3) from its graph: proxy
// degrees D_b[i] and adjacency rows adj_b[i * kMaxWords ..] (global or shared
// memory).  Every thread of the CTA calls it.
__device__ __forceinline__ void select_core(const DapdArgs& a, int b, bool late, int M, bool m, float c,
                                            const long long* D_b, const uint32_t* adj_b) {
    __shared__ unsigned long long s_kh[DLM_MAX_BLK], s_kl[DLM_MAX_BLK];
    __shared__ int s_ix[DLM_MAX_BLK];
    __shared__ uint32_t s_intra[DLM_MAX_BLK];
    __shared__ uint32_t s_kept[kMaxWords];
    __shared__ float s_v[kThreads / 32];
    __shared__ int s_i[kThreads / 32];
    const int t = threadIdx.x;
    uint8_t* sel = a.selected + (int64_t)b * a.blk;
    if (late) {
        bool s = m && c > a.bulk_conf;
        int n = __syncthreads_count(s);
        if (n == 0 && M > 0) {
            float v = m ? c : -INFINITY;
            int idx = m ? t : 0x7fffffff;
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
                if (t == 0) s_i[0] = idx;
            }
            __syncthreads();
            s = (t == s_i[0]);
            n = 1;
        }
        if (a.preunmask_certain && m && !s && c == 1.0f) s = true;
        n = __syncthreads_count(s);
        if (t < a.blk) sel[t] = s ? 1 : 0;
        if (t == 0) a.n_selected[b] = n;
        return;
    }
    // keys of the masked nodes, one per thread; unused slots sort last
    int n2 = 1;
    while (n2 < a.blk) n2 <<= 1;
    unsigned long long kh = 0, kl = 0;
    int ix = 0x7fffffff;
    if (m) {
        const SortKey k = make_sort_key(D_b[t], c, a.order_mode);
        kh = k.hi;
        kl = k.lo;
        ix = t;
    }
    if (t < a.blk) sel[t] = 0;
    // bitonic sort into "goes before" order, slot t in thread t: exchanges with
    // a partner in the same warp go by shuffles, the others (distance >= 32)
    // through shared memory
    const bool sorter = (t & ~31) < n2;  // whole warps that hold slots
    for (int k = 2; k <= n2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long ph = 0, pl = 0;
            int pi = 0;
            if (j >= 32) {
                __syncthreads();  // the previous exchange's reads are done
                if (t < n2) {
                    s_kh[t] = kh;
                    s_kl[t] = kl;
                    s_ix[t] = ix;
                }
                __syncthreads();
                if (t < n2) {
                    ph = s_kh[t ^ j];
                    pl = s_kl[t ^ j];
                    pi = s_ix[t ^ j];
                }
            } else if (sorter) {
                ph = __shfl_xor_sync(DLM_FULL_MASK, kh, j);
                pl = __shfl_xor_sync(DLM_FULL_MASK, kl, j);
                pi = __shfl_xor_sync(DLM_FULL_MASK, ix, j);
            }
            if (t < n2) {
                // the lower slot of an ascending pair (and the upper one of a
                // descending pair) keeps the element that goes first
                const bool keep_first = ((t & j) == 0) == ((t & k) == 0);
                const bool mine_first = key_before(kh, kl, ix, ph, pl, pi);
                if (keep_first != mine_first) {
                    kh = ph;
                    kl = pl;
                    ix = pi;
                }
            }
        }
    }
    __syncthreads();
    if (t < n2) s_ix[t] = ix;
    __syncthreads();
    // greedy scan in key order over the graph (node coordinates); first, for
    // every order position at once, its earlier neighbours within its chunk of
    // 32 (read from their rows: bit v of row v_k, the graph being symmetric)
    if (t < M) {
        const int c0 = t & ~31, v = s_ix[t];
        uint32_t intra = 0u;
        for (int q = 0; q < (t & 31); ++q)
            intra |= ((adj_b[s_ix[c0 + q] * kMaxWords + (v >> 5)] >> (v & 31)) & 1u) << q;
        s_intra[t] = intra;
    }
    __syncthreads();
    const int nw = (a.blk + 31) >> 5;
    if (t < 32) greedy_scan_sym(adj_b, s_ix, s_intra, M, nw, s_kept);
    __syncthreads();
    int mine = 0;
    if (m && (((s_kept[t >> 5] >> (t & 31)) & 1u) || (a.preunmask_certain && c == 1.0f))) {
        sel[t] = 1;
        mine = 1;
    }
    const int total = __syncthreads_count(mine);
    if (t == 0) a.n_selected[b] = total;
}

// Blocks of up to kDecideMaxBlk positions: the graph (from the sums A left by
// the attention pass) and the selection in one CTA per sequence, the graph
// kept in shared memory.
constexpr int kDecideMaxBlk = 64;

__global__ void __launch_bounds__(kThreads) dapd_decide_kernel(DapdArgs a) {
    constexpr int LD = kDecideMaxBlk + 1;  // odd row length: a warp's column reads hit distinct bank pairs
    __shared__ uint32_t s_gadj[kDecideMaxBlk * kMaxWords];
    __shared__ long long s_D[kDecideMaxBlk];
    __shared__ long long s_A[kDecideMaxBlk * LD];  // the masked rows of the sums A
    __shared__ uint8_t s_mk[kDecideMaxBlk];
    const int b = blockIdx.x, t = threadIdx.x;
    // the sums A into shared memory (coalesced asynchronous copies, so the
    // transposed reads A_ji are shared-memory reads too), issued with the
    // per-position inputs and the header: one round trip for all of them.
    // Every row is copied; rows of unmasked positions (never stored by the
    // attention pass) are never read.
    {
        const long long* A = a.A + (int64_t)b * a.blk * a.blk;
        for (int q = threadIdx.x; q < a.blk * a.blk; q += kThreads) {
            const int r = q / a.blk, k = q - r * a.blk;
            cp_async8(&s_A[r * LD + k], A + q);
        }
    }
    const bool in = t < a.blk;
    const bool m = in && a.masked[(int64_t)b * a.blk + t] != 0;
    const float c = in ? a.conf[(int64_t)b * a.blk + t] : 0.f;
    // called after a separate attention pass (dlm_dapd_select), the edge
    // threshold and score scale come from the workspace header it wrote
    const long long thresh = a.thresh_from_ws ? a.hdr[0] : a.edge_thresh;
    const float scale = a.thresh_from_ws ? __int_as_float((int)a.hdr[1]) : a.s_scale;
    if (in) s_mk[t] = m;
    const int M = __syncthreads_count(m);
    const bool late = (float)M < a.bulk_frac * (float)a.blk;
    asm volatile("cp.async.wait_all;" ::: "memory");  // (late too: no copy outlives the CTA)
    if (!late) {
        __syncthreads();
        for (int i = threadIdx.x >> 5; i < a.blk; i += kThreads / 32) {
            if (!s_mk[i]) continue;  // warp-uniform
            RowLoad L;
            graph_row_load(a, b, i, s_A + i * LD, s_A, LD, 0, s_mk, L);
            graph_row_finish(a, b, i, thresh, scale, L, s_gadj + i * kMaxWords, s_D + i);
        }
        __syncthreads();
    }
    select_core(a, b, late, M, m, c, s_D, s_gadj);
}

// Blocks of up to 32 positions without the float outputs: one warp per
// sequence, lane i holding node i.  Its graph row is a 32-bit adjacency mask
// and its degree D_i in registers (the block's sums are copied into shared
// memory in the same round trip as the per-position inputs), the keys are
// ordered by a 15-stage bitonic network of shuffles, and the greedy walks the
// order with two shuffles per node; no block barrier anywhere.  Same results
// as dapd_decide_kernel.
__global__ void __launch_bounds__(32) dapd_decide_warp_kernel(DapdArgs a) {
    constexpr int LD = 33;  // odd row length: the row reads A_ij of a warp spread over the banks
    __shared__ long long s_A[32 * LD];
    const int b = blockIdx.x, t = threadIdx.x, blk = a.blk;
    {
        const long long* A = a.A + (int64_t)b * blk * blk;
        for (int q = t; q < blk * blk; q += 32) {
            const int r = q / blk, k = q - r * blk;
            cp_async8(&s_A[r * LD + k], A + q);
        }
    }
    const bool in = t < blk;
    const bool m = in && a.masked[(int64_t)b * blk + t] != 0;
    const float c = in ? a.conf[(int64_t)b * blk + t] : 0.f;
    const long long thresh = a.thresh_from_ws ? a.hdr[0] : a.edge_thresh;
    const uint32_t mm = __ballot_sync(DLM_FULL_MASK, m);
    const int M = __popc(mm);
    const bool late = (float)M < a.bulk_frac * (float)blk;
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    bool s;
    if (late) {
        s = m && c > a.bulk_conf;
        if (__ballot_sync(DLM_FULL_MASK, s) == 0u && M > 0) {
            float v = m ? c : -INFINITY;
            int idx = m ? t : 0x7fffffff;
            warp_argmax(v, idx);
            s = (t == idx);
        }
    } else {
        // graph row of node t: I_tj = A_tj + A_jt over masked j != t
        uint32_t adj = 0u;
        long long D = 0;
        if (m) {
            for (int j = 0; j < blk; ++j) {
                if (j == t || !((mm >> j) & 1u)) continue;
                const long long I = s_A[t * LD + j] + s_A[j * LD + t];
                D += I;
                if (I > thresh) adj |= 1u << j;
            }
        }
        // keys in "goes before" order, slot q in lane q; unused slots last
        unsigned long long kh = 0, kl = 0;
        int ix = 0x7fffffff;
        if (m) {
            const SortKey k = make_sort_key(D, c, a.order_mode);
            kh = k.hi;
            kl = k.lo;
            ix = t;
        }
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const unsigned long long ph = __shfl_xor_sync(DLM_FULL_MASK, kh, j);
                const unsigned long long pl = __shfl_xor_sync(DLM_FULL_MASK, kl, j);
                const int pi = __shfl_xor_sync(DLM_FULL_MASK, ix, j);
                const bool keep_first = ((t & j) == 0) == ((t & k) == 0);
                if (keep_first != key_before(kh, kl, ix, ph, pl, pi)) {
                    kh = ph;
                    kl = pl;
                    ix = pi;
                }
            }
        }
        // greedy in key order: keep a node iff no kept node is a neighbour
        uint32_t kept = 0u;
        for (int q = 0; q < M; ++q) {
            const int v = __shfl_sync(DLM_FULL_MASK, ix, q);
            const uint32_t nb = __shfl_sync(DLM_FULL_MASK, adj, v);
            if ((nb & kept) == 0u) kept |= 1u << v;
        }
        s = m && ((kept >> t) & 1u);
    }
    if (a.preunmask_certain && m && !s && c == 1.0f) s = true;
    const int n = __popc(__ballot_sync(DLM_FULL_MASK, s));
    if (in) a.selected[(int64_t)b * blk + t] = s ? 1 : 0;
    if (t == 0) a.n_selected[b] = n;
}

// Larger blocks: a cluster of ceil(blk / 32) CTAs per sequence.  CTA r
// copies the columns [32r, 32r + 32) of the sums A (every masked row: 256-byte
// runs, asynchronous 8-byte copies) into shared memory, so the transposed
// reads A_ji of its 32 rows are coalesced, builds those graph rows straight
// into the leader CTA's shared memory (distributed shared memory), and the
// leader then selects; the graph never goes through global memory.
constexpr int kClusterRows = 32;

size_t cluster_dyn_smem(int blk) { return ((size_t)blk * kColStride + (size_t)kClusterRows * blk) * sizeof(long long); }

__global__ void __launch_bounds__(kThreads) dapd_decide_cluster_kernel(DapdArgs a) {
    __shared__ uint32_t s_gadj[DLM_MAX_BLK * kMaxWords];
    __shared__ long long s_D[DLM_MAX_BLK];
    extern __shared__ long long s_dyn[];  // columns [blk][kColStride], then rows [32][blk]
    long long* const s_colT = s_dyn;
    long long* const s_rowA = s_dyn + a.blk * kColStride;
    __shared__ uint8_t s_mk[DLM_MAX_BLK];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / (int)cluster.num_blocks();
    const int col0 = rank * kClusterRows;
    const int ncol = min(kClusterRows, a.blk - col0);
    const int t = threadIdx.x;
    const bool in = t < a.blk;
    const bool m = in && a.masked[(int64_t)b * a.blk + t] != 0;
    const float c = in ? a.conf[(int64_t)b * a.blk + t] : 0.f;
    const long long thresh = a.thresh_from_ws ? a.hdr[0] : a.edge_thresh;
    const float scale = a.thresh_from_ws ? __int_as_float((int)a.hdr[1]) : a.s_scale;
    if (t < DLM_MAX_BLK) s_mk[t] = m;
    const int M = __syncthreads_count(m);
    const bool late = (float)M < a.bulk_frac * (float)a.blk;  // the same for the whole cluster
    if (!late) {
        // asynchronous copies into shared memory: lane l of warp w takes column
        // col0 + l of the masked rows w, w + 8, ...; the CTA's own masked rows
        // go whole, in 16-byte pieces (8-byte ones when a row is not 16-byte
        // aligned: odd blk)
        const long long* A = a.A + (int64_t)b * a.blk * a.blk;
        const int l = threadIdx.x & 31;
        if (l < ncol)
            for (int j = threadIdx.x >> 5; j < a.blk; j += kThreads / 32)
                if (s_mk[j]) cp_async8(&s_colT[j * kColStride + l], A + (int64_t)j * a.blk + col0 + l);
        if ((a.blk & 1) == 0) {
            const int ppr = a.blk / 2;  // 16-byte pieces per row
            for (int q = threadIdx.x; q < ncol * ppr; q += kThreads) {
                const int r = q / ppr, k = q - r * ppr;
                if (s_mk[col0 + r]) cp_async16(&s_rowA[r * a.blk + 2 * k], A + (int64_t)(col0 + r) * a.blk + 2 * k);
            }
        } else {
            for (int q = threadIdx.x; q < ncol * a.blk; q += kThreads) {
                const int r = q / a.blk, k = q - r * a.blk;
                if (s_mk[col0 + r]) cp_async8(&s_rowA[r * a.blk + k], A + (int64_t)(col0 + r) * a.blk + k);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    cluster.sync();  // the cluster runs and every column copy is in place
    if (!late) {
        uint32_t* adj0 = cluster.map_shared_rank(s_gadj, 0);
        long long* D0 = cluster.map_shared_rank(s_D, 0);
        // the warp's rows i = col0 + warp + 8r: every row's loads first, then the decisions
        constexpr int R = kClusterRows / (kThreads / 32);
        const int warp = threadIdx.x >> 5;
        RowLoad L[R];
        bool live[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = col0 + warp + r * (kThreads / 32);
            live[r] = i < col0 + ncol && s_mk[i];
            if (live[r]) graph_row_load(a, b, i, s_rowA + (i - col0) * a.blk, s_colT, kColStride, col0, s_mk, L[r]);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = col0 + warp + r * (kThreads / 32);
            if (live[r]) graph_row_finish(a, b, i, thresh, scale, L[r], adj0 + i * kMaxWords, D0 + i);
        }
        cluster.sync();  // every row is in the leader's shared memory
    }
    if (rank == 0) select_core(a, b, late, M, m, c, s_D, s_gadj);
}

template <int DT>
cudaError_t launch_accum(const DapdArgs& a, cudaStream_t s) {
    const int tiles = (a.blk + a.row_tile - 1) / a.row_tile;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.batch * tiles * a.split));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (a.split > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = a.split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, dapd_accum_kernel<DT>, a);
}

// ---- bulk-tensor path: tensor map of the attention as a 5-d tensor ------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Describe [B][L][H][rows][cols] (element strides sb, sl, sh, sr, 1) to the
// TMA engine, clipped to the block's rows and columns so reads past the block
// fill with zeros.  Returns false when the tensor cannot be described (the
// register-load kernel is used then).
bool encode_attention_map(DapdArgs& a, CUtensorMap* map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int esz = a.dtype == DLM_F32 ? 4 : 2;
    const int epv = 16 / esz;
    const int CB = (a.blk + epv - 1) / epv * epv;
    if (CB > 256 || a.row_tile > 256) return false;
    if ((reinterpret_cast<uintptr_t>(a.attn) & 15u) != 0 || ((int64_t)a.block_start * esz) % 16 != 0) return false;
    const int64_t strides[4] = {a.sr, a.sh, a.sl, a.sb};
    for (int k = 0; k < 4; ++k)
        if (strides[k] <= 0 || (strides[k] * esz) % 16 != 0 || strides[k] * esz >= (1LL << 40)) return false;
    int HB = kBoxBytes / (CB * a.row_tile * esz);
    HB = std::max(1, std::min(HB, std::min(a.n_heads, 256)));
    const cuuint64_t dims[5] = {(cuuint64_t)(a.block_start + a.blk), (cuuint64_t)(a.block_start + a.blk),
                                (cuuint64_t)a.n_heads, (cuuint64_t)a.n_layers, (cuuint64_t)a.batch};
    const cuuint64_t gstr[4] = {(cuuint64_t)(a.sr * esz), (cuuint64_t)(a.sh * esz), (cuuint64_t)(a.sl * esz),
                                (cuuint64_t)(a.sb * esz)};
    const cuuint32_t box[5] = {(cuuint32_t)CB, (cuuint32_t)a.row_tile, (cuuint32_t)HB, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType dt = a.dtype == DLM_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : a.dtype == DLM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUresult r = enc(map, dt, 5, const_cast<void*>(a.attn), dims, gstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    a.box_cols = CB;
    a.box_heads = HB;
    a.head_groups = (a.n_heads + HB - 1) / HB;
    a.box_bytes = CB * a.row_tile * HB * esz;
    return true;
}

constexpr int kMaxDev = 64;

// ring of kStages boxes, large enough to hold the per-thread partials later
size_t tma_dyn_smem(const DapdArgs& a) {
    const int epv = a.dtype == DLM_F32 ? 4 : 8;
    const size_t ring = (size_t)kStages * (size_t)((a.box_bytes + 127) & ~127);
    const size_t red = (size_t)kThreads * 2 * epv * sizeof(float);
    return ring > red ? ring : red;
}

// allow the ring's dynamic shared memory (once per device)
template <int DT>
cudaError_t tma_smem_attribute() {
    static std::mutex mu;
    static bool smem_set[kMaxDev] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    const bool cached = dev >= 0 && dev < kMaxDev;
    if (!cached || !smem_set[dev]) {  // devices past the table are set on every call
        e = cudaFuncSetAttribute(dapd_accum_tma_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kStages * kBoxBytes + 16384));
        if (e != cudaSuccess) return e;
        if (cached) smem_set[dev] = true;
    }
    return cudaSuccess;
}

// allow the column copy's dynamic shared memory (once per device)
cudaError_t cluster_smem_attribute() {
    static std::mutex mu;
    static bool smem_set[kMaxDev] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    const bool cached = dev >= 0 && dev < kMaxDev;
    if (!cached || !smem_set[dev]) {
        e = cudaFuncSetAttribute(dapd_decide_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)cluster_dyn_smem(DLM_MAX_BLK));
        if (e != cudaSuccess) return e;
        if (cached) smem_set[dev] = true;
    }
    return cudaSuccess;
}

template <int DT>
cudaError_t launch_accum_tma(const DapdArgs& a, const CUtensorMap& map, cudaStream_t s) {
    const size_t dyn = tma_dyn_smem(a);
    cudaError_t e = tma_smem_attribute<DT>();
    if (e != cudaSuccess) return e;
    const int tiles = (a.blk + a.row_tile - 1) / a.row_tile;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.batch * tiles * a.split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (a.split > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = a.split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, dapd_accum_tma_kernel<DT>, map, a);
}

// Downstream influence of every block position from the exact sums:
// infl_j = sum over masked rows i of A_ij / (L H 2^32), the attention j
// receives from the masked queries averaged over layers and heads.  One CTA
// per sequence, one thread per column; the 64-bit sum is exact (at most
// 256 rows of at most 511 * 2^32 each) and converted once.
__global__ void __launch_bounds__(kThreads) influence_kernel(DapdArgs a, float* infl) {
    const int b = blockIdx.x, j = threadIdx.x;
    __shared__ unsigned char s_mk[DLM_MAX_BLK];
    if (j < a.blk) s_mk[j] = a.masked[(int64_t)b * a.blk + j];
    __syncthreads();
    if (j >= a.blk) return;
    const long long* A = a.A + (int64_t)b * a.blk * a.blk + j;
    long long sum = 0;
    for (int i = 0; i < a.blk; ++i)
        if (s_mk[i]) sum += A[(int64_t)i * a.blk];
    const double unit = (double)a.n_layers * (double)a.n_heads * 4294967296.0;
    infl[(int64_t)b * a.blk + j] = (float)((double)sum / unit);
}

}  // namespace

size_t dapd_workspace_bytes(int batch, int blk) {
    size_t A = ((size_t)batch * blk * blk * 8 + 255) & ~(size_t)255;
    size_t Ds = ((size_t)batch * blk * 8 + 255) & ~(size_t)255;
    size_t adj = ((size_t)batch * blk * kMaxWords * 4 + 255) & ~(size_t)255;
    return A + Ds + adj + 256;  // + header: edge threshold and score scale
}

void dapd_carve(DapdArgs& a, void* ws) {
    char* p = static_cast<char*>(ws);
    a.A = reinterpret_cast<long long*>(p);
    p += ((size_t)a.batch * a.blk * a.blk * 8 + 255) & ~(size_t)255;
    a.Dsum = reinterpret_cast<long long*>(p);
    p += ((size_t)a.batch * a.blk * 8 + 255) & ~(size_t)255;
    a.adj = reinterpret_cast<uint32_t*>(p);
    p += ((size_t)a.batch * a.blk * kMaxWords * 4 + 255) & ~(size_t)255;
    a.hdr = reinterpret_cast<long long*>(p);
}

// Test hook: a first-wait limit (clock cycles) for the next attention passes
// of this process, < 0 for none.  Exported without a declaration in dlm.h.
std::atomic<long long> g_test_first_wait_limit{-1};

cudaError_t launch_dapd_graph(DapdArgs& a, int num_sms, cudaStream_t s, bool graph_kernel) {
    a.first_wait_limit = g_test_first_wait_limit.load(std::memory_order_relaxed);
    const int epv = a.dtype == DLM_F32 ? 4 : 8;
    const int vpr = (a.blk + epv - 1) / epv;
    a.row_tile = max(1, min(a.blk, kThreads / vpr));
    const int tiles = (a.blk + a.row_tile - 1) / a.row_tile;
    const int LH = a.n_layers * a.n_heads;
    const long long base = (long long)a.batch * tiles;
    CUtensorMap map;
    const bool tma = encode_attention_map(a, &map);
    const int units = tma ? a.n_layers * a.head_groups : LH;  // work items split over a cluster
    // cluster size over the layer*head range: the register-load kernel wants
    // about two CTAs per SM; the bulk-copy kernel keeps 96 KB in flight per CTA
    // and is fastest in the step with ~1.5 CTAs per SM (on the 64 x 32 block a
    // split of 2 reads cold attention 7 % faster alone but makes the step
    // 2 us slower: in the step the pass fills the row pass's draining wave,
    // where more CTAs take more of the freed slots)
    int split = tma ? (int)((3LL * num_sms + base) / (2 * base)) : (int)((2LL * num_sms + base - 1) / base);
    split = max(1, min(8, min(split, units)));
    a.split = split;
    cudaError_t e;
    switch (a.dtype) {
    case DLM_F16: e = tma ? launch_accum_tma<DLM_F16>(a, map, s) : launch_accum<DLM_F16>(a, s); break;
    case DLM_BF16: e = tma ? launch_accum_tma<DLM_BF16>(a, map, s) : launch_accum<DLM_BF16>(a, s); break;
    default: e = tma ? launch_accum_tma<DLM_F32>(a, map, s) : launch_accum<DLM_F32>(a, s); break;
    }
    if (e != cudaSuccess) return e;
    if (!graph_kernel) return cudaSuccess;  // the selection builds the graph
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)((a.blk + kThreads / 32 - 1) / (kThreads / 32)), (unsigned)a.batch);
    cfg.blockDim = dim3(kThreads);
    return cudaLaunchKernelEx(&cfg, dapd_graph_kernel, a);
}

cudaError_t launch_dapd_select(const DapdArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kThreads);
    if (a.blk <= 32 && !a.s_out && !a.dtilde_out && !a.deg_out) {
        cfg.blockDim = dim3(32);
        return cudaLaunchKernelEx(&cfg, dapd_decide_warp_kernel, a);
    }
    if (a.blk <= kDecideMaxBlk) return cudaLaunchKernelEx(&cfg, dapd_decide_kernel, a);
    const int csize = (a.blk + kClusterRows - 1) / kClusterRows;  // 3..8
    const cudaError_t e = cluster_smem_attribute();
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(a.batch * csize));
    cfg.dynamicSmemBytes = cluster_dyn_smem(a.blk);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dapd_decide_cluster_kernel, a);
}

cudaError_t launch_attention_influence(DapdArgs& a, int num_sms, float* infl, cudaStream_t s) {
    a.bulk_frac = 0.f;  // every sequence's masked rows are summed, whatever its masked fraction
    cudaError_t e = launch_dapd_graph(a, num_sms, s, false);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.gridDim = dim3((unsigned)a.batch);
    cfg.blockDim = dim3(kThreads);
    return cudaLaunchKernelEx(&cfg, influence_kernel, a, infl);
}

cudaError_t launch_dapd(DapdArgs& a, int num_sms, cudaStream_t s) {
    // attention pass, then one graph-and-selection kernel (which also writes
    // the float outputs when they are asked for)
    cudaError_t e = launch_dapd_graph(a, num_sms, s, false);
    if (e != cudaSuccess) return e;
    return launch_dapd_select(a, s);
}

}  // namespace dlm

// Test-only entry (not declared in dlm.h): the first bulk-copy wait of every
// later attention pass gives up after `cycles` clock cycles of non-blocking
// probes and takes the timeout path (the copies in flight are still waited
// for, with the normal limit); cycles < 0 restores the normal limit.
extern "C" void dlm_test_set_first_wait_limit(long long cycles) {
    dlm::g_test_first_wait_limit.store(cycles < 0 ? -1 : cycles, std::memory_order_relaxed);
}
