// Expert histogram and token permutation by expert, without atomics. The
// same kernels, with another key policy, order the rows of the
// expert-parallel dispatch (by destination rank) and receipt (by local expert).
//
// The routed (token, slot) pairs, taken in token order, are cut into blocks
// of kTokPerBlk tokens; each block is split into 8 contiguous warp segments.
//  1. hist_kernel:    per-warp histograms of each segment with
//                     __match_any_sync (the lowest lane of each run of equal
//                     experts adds the run length), summed to per-block counts.
//  2. scan_kernel:    one CTA: per-expert totals, exclusive prefix sum over
//                     experts (offsets), and each block's starting row for
//                     each expert (offsets + counts of earlier blocks).
//  3. scatter_kernel: recomputes the per-warp histograms, turns them into
//                     per-warp starting rows, then assigns rows in order:
//                     rank inside a 32-pair batch = popc(same-expert lanes
//                     below me). Writes row_of and sorted_token (whose tail
//                     T*K + t holds t, the shared expert's rows).
//  4. gather_kernel:  one warp per grouped row copies the E4M3 row and its
//                     1x128 scales (16-byte vectors); shared-expert rows
//                     T*K + t copy token t.
// Result: rows ordered by (expert ascending, token ascending), the order a
// stable sort of the pairs by expert gives.
#pragma once

#include "common.cuh"

namespace moe {
namespace perm {

constexpr int kTokPerBlk = 256;
constexpr int kWarps = 8;

__device__ __forceinline__ int load_pair_expert(const int32_t* idx, int64_t i, int64_t n, int E) {
    if (i >= n) return -1;
    int e = __ldg(idx + i);
    if (e < 0 || e >= E) { set_status(MOE_ERR_DEVICE_CHECK); return -1; }
    return e;
}

// Key policies: the group (key) of routed pair i = (row i / K, slot i % K), or
// -1 for a pair that goes nowhere.
//   KeyExpert  the pair's expert (the layer's own permutation); an expert id
//              outside [0, E) is reported (MOE_ERR_DEVICE_CHECK) and skipped
//   KeyWindow  expert-parallel receiver: the expert minus `lo` for experts in
//              [lo, lo + n) (this rank's), -1 for other valid experts; the
//              choice rows are `stride` ints apart
//   KeyDest    expert-parallel sender: the rank owning the expert (per_rank
//              contiguous experts each), -1 when an earlier slot of the same
//              token already goes to that rank (a token is sent once per rank)
struct KeyExpert {
    const int32_t* idx;
    int E;
    __device__ __forceinline__ int operator()(int64_t i, int64_t n, int) const { return load_pair_expert(idx, i, n, E); }
};

struct KeyWindow {
    const int32_t* idx;
    int64_t stride;
    int E, lo, n;
    __device__ __forceinline__ int operator()(int64_t i, int64_t np, int K) const {
        if (i >= np) return -1;
        int e = __ldg(idx + (i / K) * stride + i % K);
        if (e < 0 || e >= E) { set_status(MOE_ERR_DEVICE_CHECK); return -1; }
        e -= lo;
        return (e >= 0 && e < n) ? e : -1;
    }
};

struct KeyDest {
    const int32_t* idx;
    int E, per_rank;
    __device__ __forceinline__ int operator()(int64_t i, int64_t np, int K) const {
        if (i >= np) return -1;
        const int64_t t = i / K;
        const int k = static_cast<int>(i - t * K);
        const int e = __ldg(idx + i);
        if (e < 0 || e >= E) { set_status(MOE_ERR_DEVICE_CHECK); return -1; }
        const int r = e / per_rank;
        for (int j = 0; j < k; ++j) {
            const int ej = __ldg(idx + t * K + j);
            if (ej >= 0 && ej < E && ej / per_rank == r) return -1;
        }
        return r;
    }
};

// hist[w][e] for warp w's segment of block `blk`.
template <class Key>
__device__ __forceinline__ void warp_histograms(const Key& key, int64_t npairs, int K, int E,
                                                int* hist, int64_t& seg_begin, int64_t& seg_end) {
    const int w = threadIdx.x >> 5;
    const int64_t blk_begin = static_cast<int64_t>(blockIdx.x) * kTokPerBlk * K;
    const int64_t blk_end = min(blk_begin + static_cast<int64_t>(kTokPerBlk) * K, npairs);
    const int64_t seg = (blk_end - blk_begin + kWarps - 1) / kWarps;
    seg_begin = min(blk_begin + w * seg, blk_end);
    seg_end = min(seg_begin + seg, blk_end);
    int* h = hist + w * E;
    for (int64_t b = seg_begin; b < seg_end; b += 32) {
        const int e = key(b + lane_id(), seg_end, K);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (__ffs(same) - 1) == static_cast<int>(lane_id())) h[e] += __popc(same);
        __syncwarp();
    }
}

template <class Key>
__global__ void __launch_bounds__(kWarps * 32) hist_kernel(Key key, int64_t npairs, int K, int E,
                                                           int32_t* __restrict__ blk_counts) {
    extern __shared__ int hist[];   // [kWarps][E]
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    int64_t sb, se;
    warp_histograms(key, npairs, K, E, hist, sb, se);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c += hist[w * E + e];
        blk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = c;
    }
}

// Single CTA of 1024 threads. blk_base[b][e] = offsets[e] + sum_{b' < b} blk_counts[b'][e].
// shared_tail: offsets[E] = T*K and offsets[E+1] = T*K + T (the layer's shared-expert
// rows follow the routed ones); otherwise offsets[E] = the total of every key.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ blk_counts, int nblk, int E, int T,
                                                    int K, int32_t* __restrict__ blk_base,
                                                    int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
                                                    bool shared_tail = true) {
    __shared__ int warp_sums[32];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int b = 0; b < nblk; ++b) {
            const int c = blk_counts[static_cast<int64_t>(b) * E + e];
            blk_base[static_cast<int64_t>(b) * E + e] = run;
            run += c;
        }
    }
    // exclusive scan of the totals over experts
    const int lane = static_cast<int>(lane_id()), w = e >> 5;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = warp_sums[lane];
        int vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, vi, o);
            if (lane >= o) vi += t;
        }
        warp_sums[lane] = vi - v;
    }
    __syncthreads();
    const int off = warp_sums[w] + incl - run;
    if (e < E) {
        offsets[e] = off;
        if (counts != nullptr) counts[e] = run;
        for (int b = 0; b < nblk; ++b) blk_base[static_cast<int64_t>(b) * E + e] += off;
    }
    if (shared_tail && e == 0) {
        offsets[E] = T * K;
        offsets[E + 1] = T * K + T;
    }
    if (!shared_tail && e == E - 1) offsets[E] = off + run;
}

// shared_tail: also write the shared-expert rows' tokens (sorted_token[T*K + t] = t);
// otherwise pairs that go nowhere (key -1) get row_of = -1.
template <class Key>
__global__ void __launch_bounds__(kWarps * 32) scatter_kernel(Key key, int64_t npairs, int K, int E,
                                                              const int32_t* __restrict__ blk_base,
                                                              int32_t* __restrict__ row_of,
                                                              int32_t* __restrict__ sorted_token,
                                                              bool shared_tail = true) {
    extern __shared__ int hist[];   // [kWarps][E]
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    int64_t sb, se;
    warp_histograms(key, npairs, K, E, hist, sb, se);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = blk_base[static_cast<int64_t>(blockIdx.x) * E + e];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    // shared-expert rows T*K + t read token t
    if (shared_tail) {
        const int64_t T = npairs / K;
        const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokPerBlk;
        for (int64_t t = t0 + threadIdx.x; t < min(t0 + kTokPerBlk, T); t += blockDim.x)
            sorted_token[npairs + t] = static_cast<int32_t>(t);
    }
    int* h = hist + (threadIdx.x >> 5) * E;
    const uint32_t lane = lane_id();
    for (int64_t b = sb; b < se; b += 32) {
        const int64_t i = b + lane;
        const int e = key(i, se, K);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        const int row = (e >= 0) ? h[e] + rank : 0;
        __syncwarp();
        if (e >= 0 && (__ffs(same) - 1) == static_cast<int>(lane)) h[e] += __popc(same);
        __syncwarp();
        if (e >= 0) {
            row_of[i] = row;
            sorted_token[row] = static_cast<int32_t>(i / K);
        } else if (!shared_tail && i < se) {
            row_of[i] = -1;
        }
    }
}

// One warp per grouped row r in [0, T*K + T).
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ sorted_token, int T, int K, int d,
                                                     const uint8_t* __restrict__ xq, const float* __restrict__ xs,
                                                     uint8_t* __restrict__ xq_perm, float* __restrict__ xs_perm) {
    const int64_t rows = static_cast<int64_t>(T) * K + T;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    int src = __ldg(sorted_token + r);
    if (src < 0 || src >= T) { set_status(MOE_ERR_DEVICE_CHECK); src = 0; }
    const uint4* s = reinterpret_cast<const uint4*>(xq + static_cast<int64_t>(src) * d);
    uint4* dst = reinterpret_cast<uint4*>(xq_perm + r * d);
    for (int c = lane_id(); c < d / 16; c += 32) dst[c] = __ldg(s + c);
    const int nk = d / 128;
    for (int c = lane_id(); c < nk; c += 32) xs_perm[r * nk + c] = __ldg(xs + static_cast<int64_t>(src) * nk + c);
}

}  // namespace perm
}  // namespace moe
