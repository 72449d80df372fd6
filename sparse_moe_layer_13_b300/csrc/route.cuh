// Router kernels (《DeepSeek-V3 Technical Report》深度解读报告 §2.2-§2.4).
//
//  * select_token: one warp per token, given the token's logits. Lane l holds experts l, l+32,
//    ... (coalesced logit loads). s = sigmoid(z + o), s' = s + b. Lane g < G
//    scans group g's biased affinities and sums its gk largest; groups are
//    ranked by shuffles (equal scores: lower index first) and the top M kept;
//    K rounds of a warp arg-max over the kept experts pick the experts by
//    descending s' (equal values: lower index first). Gates are the raw s of
//    the chosen experts divided by their sum.
#pragma once

#include "common.cuh"

namespace moe {
namespace route {

constexpr int kMaxEPL = 32;      // experts per lane: E <= 1024
constexpr int kMaxGK = 16;
constexpr int kSelWarps = 4;     // tokens per CTA of the select kernel

// One token's selection, by one warp. z[i] holds the token's router logit of
// expert e = lane + 32 i (e < E); sp, sr are this warp's shared-memory rows
// (biased and raw affinity, E floats each). Writes the token's K expert ids
// and gates. EPL: experts per lane (>= ceil(E/32)); MAXGK: >= gk (length of
// the per-group insertion list). Both compile-time so the per-lane arrays
// stay in registers.
template <int EPL, int MAXGK>
__device__ __forceinline__ void select_token(const float (&z)[EPL], int64_t t, int E, int G, int M, int K, int gk,
                                             const float* __restrict__ offset, const float* __restrict__ bias,
                                             float* sp, float* sr, int32_t* __restrict__ topk_idx,
                                             float* __restrict__ topk_gate) {
    const int lane = static_cast<int>(lane_id());
    const int n = E / G;
    float sb[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        sb[i] = -INFINITY;
        if (e < E) {
            float zz = z[i];
            if (offset != nullptr) zz += __ldg(offset + e);
            const float s = __fdiv_rn(1.0f, 1.0f + expf(-zz));
            sb[i] = s + __ldg(bias + e);
            sp[e] = sb[i];
            sr[e] = s;
        }
    }
    __syncwarp();
    // group scores: sum of the gk largest biased affinities of each group
    float score = -INFINITY;
    if (lane < G) {
        float top[MAXGK];
#pragma unroll
        for (int j = 0; j < MAXGK; ++j) top[j] = -INFINITY;
        for (int e = lane * n; e < (lane + 1) * n; ++e) {
            float v = sp[e];
#pragma unroll
            for (int j = 0; j < MAXGK; ++j) {      // insertion into a descending list
                if (j < gk && v > top[j]) { const float tmp = top[j]; top[j] = v; v = tmp; }
            }
        }
        score = 0.0f;
#pragma unroll
        for (int j = 0; j < MAXGK; ++j) if (j < gk) score += top[j];
    }
    int rank = 0;
    for (int g2 = 0; g2 < G; ++g2) {
        const float o = __shfl_sync(0xffffffffu, score, g2);
        if (o > score || (o == score && g2 < lane)) ++rank;
    }
    const uint32_t keep = __ballot_sync(0xffffffffu, lane < G && rank < M);
    // drop experts of groups that were not kept
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((keep >> (e / n)) & 1u)) sb[i] = -INFINITY;
    }
    int my_e = 0;
    float my_s = 0.0f;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int be = 0x7fffffff, bi = -1;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (sb[i] > bv) { bv = sb[i]; be = lane + 32 * i; bi = i; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if (bi >= 0 && lane + 32 * bi == be) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) if (i == bi) sb[i] = -INFINITY;
        }
        if (lane == k) { my_e = be; my_s = sr[be]; }
    }
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, my_s, k);
    if (lane < K) {
        topk_idx[t * K + lane] = my_e;
        topk_gate[t * K + lane] = __fdiv_rn(my_s, sum);
    }
    __syncwarp();
}

// Selection over logits stored as K-split partials z[split][t][e], summed in
// split order; one warp per token.
template <int EPL, int MAXGK>
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ z, int ksplit, int T, int E, int G, int M, int K, int gk,
              const float* __restrict__ offset, const float* __restrict__ bias,
              int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate) {
    extern __shared__ float sel_smem[];          // [kSelWarps][2][E]: biased, raw
    const int w = threadIdx.x >> 5;
    const int lane = static_cast<int>(lane_id());
    float* sp = sel_smem + static_cast<size_t>(w) * 2 * E;
    float* sr = sp + E;
    const int64_t TE = static_cast<int64_t>(T) * E;
    for (int t = blockIdx.x * kSelWarps + w; t < T; t += gridDim.x * kSelWarps) {
        const float* zt = z + static_cast<int64_t>(t) * E;
        float zz[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            zz[i] = 0.0f;
            if (e < E) {
                float v = __ldg(zt + e);
                for (int sp_i = 1; sp_i < ksplit; ++sp_i)       // K-split partials, fixed order
                    v += __ldg(zt + sp_i * TE + e);
                zz[i] = v;
            }
        }
        select_token<EPL, MAXGK>(zz, t, E, G, M, K, gk, offset, bias, sp, sr, topk_idx, topk_gate);
    }
}

}  // namespace route
}  // namespace moe

namespace moe {
namespace route {

// Sequence-wise balance statistics (《DeepSeek-V3 Technical Report》深度解读报告 §2.3:
// L_Bal with a very small weight; read as L = alpha * sum_i f_i * P_i per sequence,
// f_i = E / (K L) * #{t : i chosen by t}, P_i = mean over t of s[t][i] / sum_j s[t][j]).
//
// balance_partial_kernel: one warp per 32-token chunk (chunks never straddle a
// sequence); lane l holds experts l, l+32, ... The affinities are recomputed from
// the router's stored logits (K-split partials or their sums, as the workspace
// word says) exactly as the selection computes them; the token's
// sum over experts is a fixed butterfly. Per-chunk sums of s / sum and of choice
// counts go to p_part / c_part [chunk][E].
template <int EPL>
__global__ void __launch_bounds__(128)
balance_partial_kernel(const float* __restrict__ z, const int* __restrict__ splits, int T, int E, int K,
                       const float* __restrict__ offset, const int32_t* __restrict__ topk_idx,
                       float* __restrict__ p_part, int32_t* __restrict__ c_part) {
    const int lane = static_cast<int>(lane_id());
    const int ksplit = *splits;                 // as the router stored the logits
    const int nchunk = T / 32;
    const int64_t TE = static_cast<int64_t>(T) * E;
    for (int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < nchunk; c += (gridDim.x * blockDim.x) >> 5) {
        float p[EPL];
        int cnt[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) { p[i] = 0.0f; cnt[i] = 0; }
        for (int t = c * 32; t < c * 32 + 32; ++t) {
            const float* zt = z + static_cast<int64_t>(t) * E;
            float s[EPL];
            float local = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                s[i] = 0.0f;
                if (e < E) {
                    float zz = __ldg(zt + e);
                    for (int sp_i = 1; sp_i < ksplit; ++sp_i) zz += __ldg(zt + sp_i * TE + e);
                    if (offset != nullptr) zz += __ldg(offset + e);
                    s[i] = __fdiv_rn(1.0f, 1.0f + expf(-zz));
                    local += s[i];
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
            const int mine = lane < K ? __ldg(topk_idx + static_cast<int64_t>(t) * K + lane) : -1;
#pragma unroll
            for (int i = 0; i < EPL; ++i) p[i] += __fdiv_rn(s[i], local);
            for (int k = 0; k < K; ++k) {
                const int ek = __shfl_sync(0xffffffffu, mine, k);
#pragma unroll
                for (int i = 0; i < EPL; ++i) cnt[i] += (ek == lane + 32 * i) ? 1 : 0;
            }
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                p_part[static_cast<int64_t>(c) * E + e] = p[i];
                c_part[static_cast<int64_t>(c) * E + e] = cnt[i];
            }
        }
    }
}

// One warp per sequence: chunk sums in chunk order, then f, P and the loss
// (the sum over experts in a fixed order: lanes, then a butterfly).
__global__ void __launch_bounds__(128)
balance_final_kernel(const float* __restrict__ p_part, const int32_t* __restrict__ c_part, int nseq, int seq_len,
                     int E, int K, float alpha, float* __restrict__ f_out, float* __restrict__ p_out,
                     float* __restrict__ loss_out) {
    const int lane = static_cast<int>(lane_id());
    const int q = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (q >= nseq) return;
    const int cps = seq_len / 32;                      // chunks per sequence
    const float fscale = static_cast<float>(E) / (static_cast<float>(K) * static_cast<float>(seq_len));
    float acc = 0.0f;
    for (int e = lane; e < E; e += 32) {
        float ps = 0.0f;
        int cs = 0;
        for (int c = q * cps; c < (q + 1) * cps; ++c) {
            ps += p_part[static_cast<int64_t>(c) * E + e];
            cs += c_part[static_cast<int64_t>(c) * E + e];
        }
        const float P = ps / static_cast<float>(seq_len);
        const float f = fscale * static_cast<float>(cs);
        if (f_out != nullptr) f_out[static_cast<int64_t>(q) * E + e] = f;
        if (p_out != nullptr) p_out[static_cast<int64_t>(q) * E + e] = P;
        acc += f * P;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) loss_out[q] = alpha * acc;
}

}  // namespace route
}  // namespace moe
