// Router kernels (《DeepSeek-V3 Technical Report》深度解读报告 §2.2-§2.4).
//
//  * select_kernel: one warp per token; the logits arrive as K-split FP32
//    partials z[s][t][e], summed in split order. Lane l holds experts l, l+32,
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

// EPL: experts per lane (>= ceil(E/32)); MAXGK: >= gk (length of the
// per-group insertion list). Both compile-time so the per-lane arrays stay
// in registers.
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
    const int n = E / G;
    const int64_t TE = static_cast<int64_t>(T) * E;
    for (int t = blockIdx.x * kSelWarps + w; t < T; t += gridDim.x * kSelWarps) {
        const float* zt = z + static_cast<int64_t>(t) * E;
        float sb[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            sb[i] = -INFINITY;
            if (e < E) {
                float zz = __ldg(zt + e);
                for (int sp_i = 1; sp_i < ksplit; ++sp_i)       // K-split partials, fixed order
                    zz += __ldg(zt + sp_i * TE + e);
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
            topk_idx[static_cast<int64_t>(t) * K + lane] = my_e;
            topk_gate[static_cast<int64_t>(t) * K + lane] = __fdiv_rn(my_s, sum);
        }
        __syncwarp();
    }
}

}  // namespace route
}  // namespace moe
