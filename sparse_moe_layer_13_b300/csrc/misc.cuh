// Combine, bias update and the bounded-wait self test.
#pragma once

#include "common.cuh"

namespace moe {

// y[t] = shared[t] + sum_k gate[t][k] * routed[row_of[t][k]] (+ residual[t]),
// FP32 accumulation in that order, bf16 result (《DeepSeek-V3 Technical
// Report》深度解读报告 §2.2). One CTA per token, 8 bf16 (16 bytes) per step.
__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ routed, const uint16_t* __restrict__ shared,
                                                      const int32_t* __restrict__ row_of, const float* __restrict__ gate,
                                                      const uint16_t* __restrict__ residual, int T, int K, int d,
                                                      uint16_t* __restrict__ y) {
    __shared__ int rows[16];
    __shared__ float gates[16];
    const int t = blockIdx.x;
    const int64_t nrows = static_cast<int64_t>(T) * K;
    if (threadIdx.x < K) {
        int r = __ldg(row_of + static_cast<int64_t>(t) * K + threadIdx.x);
        float g = __ldg(gate + static_cast<int64_t>(t) * K + threadIdx.x);
        if (r < 0 || r >= nrows) { set_status(MOE_ERR_DEVICE_CHECK); r = 0; g = 0.0f; }
        rows[threadIdx.x] = r;
        gates[threadIdx.x] = g;
    }
    __syncthreads();
    const int nv = d / 8;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float acc[8];
        const uint4 sh = __ldg(reinterpret_cast<const uint4*>(shared + static_cast<int64_t>(t) * d) + v);
        acc[0] = bf16_lo(sh.x); acc[1] = bf16_hi(sh.x); acc[2] = bf16_lo(sh.y); acc[3] = bf16_hi(sh.y);
        acc[4] = bf16_lo(sh.z); acc[5] = bf16_hi(sh.z); acc[6] = bf16_lo(sh.w); acc[7] = bf16_hi(sh.w);
        for (int k = 0; k < K; ++k) {
            const float g = gates[k];
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(routed + static_cast<int64_t>(rows[k]) * d) + v);
            acc[0] = fmaf(g, bf16_lo(u.x), acc[0]); acc[1] = fmaf(g, bf16_hi(u.x), acc[1]);
            acc[2] = fmaf(g, bf16_lo(u.y), acc[2]); acc[3] = fmaf(g, bf16_hi(u.y), acc[3]);
            acc[4] = fmaf(g, bf16_lo(u.z), acc[4]); acc[5] = fmaf(g, bf16_hi(u.z), acc[5]);
            acc[6] = fmaf(g, bf16_lo(u.w), acc[6]); acc[7] = fmaf(g, bf16_hi(u.w), acc[7]);
        }
        if (residual != nullptr) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(residual + static_cast<int64_t>(t) * d) + v);
            acc[0] += bf16_lo(u.x); acc[1] += bf16_hi(u.x); acc[2] += bf16_lo(u.y); acc[3] += bf16_hi(u.y);
            acc[4] += bf16_lo(u.z); acc[5] += bf16_hi(u.z); acc[6] += bf16_lo(u.w); acc[7] += bf16_hi(u.w);
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]); o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]); o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * d)[v] = o;
    }
}

// b_e <- b_e + gamma * sign(T*K - E*c_e) (《DeepSeek-V3 Technical Report》深度解读报告 §2.3).
__global__ void bias_update_kernel(int E, int T, int K, const int32_t* __restrict__ counts, float gamma,
                                   float* __restrict__ bias) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int64_t diff = static_cast<int64_t>(T) * K - static_cast<int64_t>(E) * counts[e];
    if (diff > 0) bias[e] = __fadd_rn(bias[e], gamma);
    else if (diff < 0) bias[e] = __fadd_rn(bias[e], -gamma);
}

// Waits on a barrier that nothing completes; the bounded wait must give up
// after limit_ns and record MOE_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0, nullptr, limit_ns);
    }
}

}  // namespace moe
