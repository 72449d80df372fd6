// Combine, bias update and the bounded-wait self test.
#pragma once

#include "common.cuh"

namespace moe {

// y[t] = shared[t] + sum_k gate[t][k] * routed[row_of[t][k]] (+ residual[t]),
// FP32 accumulation in that order, bf16 result (《DeepSeek-V3 Technical
// Report》深度解读报告 §2.2). Routed outputs bf16, shared output FP32. One CTA
// per token, 4 columns (8 bytes bf16 / 16 bytes FP32) per step.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ routed, const float* __restrict__ shared,
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
    const int nv = d / 4;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float4 acc = __ldg(reinterpret_cast<const float4*>(shared + static_cast<int64_t>(t) * d) + v);
        for (int k = 0; k < K; ++k) {
            const float g = gates[k];
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(routed + static_cast<int64_t>(rows[k]) * d) + v);
            acc.x = fmaf(g, bf16_lo(u.x), acc.x); acc.y = fmaf(g, bf16_hi(u.x), acc.y);
            acc.z = fmaf(g, bf16_lo(u.y), acc.z); acc.w = fmaf(g, bf16_hi(u.y), acc.w);
        }
        if (residual != nullptr) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(residual + static_cast<int64_t>(t) * d) + v);
            acc.x += bf16_lo(u.x); acc.y += bf16_hi(u.x); acc.z += bf16_lo(u.y); acc.w += bf16_hi(u.y);
        }
        uint2 o;
        o.x = pack_bf16x2(acc.x, acc.y);
        o.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2*>(y + static_cast<int64_t>(t) * d)[v] = o;
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
