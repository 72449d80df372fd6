// Expert-parallel dispatch and combine with node-limited routing
// (《DeepSeek-V3 Technical Report》深度解读报告 §2.4: each token reaches at most
// M nodes; §3.2: tokens cross nodes by all-to-all). Ranks own contiguous
// ranges of E/R experts; with R dividing G, a rank holds whole expert groups,
// so a token's group limit M bounds the ranks it is sent to.
//
// A token goes to each rank that owns one of its chosen experts once, as one
// packed row (its E4M3 codes, 1x128 scales, and its choice and gate rows):
//   [codes u8 d][scales f32 d/128][topk_idx i32 K][topk_gate f32 K][pad to 16 B]
// Send rows are ordered by (destination rank, token): the permutation
// kernels with the destination key. The receiver orders the (row, slot)
// pairs that fall in its own range by (local expert, row) with the window
// key, gathers the codes and scales into grouped rows for the grouped GEMMs,
// and sums each received row's gate-weighted expert outputs into one FP32
// partial row, which goes back to the token's rank in the received order.
// The home rank adds its shared expert's output and the partials returned
// for each token, in slot order of the token's first expert on each rank.
#pragma once

#include "common.cuh"

namespace moe {
namespace ep {

// Bytes of one packed row (16-byte multiple).
__host__ __device__ inline int64_t row_bytes(int d, int K) {
    const int64_t b = static_cast<int64_t>(d) + 4 * (d / 128) + 8 * static_cast<int64_t>(K);
    return (b + 15) / 16 * 16;
}

// One warp per send row r < *total (the device-side count of send rows; the
// grid covers the capacity `cap`): copies token send_token[r]'s codes, scales,
// choice and gates.
__global__ void __launch_bounds__(256) pack_kernel(const int32_t* __restrict__ total,
                                                   const int32_t* __restrict__ send_token, int64_t cap, int T, int d,
                                                   int K, const uint8_t* __restrict__ xq, const float* __restrict__ xs,
                                                   const int32_t* __restrict__ topk_idx,
                                                   const float* __restrict__ topk_gate, uint8_t* __restrict__ out) {
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= cap || r >= __ldg(total)) return;
    const int lane = static_cast<int>(lane_id());
    int t = __ldg(send_token + r);
    if (t < 0 || t >= T) { set_status(MOE_ERR_DEVICE_CHECK); t = 0; }
    uint8_t* row = out + r * row_bytes(d, K);
    const uint4* src = reinterpret_cast<const uint4*>(xq + static_cast<int64_t>(t) * d);
    for (int c = lane; c < d / 16; c += 32) reinterpret_cast<uint4*>(row)[c] = __ldg(src + c);
    const int nk = d / 128;
    float* sc = reinterpret_cast<float*>(row + d);
    for (int c = lane; c < nk; c += 32) sc[c] = __ldg(xs + static_cast<int64_t>(t) * nk + c);
    int32_t* ri = reinterpret_cast<int32_t*>(row + d + 4 * nk);
    float* rg = reinterpret_cast<float*>(ri + K);
    if (lane < K) {
        ri[lane] = __ldg(topk_idx + static_cast<int64_t>(t) * K + lane);
        rg[lane] = __ldg(topk_gate + static_cast<int64_t>(t) * K + lane);
    }
}

// One warp per local grouped row p: codes and scales of received row sorted_row[p].
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ offsets, int n_local,
                                                     const int32_t* __restrict__ sorted_row, int64_t n_recv,
                                                     const uint8_t* __restrict__ recv, int d, int K,
                                                     uint8_t* __restrict__ xq_local, float* __restrict__ xs_local) {
    const int64_t p = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (p >= __ldg(offsets + n_local)) return;
    const int lane = static_cast<int>(lane_id());
    int64_t src = __ldg(sorted_row + p);
    if (src < 0 || src >= n_recv) { set_status(MOE_ERR_DEVICE_CHECK); src = 0; }
    const uint8_t* row = recv + src * row_bytes(d, K);
    const uint4* s = reinterpret_cast<const uint4*>(row);
    uint4* dst = reinterpret_cast<uint4*>(xq_local + p * d);
    for (int c = lane; c < d / 16; c += 32) dst[c] = s[c];
    const int nk = d / 128;
    const float* sc = reinterpret_cast<const float*>(row + d);
    for (int c = lane; c < nk; c += 32) xs_local[p * nk + c] = sc[c];
}

// One CTA per received row i: partial[i] = sum over its slots k that this
// rank served (row_of[i][k] >= 0), in slot order, of gate[i][k] * out[row_of[i][k]],
// FP32 accumulation of the bf16 expert outputs.
__global__ void __launch_bounds__(256) partial_kernel(const uint8_t* __restrict__ recv, int d, int K,
                                                      const int32_t* __restrict__ row_of, int64_t n_rows_out,
                                                      const uint16_t* __restrict__ out, float* __restrict__ partial) {
    __shared__ int rows[16];
    __shared__ float gates[16];
    const int64_t i = blockIdx.x;
    if (threadIdx.x < K) {
        const float* rg = reinterpret_cast<const float*>(recv + i * row_bytes(d, K) + d + 4 * (d / 128) + 4 * K);
        int r = __ldg(row_of + i * K + threadIdx.x);
        float g = rg[threadIdx.x];
        if (r >= n_rows_out) { set_status(MOE_ERR_DEVICE_CHECK); r = -1; }
        if (r < 0) g = 0.0f;
        rows[threadIdx.x] = r;
        gates[threadIdx.x] = g;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < d / 4; v += blockDim.x) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int k = 0; k < K; ++k) {
            if (rows[k] < 0) continue;
            const float g = gates[k];
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(out + static_cast<int64_t>(rows[k]) * d) + v);
            acc.x = fmaf(g, bf16_lo(u.x), acc.x); acc.y = fmaf(g, bf16_hi(u.x), acc.y);
            acc.z = fmaf(g, bf16_lo(u.y), acc.z); acc.w = fmaf(g, bf16_hi(u.y), acc.w);
        }
        reinterpret_cast<float4*>(partial + i * d)[v] = acc;
    }
}

// One CTA per home token t: y[t] = shared[t] + sum over the token's send rows
// (send_row_of[t][k] >= 0, slot order) of the partial returned for that row
// (+ residual[t]), FP32 accumulation, bf16 result.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ shared, const float* __restrict__ ret,
                                                      const int32_t* __restrict__ send_row_of, int64_t S,
                                                      const uint16_t* __restrict__ residual, int T, int K, int d,
                                                      uint16_t* __restrict__ y) {
    __shared__ int rows[16];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        int r = __ldg(send_row_of + static_cast<int64_t>(t) * K + threadIdx.x);
        if (r >= S) { set_status(MOE_ERR_DEVICE_CHECK); r = -1; }
        rows[threadIdx.x] = r;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < d / 4; v += blockDim.x) {
        float4 acc = __ldg(reinterpret_cast<const float4*>(shared + static_cast<int64_t>(t) * d) + v);
        for (int k = 0; k < K; ++k) {
            if (rows[k] < 0) continue;
            const float4 p = __ldg(reinterpret_cast<const float4*>(ret + static_cast<int64_t>(rows[k]) * d) + v);
            acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
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

}  // namespace ep
}  // namespace moe
