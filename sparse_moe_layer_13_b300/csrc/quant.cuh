// Fine-grained FP8 quantisation ("DeepSeek-V3的MoE架构设计革新" §2 FP8 training,
// item 1: activations per 1x128 tile, weights per 128x128 block; E4M3 largest
// finite value 448 per "DeepSeek-V3技术解析" §6.2).
//   scale = fl32(amax / 448), code = E4M3_RNE_SATFINITE(fl32(v / scale));
//   POW2 kernels take the power-of-two scale of tile_scale<true> instead.
#pragma once

#include "common.cuh"

namespace moe {

// Eight lanes per 1x128 tile: 16 bf16 values per lane (two 16-byte loads), amax
// by shuffles inside the eight lanes, 16 E4M3 codes per lane (one 16-byte
// store); each warp step covers four tiles and a thread keeps two steps in
// flight. Grid-stride over groups of four tiles, so any grid size is valid.
// SCATTER: row r of x is token r of a routed batch; its codes and scale go
// to the K grouped rows row_of[r][0..K) and to the shared-expert row
// rows*K + r of q / scale instead of to row r (K <= 16: lane j of the eight
// loads row_of[r][j] and row_of[r][8 + j]). A grouped row outside
// [0, rows*K) is reported and not written.
template <bool SCATTER, bool POW2>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                          float* __restrict__ scale,
                                                          const int32_t* __restrict__ row_of, int K) {
    const int64_t tiles_per_row = cols / 128;
    const int64_t ntiles = rows * tiles_per_row;
    const int64_t nquads = (ntiles + 3) / 4;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const uint32_t lane = lane_id();
    const uint32_t sub = lane & 7;
    const uint32_t base = lane & 24;                       // first lane of this tile's eight
    for (int64_t p0 = warp; p0 < nquads; p0 += 2 * nwarps) {
        uint4 w[2][2];
        int64_t tile[2];
        bool live[2];
        int dst[2][2] = {{0, 0}, {0, 0}};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            tile[u] = 4 * (p0 + u * nwarps) + (lane >> 3);
            live[u] = (p0 + u * nwarps) < nquads && tile[u] < ntiles;
            w[u][0] = w[u][1] = make_uint4(0, 0, 0, 0);
            if (live[u]) {
                const int64_t r = tile[u] / tiles_per_row, c = tile[u] - r * tiles_per_row;
                const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + c * 128) + 2 * sub;
                w[u][0] = __ldg(src);
                w[u][1] = __ldg(src + 1);
                if (SCATTER) {
                    if (static_cast<int>(sub) < K) dst[u][0] = __ldg(row_of + r * K + sub);
                    if (static_cast<int>(sub) + 8 < K) dst[u][1] = __ldg(row_of + r * K + 8 + sub);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float v[16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                v[8 * h + 0] = bf16_lo(w[u][h].x); v[8 * h + 1] = bf16_hi(w[u][h].x);
                v[8 * h + 2] = bf16_lo(w[u][h].y); v[8 * h + 3] = bf16_hi(w[u][h].y);
                v[8 * h + 4] = bf16_lo(w[u][h].z); v[8 * h + 5] = bf16_hi(w[u][h].z);
                v[8 * h + 6] = bf16_lo(w[u][h].w); v[8 * h + 7] = bf16_hi(w[u][h].w);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float s = tile_scale<POW2>(amax);
            uint4 codes;
            codes.x = e4m3x4(quant_ratio(v[0], s), quant_ratio(v[1], s), quant_ratio(v[2], s), quant_ratio(v[3], s));
            codes.y = e4m3x4(quant_ratio(v[4], s), quant_ratio(v[5], s), quant_ratio(v[6], s), quant_ratio(v[7], s));
            codes.z = e4m3x4(quant_ratio(v[8], s), quant_ratio(v[9], s), quant_ratio(v[10], s), quant_ratio(v[11], s));
            codes.w = e4m3x4(quant_ratio(v[12], s), quant_ratio(v[13], s), quant_ratio(v[14], s),
                             quant_ratio(v[15], s));
            const int64_t r = tile[u] / tiles_per_row, c = tile[u] - r * tiles_per_row;
            if (!SCATTER) {
                if (!live[u]) continue;
                reinterpret_cast<uint4*>(q + r * cols + c * 128)[sub] = codes;
                if (sub == 0) scale[r * tiles_per_row + c] = s;
            } else {
                // every lane of the warp takes part in the shuffles, live or not
                const int64_t routed = rows * K;
                for (int k = 0; k <= K; ++k) {
                    const int from = __shfl_sync(0xffffffffu, k < 8 ? dst[u][0] : dst[u][1], base + (k & 7));
                    const int64_t row = k < K ? static_cast<int64_t>(from) : routed + r;
                    if (!live[u]) continue;
                    if (k < K && (row < 0 || row >= routed)) {
                        if (sub == 0) set_status(MOE_ERR_DEVICE_CHECK);
                        continue;
                    }
                    reinterpret_cast<uint4*>(q + row * cols + c * 128)[sub] = codes;
                    if (sub == 0) scale[row * tiles_per_row + c] = s;
                }
            }
        }
    }
}

// One CTA (256 threads) per 128x128 block of one matrix.
template <bool POW2>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const float* __restrict__ w, int64_t rows, int64_t cols,
                                                            uint8_t* __restrict__ q, float* __restrict__ scale) {
    const int64_t bc = cols / 128, br = rows / 128;
    const int64_t blk = blockIdx.x;                      // over batch * br * bc
    const int64_t mat = blk / (br * bc);
    const int64_t rb = (blk / bc) % br, cb = blk % bc;
    const float* src = w + mat * rows * cols + rb * 128 * cols + cb * 128;
    uint8_t* dst = q + mat * rows * cols + rb * 128 * cols + cb * 128;
    __shared__ float red[8];
    // each thread: rows (tid/32) + 8*i, 4 columns at 4*(tid%32)
    const int tr = threadIdx.x >> 5, tc = (threadIdx.x & 31) * 4;
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src + (tr + 8 * i) * cols + tc));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float s = tile_scale<POW2>(amax);
    for (int i = 0; i < 16; ++i) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src + (tr + 8 * i) * cols + tc));
        *reinterpret_cast<uint32_t*>(dst + (tr + 8 * i) * cols + tc) =
            e4m3x4(quant_ratio(v.x, s), quant_ratio(v.y, s), quant_ratio(v.z, s), quant_ratio(v.w, s));
    }
    if (threadIdx.x == 0) scale[mat * br * bc + rb * bc + cb] = s;
}

// W13 row r of matrix b, for I-block j = r / 256 and p = r % 256:
//   p in [0,64)    -> W1 row 128j + p
//   p in [64,128)  -> W3 row 128j + p - 64
//   p in [128,192) -> W1 row 128j + p - 64
//   p in [192,256) -> W3 row 128j + p - 128
// One warp per output row, 16-byte copies.
__global__ void __launch_bounds__(256) pack_w13_kernel(const uint8_t* __restrict__ q1, const uint8_t* __restrict__ q3,
                                                       int64_t batch, int64_t I, int64_t d,
                                                       uint8_t* __restrict__ q13) {
    const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (row >= batch * 2 * I) return;
    const int64_t b = row / (2 * I), r = row % (2 * I);
    const int64_t j = r / 256, p = r % 256;
    const bool up = (p >= 64 && p < 128) || p >= 192;
    const int64_t src_row = 128 * j + (p < 128 ? (p % 64) : 64 + (p % 64));
    const uint8_t* src = (up ? q3 : q1) + (b * I + src_row) * d;
    uint8_t* dst = q13 + row * d;
    for (int64_t c = lane_id() * 16; c < d; c += 32 * 16)
        *reinterpret_cast<uint4*>(dst + c) = __ldg(reinterpret_cast<const uint4*>(src + c));
}

__global__ void pack_w13_scale_kernel(const float* __restrict__ s1, const float* __restrict__ s3, int64_t batch,
                                      int64_t nbi, int64_t nbk, float* __restrict__ s13) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;   // over batch*2*nbi*nbk
    if (i >= batch * 2 * nbi * nbk) return;
    const int64_t kc = i % nbk, rb = (i / nbk) % (2 * nbi), b = i / (nbk * 2 * nbi);
    const float* src = (rb & 1) ? s3 : s1;
    s13[i] = src[(b * nbi + rb / 2) * nbk + kc];
}

}  // namespace moe
