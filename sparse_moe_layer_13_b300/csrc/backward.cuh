// Backward pass of the layer: the bandwidth-bound kernels around the FP8
// GEMMs. The pages give the forward and an FP8 training recipe ("DeepSeek-V3
// 的MoE架构设计革新" §2 FP8 training: activations per 1x128 tile, weights per
// 128x128 block) and say the balancing bias leaves the gradient untouched
// (《DeepSeek-V3 Technical Report》深度解读报告 §2.3). The chosen experts are
// held fixed; gradients flow through the gates, the sigmoid affinities and
// the SwiGLU experts.
//
//   combine_backward_kernel   dg = dy . out_k, dO_k = g_k dy -> 1x128 E4M3
//   route_backward_kernel     dz_k = ds_k s_k (1 - s_k), ds = (dg - g.dg) / S
//   router_wgrad_kernel       dWr[e] = sum over e's rows of dz * x
//   swiglu_backward_kernel    dA, dB of h = SiLU(a) b; 1x128 E4M3 of [dA | dB]
//   dx_combine_kernel         dx = dx_shared + sum_k (dx_k + dz_k Wr[e_k])
//   quant_128x1_kernel        transposed 128-token x 1-channel E4M3 tiles per group
//   transpose_blocks_kernel   128x128-block E4M3 weights, transposed with their scales
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace bwd {

// Two E4M3 codes (low byte first) -> exact FP32 values.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
    uint32_t h2;
    asm("{\n.reg .b16 c;\nmov.b16 c, %1;\ncvt.rn.f16x2.e4m3x2 %0, c;\n}\n" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
    return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One CTA (8 warps) per token t. Row K of the token's K+1 rows is the shared
// expert's row T*K + t (gradient dy itself, gate 1). Warp w takes the 1x128
// tiles w, w+8, ...; lane l holds 4 columns. rgate[r] receives the gate of
// grouped row r (1 for shared rows). dgate sums the per-warp partial dot
// products in warp order.
// The expert-output gradient of routed row k is g_k * dy[t]. Since g_k > 0
// scales a tile uniformly, its 1x128 quantisation under the FP32 rule has
// the codes of dy's own tile and the scale g_k * s_dy: the tile is quantised
// once and every row gets scale fl32(g_k * s_dy). (Quantising fl32(g_k * dy)
// again would put the ratios 448 * y / y_max, often exact E4M3 midpoints for
// bf16 dy, at the mercy of the gate's last bit.) A power-of-two scale cannot
// absorb g_k, so POW2 quantises fl32(g_k * dy) row by row.
template <bool POW2>
__global__ void __launch_bounds__(256)
combine_backward_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ routed,
                        const int32_t* __restrict__ row_of, const float* __restrict__ gate, int T, int K, int d,
                        uint8_t* __restrict__ dOq, float* __restrict__ dOs, float* __restrict__ rgate,
                        float* __restrict__ dgate) {
    __shared__ int64_t rows[17];
    __shared__ float gates[17];
    __shared__ float red[8][16];
    const int t = blockIdx.x;
    const int64_t TK = static_cast<int64_t>(T) * K;
    if (threadIdx.x < K) {
        int64_t r = __ldg(row_of + static_cast<int64_t>(t) * K + threadIdx.x);
        float g = __ldg(gate + static_cast<int64_t>(t) * K + threadIdx.x);
        if (r < 0 || r >= TK) { set_status(MOE_ERR_DEVICE_CHECK); r = -1; }
        else rgate[r] = g;
        rows[threadIdx.x] = r;
        gates[threadIdx.x] = g;
    } else if (threadIdx.x == K) {
        rows[K] = TK + t;
        gates[K] = 1.0f;
        rgate[TK + t] = 1.0f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const int lane = static_cast<int>(lane_id());
    const int ntile = d / 128;
    const uint16_t* dyt = dy + static_cast<int64_t>(t) * d;
    float part[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) part[k] = 0.0f;
    for (int tile = warp; tile < ntile; tile += 8) {
        const int64_t col = static_cast<int64_t>(tile) * 128 + lane * 4;
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(dyt + col));
        const float y0 = bf16_lo(u.x), y1 = bf16_hi(u.x), y2 = bf16_lo(u.y), y3 = bf16_hi(u.y);
        // dg partial sums (K <= 16, unrolled so part[] stays in registers)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k < K && rows[k] >= 0) {
                const uint2 o = __ldg(reinterpret_cast<const uint2*>(routed + rows[k] * d + col));
                part[k] = fmaf(y0, bf16_lo(o.x), part[k]);
                part[k] = fmaf(y1, bf16_hi(o.x), part[k]);
                part[k] = fmaf(y2, bf16_lo(o.y), part[k]);
                part[k] = fmaf(y3, bf16_hi(o.y), part[k]);
            }
        }
        if (!POW2) {
            const float amax = warp_max(fmaxf(fmaxf(fabsf(y0), fabsf(y1)), fmaxf(fabsf(y2), fabsf(y3))));
            const float s = tile_scale<false>(amax);
            const uint32_t codes =
                e4m3x4(quant_ratio(y0, s), quant_ratio(y1, s), quant_ratio(y2, s), quant_ratio(y3, s));
            for (int k = 0; k <= K; ++k) {
                const int64_t r = rows[k];
                if (r < 0) continue;
                *reinterpret_cast<uint32_t*>(dOq + r * d + col) = codes;
                if (lane == 0) dOs[r * ntile + tile] = k < K ? __fmul_rn(gates[k], s) : s;
            }
        } else {
            for (int k = 0; k <= K; ++k) {
                const int64_t r = rows[k];
                const float g = gates[k];
                float v0 = y0, v1 = y1, v2 = y2, v3 = y3;
                if (k < K) { v0 = __fmul_rn(g, y0); v1 = __fmul_rn(g, y1); v2 = __fmul_rn(g, y2); v3 = __fmul_rn(g, y3); }
                const float amax = warp_max(fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
                const float s = tile_scale<true>(amax);
                if (r < 0) continue;
                *reinterpret_cast<uint32_t*>(dOq + r * d + col) =
                    e4m3x4(quant_ratio(v0, s), quant_ratio(v1, s), quant_ratio(v2, s), quant_ratio(v3, s));
                if (lane == 0) dOs[r * ntile + tile] = s;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if (k < K) {
            const float p = warp_sum(part[k]);
            if (lane == 0) red[warp][k] = p;
        }
    }
    __syncthreads();
    if (threadIdx.x < K) {
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) acc += red[w][threadIdx.x];
        dgate[static_cast<int64_t>(t) * K + threadIdx.x] = acc;
    }
}

// One warp per token; lane k < K holds chosen expert k. The affinity is
// recomputed from the router's stored logits (K-split partials or their sums,
// as the workspace word `splits` says) with the selection's own arithmetic,
// so s and S are the values the gates were made from.
__global__ void __launch_bounds__(128)
route_backward_kernel(const float* __restrict__ z, const int* __restrict__ splits, int T, int E, int K,
                      const float* __restrict__ offset, const int32_t* __restrict__ topk_idx,
                      const float* __restrict__ dgate, float* __restrict__ dz) {
    const int lane = static_cast<int>(lane_id());
    const int ksplit = *splits;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int64_t TE = static_cast<int64_t>(T) * E;
    float s = 0.0f, dg = 0.0f;
    if (lane < K) {
        int e = __ldg(topk_idx + static_cast<int64_t>(t) * K + lane);
        if (e < 0 || e >= E) { set_status(MOE_ERR_DEVICE_CHECK); e = 0; }
        const float* zt = z + static_cast<int64_t>(t) * E;
        float zz = __ldg(zt + e);
        for (int sp = 1; sp < ksplit; ++sp) zz += __ldg(zt + sp * TE + e);
        if (offset != nullptr) zz += __ldg(offset + e);
        s = __fdiv_rn(1.0f, 1.0f + expf(-zz));
        dg = __ldg(dgate + static_cast<int64_t>(t) * K + lane);
    }
    float S = 0.0f;
    for (int k = 0; k < K; ++k) S += __shfl_sync(0xffffffffu, s, k);
    const float g = __fdiv_rn(s, S);
    float gdg = 0.0f;
    for (int k = 0; k < K; ++k) gdg += __shfl_sync(0xffffffffu, g * dg, k);
    if (lane < K) {
        const float ds = __fdiv_rn(dg - gdg, S);
        dz[static_cast<int64_t>(t) * K + lane] = ds * s * (1.0f - s);
    }
}

// dWr[e][c] = sum over expert e's grouped rows r (token t_r, slot k_r) of
// dz[t_r][k_r] * x[t_r][c], in row order. Grid (E, d / 512); thread: two columns.
__global__ void __launch_bounds__(256)
router_wgrad_kernel(const uint16_t* __restrict__ x, int T, int K, int d, const int32_t* __restrict__ offsets,
                    const int32_t* __restrict__ sorted_token, const int32_t* __restrict__ row_of,
                    const float* __restrict__ dz, float* __restrict__ dWr) {
    __shared__ int tok[32];
    __shared__ float wgt[32];
    const int e = blockIdx.x;
    const int c = blockIdx.y * 512 + threadIdx.x * 2;
    const int64_t TK = static_cast<int64_t>(T) * K;
    const int r0 = __ldg(offsets + e), r1 = __ldg(offsets + e + 1);
    float a0 = 0.0f, a1 = 0.0f;
    for (int rb = r0; rb < r1; rb += 32) {
        __syncthreads();
        if (threadIdx.x < 32) {
            const int r = rb + static_cast<int>(threadIdx.x);
            int tt = 0;
            float w = 0.0f;
            if (r < r1) {
                tt = (r >= 0 && r < TK) ? __ldg(sorted_token + r) : -1;
                if (tt < 0 || tt >= T) { set_status(MOE_ERR_DEVICE_CHECK); tt = 0; }
                else {
                    int kk = -1;
                    for (int k = 0; k < K; ++k)
                        if (__ldg(row_of + static_cast<int64_t>(tt) * K + k) == r) kk = k;
                    if (kk < 0) set_status(MOE_ERR_DEVICE_CHECK);
                    else w = __ldg(dz + static_cast<int64_t>(tt) * K + kk);
                }
            }
            tok[threadIdx.x] = tt;
            wgt[threadIdx.x] = w;
        }
        __syncthreads();
        const int n = min(32, r1 - rb);
        if (c < d) {
#pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(x + static_cast<int64_t>(tok[j]) * d + c));
                a0 = fmaf(wgt[j], bf16_lo(u), a0);
                a1 = fmaf(wgt[j], bf16_hi(u), a1);
            }
        }
    }
    if (c < d) *reinterpret_cast<float2*>(dWr + static_cast<int64_t>(e) * d + c) = make_float2(a0, a1);
}

// One warp per (grouped row, 128 columns of I). Pre-activations a (gate) and
// b (up) come in the SwiGLU tile layout of the gate/up GEMM: for I-block j the
// 256 columns 256j.. hold gate[128j..+64), up[128j..+64), gate[128j+64..+128),
// up[128j+64..+128). dA and dB overwrite a and b in place (same layout); their
// 1x128 E4M3 codes go to dab_q [rows][2I] as [dA | dB] (the K order of the
// transposed-W1|W3 data-gradient GEMM), scales to dab_s [rows][2I/128].
template <bool POW2>
__global__ void __launch_bounds__(256)
swiglu_backward_kernel(float* __restrict__ ab, const float* __restrict__ dh, int64_t ld_dh, int64_t rows, int I,
                       uint8_t* __restrict__ dab_q, float* __restrict__ dab_s) {
    const int lane = static_cast<int>(lane_id());
    const int nj = I / 128;
    const int64_t warps = static_cast<int64_t>(rows) * nj;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < warps; w += nw) {
        const int64_t r = w / nj;
        const int j = static_cast<int>(w - r * nj);
        const int i0 = 128 * j + 4 * lane;
        const int64_t gcol = 256 * j + 128 * (lane >> 4) + 4 * (lane & 15);
        float* abr = ab + r * 2 * I;
        const float4 a = *reinterpret_cast<const float4*>(abr + gcol);
        const float4 b = *reinterpret_cast<const float4*>(abr + gcol + 64);
        const float4 g = __ldg(reinterpret_cast<const float4*>(dh + r * ld_dh + i0));
        float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w}, gv[4] = {g.x, g.y, g.z, g.w};
        float dA[4], dB[4];
        float amA = 0.0f, amB = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sig = __fdiv_rn(1.0f, 1.0f + expf(-av[i]));
            const float silu = av[i] * sig;
            dA[i] = gv[i] * bv[i] * sig * (1.0f + av[i] * (1.0f - sig));
            dB[i] = gv[i] * silu;
            amA = fmaxf(amA, fabsf(dA[i]));
            amB = fmaxf(amB, fabsf(dB[i]));
        }
        *reinterpret_cast<float4*>(abr + gcol) = make_float4(dA[0], dA[1], dA[2], dA[3]);
        *reinterpret_cast<float4*>(abr + gcol + 64) = make_float4(dB[0], dB[1], dB[2], dB[3]);
        const float sA = tile_scale<POW2>(warp_max(amA));
        const float sB = tile_scale<POW2>(warp_max(amB));
        uint8_t* q = dab_q + r * 2 * I;
        *reinterpret_cast<uint32_t*>(q + i0) =
            e4m3x4(quant_ratio(dA[0], sA), quant_ratio(dA[1], sA), quant_ratio(dA[2], sA), quant_ratio(dA[3], sA));
        *reinterpret_cast<uint32_t*>(q + I + i0) =
            e4m3x4(quant_ratio(dB[0], sB), quant_ratio(dB[1], sB), quant_ratio(dB[2], sB), quant_ratio(dB[3], sB));
        if (lane == 0) {
            dab_s[r * 2 * nj + j] = sA;
            dab_s[r * 2 * nj + nj + j] = sB;
        }
    }
}

// dx[t] = dx_shared[t] + sum_k (dx_routed[row_of[t][k]] + dz[t][k] * Wr[idx[t][k]]),
// FP32 accumulation in that order, bf16 result. One CTA per token, 4 columns a step.
__global__ void __launch_bounds__(256)
dx_combine_kernel(const uint16_t* __restrict__ dxr, const float* __restrict__ dxs, const int32_t* __restrict__ row_of,
                  const int32_t* __restrict__ topk_idx, const float* __restrict__ dz, const float* __restrict__ Wr,
                  int T, int K, int d, int E, uint16_t* __restrict__ dx) {
    __shared__ int64_t rows[16];
    __shared__ int64_t wrow[16];
    __shared__ float w[16];
    const int t = blockIdx.x;
    const int64_t TK = static_cast<int64_t>(T) * K;
    if (threadIdx.x < K) {
        int64_t r = __ldg(row_of + static_cast<int64_t>(t) * K + threadIdx.x);
        int e = __ldg(topk_idx + static_cast<int64_t>(t) * K + threadIdx.x);
        float g = __ldg(dz + static_cast<int64_t>(t) * K + threadIdx.x);
        if (r < 0 || r >= TK || e < 0 || e >= E) { set_status(MOE_ERR_DEVICE_CHECK); r = 0; e = 0; g = 0.0f; }
        rows[threadIdx.x] = r;
        wrow[threadIdx.x] = e;
        w[threadIdx.x] = g;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < d / 4; v += blockDim.x) {
        float4 acc = __ldg(reinterpret_cast<const float4*>(dxs + static_cast<int64_t>(t) * d) + v);
        for (int k = 0; k < K; ++k) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(dxr + rows[k] * d) + v);
            const float4 wr = __ldg(reinterpret_cast<const float4*>(Wr + wrow[k] * d) + v);
            const float g = w[k];
            acc.x += bf16_lo(u.x) + g * wr.x;
            acc.y += bf16_hi(u.x) + g * wr.y;
            acc.z += bf16_lo(u.y) + g * wr.z;
            acc.w += bf16_hi(u.y) + g * wr.w;
        }
        uint2 o;
        o.x = pack_bf16x2(acc.x, acc.y);
        o.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2*>(dx + static_cast<int64_t>(t) * d)[v] = o;
    }
}

// ----------------------------------------------- 128x1 grouped quantisation --
// Source of the values v[r][c] of a [rows][cols] operand.
enum Src { SRC_F32 = 0, SRC_FP8 = 1, SRC_BF16_ROWS = 2 };

struct QSrc {
    const float* f32;          // SRC_F32: [rows][ld]
    const uint8_t* q8;         // SRC_FP8: codes [rows][ld] with 1x128 scales s8 [rows][ld_s]
    const float* s8;
    const uint16_t* bf16;      // SRC_BF16_ROWS: row r is fl32(mult[r] * bf16[map[r]][.]) (mult may be null: 1)
    const int32_t* map;
    const float* mult;
    int64_t ld;
    int64_t ld_s;
    int64_t src_rows;          // SRC_BF16_ROWS: rows of bf16 (bound for map)
};

constexpr int kQ1MaxGroups = 1025;

// Grid (row-tile slots, cols / 128), 256 threads. Group g's rows
// offsets[g] .. offsets[g+1] form ceil(m_g / 128) row tiles; slot s (the s-th
// row tile over all groups in order) writes transposed columns 128 s .. 128 s
// + 127 of qT [cols][ldq] and scale row s of sT [*][cols]; rows past the
// group's end are zeros. Slots past the last tile exit.
template <int SRC, bool POW2>
__global__ void __launch_bounds__(256)
quant_128x1_kernel(QSrc src, int64_t rows, int cols, int groups, const int32_t* __restrict__ offsets,
                   uint8_t* __restrict__ qT, int64_t ldq, float* __restrict__ sT) {
    extern __shared__ float q1_smem[];
    float* tile = q1_smem;                               // [128][129]
    int* prefix = reinterpret_cast<int*>(q1_smem + 128 * 129);   // [groups + 1] tile prefix
    __shared__ float red[128];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    if (tid < 32) {
        int carry = 0;
        for (int b0 = 0; b0 < groups; b0 += 32) {
            const int g = b0 + tid;
            int v = 0;
            if (g < groups) {
                const int a = __ldg(offsets + g), b = __ldg(offsets + g + 1);
                if (a < 0 || b < a || b > rows) bad = 1;
                else v = (b - a + 127) / 128;
            }
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += u;
            }
            if (g < groups) prefix[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (tid == 0) prefix[groups] = carry;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(MOE_ERR_DEVICE_CHECK);
        return;
    }
    const int slot = blockIdx.x;
    if (slot >= prefix[groups]) return;
    if (static_cast<int64_t>(slot + 1) * 128 > ldq) {          // the caller's qT is too narrow
        if (tid == 0) set_status(MOE_ERR_DEVICE_CHECK);
        return;
    }
    int lo = 0, hi = groups - 1;                   // last g with prefix[g] <= slot
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int64_t row0 = __ldg(offsets + g) + static_cast<int64_t>(slot - prefix[g]) * 128;
    const int m = static_cast<int>(min(static_cast<int64_t>(128), __ldg(offsets + g + 1) - row0));
    const int c0 = blockIdx.y * 128;
    // load: 16-byte loads, all of a thread's issued before the tile is written (the kernel
    // is bound by HBM latency x bytes in flight). Rows past the group's end are zeros.
    if (SRC == SRC_F32) {
        // thread -> rows tid/32 + 8i (i < 16), columns 4 * (tid % 32) .. + 3
        const int tr = tid >> 5, tc = (tid & 31) * 4;
        float4 f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int rr = tr + 8 * i;
            f[i] = rr < m ? __ldg(reinterpret_cast<const float4*>(src.f32 + (row0 + rr) * src.ld + c0 + tc))
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float* d = tile + (tr + 8 * i) * 129 + tc;
            d[0] = f[i].x; d[1] = f[i].y; d[2] = f[i].z; d[3] = f[i].w;
        }
    } else if (SRC == SRC_FP8) {
        // thread -> rows tid/8 + 32i (i < 4), columns 16 * (tid % 8) .. + 15 (one 1x128 scale per row)
        const int tr = tid >> 3, tc = (tid & 7) * 16;
        uint4 w[4];
        float sc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = tr + 32 * i;
            w[i] = make_uint4(0, 0, 0, 0);
            sc[i] = 0.0f;
            if (rr < m) {
                const int64_t r = row0 + rr;
                w[i] = __ldg(reinterpret_cast<const uint4*>(src.q8 + r * src.ld + c0 + tc));
                sc[i] = __ldg(src.s8 + r * src.ld_s + (c0 >> 7));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float* d = tile + (tr + 32 * i) * 129 + tc;
            const uint32_t cw[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 lo2 = e4m3x2_to_f32(cw[k] & 0xFFFFu), hi2 = e4m3x2_to_f32(cw[k] >> 16);
                d[4 * k + 0] = __fmul_rn(lo2.x, sc[i]);
                d[4 * k + 1] = __fmul_rn(lo2.y, sc[i]);
                d[4 * k + 2] = __fmul_rn(hi2.x, sc[i]);
                d[4 * k + 3] = __fmul_rn(hi2.y, sc[i]);
            }
        }
    } else {
        // thread -> rows tid/16 + 16i (i < 8), columns 8 * (tid % 16) .. + 7
        const int tr = tid >> 4, tc = (tid & 15) * 8;
        uint4 w[8];
        float mu[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = tr + 16 * i;
            w[i] = make_uint4(0, 0, 0, 0);
            mu[i] = 1.0f;
            if (rr < m) {
                const int64_t r = row0 + rr;
                int64_t t = __ldg(src.map + r);
                if (t < 0 || t >= src.src_rows) { set_status(MOE_ERR_DEVICE_CHECK); t = 0; }
                w[i] = __ldg(reinterpret_cast<const uint4*>(src.bf16 + t * src.ld + c0 + tc));
                if (src.mult != nullptr) mu[i] = __ldg(src.mult + r);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float* d = tile + (tr + 16 * i) * 129 + tc;
            const uint32_t u[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float lo = bf16_lo(u[k]), hi = bf16_hi(u[k]);
                if (src.mult != nullptr) { lo = __fmul_rn(mu[i], lo); hi = __fmul_rn(mu[i], hi); }
                d[2 * k] = lo;
                d[2 * k + 1] = hi;
            }
        }
    }
    __syncthreads();
    // column pass: thread -> column tid % 128, rows 64 * (tid / 128) .. + 63
    const int col = tid & 127, half = tid >> 7;
    float amax = 0.0f;
    for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(tile[(half * 64 + j) * 129 + col]));
    if (half == 1) red[col] = amax;
    __syncthreads();
    if (half == 0) red[col] = fmaxf(red[col], amax);
    __syncthreads();
    const float s = tile_scale<POW2>(red[col]);
    uint8_t* dst = qT + static_cast<int64_t>(c0 + col) * ldq + static_cast<int64_t>(slot) * 128 + half * 64;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = half * 64 + q * 16 + u * 4;
            w4[u] = e4m3x4(quant_ratio(tile[j * 129 + col], s), quant_ratio(tile[(j + 1) * 129 + col], s),
                           quant_ratio(tile[(j + 2) * 129 + col], s), quant_ratio(tile[(j + 3) * 129 + col], s));
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    if (half == 0) sT[static_cast<int64_t>(slot) * cols + c0 + col] = s;
}

// One CTA per 128x128 block of q [batch][rows][cols]: the block's codes go
// transposed to qT [batch][colsT][ldT] (rows of the source become columns;
// rows cols .. colsT-1 of each matrix are left alone), its scale to
// sT [batch][colsT/128][ldT/128].
__global__ void __launch_bounds__(256)
transpose_blocks_kernel(const uint8_t* __restrict__ q, const float* __restrict__ s, int64_t rows, int64_t cols,
                        uint8_t* __restrict__ qT, float* __restrict__ sT, int64_t ldT, int64_t colsT) {
    __shared__ __align__(16) uint8_t tile[128][144];
    const int64_t bc = cols / 128, br = rows / 128;
    const int64_t blk = blockIdx.x;
    const int64_t b = blk / (br * bc);
    const int64_t rb = (blk / bc) % br, cb = blk % bc;
    const uint8_t* src = q + b * rows * cols + rb * 128 * cols + cb * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int row = idx >> 3, seg = idx & 7;
        *reinterpret_cast<uint4*>(&tile[row][seg * 16]) = __ldg(reinterpret_cast<const uint4*>(src + row * cols) + seg);
    }
    __syncthreads();
    uint8_t* dst = qT + b * colsT * ldT + cb * 128 * ldT + rb * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int oc = idx >> 3, seg = idx & 7;
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = seg * 16 + 4 * u;
            w[u] = static_cast<uint32_t>(tile[r][oc]) | (static_cast<uint32_t>(tile[r + 1][oc]) << 8) |
                   (static_cast<uint32_t>(tile[r + 2][oc]) << 16) | (static_cast<uint32_t>(tile[r + 3][oc]) << 24);
        }
        *reinterpret_cast<uint4*>(dst + oc * ldT + seg * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (threadIdx.x == 0) sT[(b * (colsT / 128) + cb) * (ldT / 128) + rb] = s[b * br * bc + rb * bc + cb];
}

}  // namespace bwd
}  // namespace moe
