// Router logits on the 5th-generation tensor cores.
//
// z[t][e] = sum_j x[t][j] * Wr[e][j] with x in bf16 (exact) and the FP32
// router weight split into three bf16 terms hi + mid + lo whose sum is Wr
// exactly (24 significand bits = 3 x 8). The GEMM runs over a contraction
// of length 3d, chunk c = (k block, term), accumulating in FP32 in TMEM, so
// the logits carry FP32-accumulation accuracy at bf16 tensor-core rate.
//
// One CTA per (128-token tile, <=256-expert tile, K split): warp 0 loads A
// (x, 128x64 bf16) and B (one term, BNx64 bf16) per chunk by TMA into a
// 4-stage ring; warp 1 issues 4 x tcgen05.mma.kind::f16 (K=16) per chunk;
// warps 2-5 copy the FP32 accumulator to z_part[split][t][e]. The selection
// kernel sums the K-split partials in a fixed order.
#pragma once

#include "common.cuh"

namespace moe {
namespace rtc {

constexpr int BM = 128;
constexpr int BK = 64;                 // bf16 elements per 128-byte row
constexpr int BN_MAX = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_MAX * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int kMaxChunksPerSplit = 24;

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + sizeof(Smem);

// Wr (FP32) -> three bf16 planes [3][E][d] with hi + mid + lo == Wr.
__global__ void split_kernel(const float* __restrict__ w, int64_t n, uint16_t* __restrict__ planes) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    planes[i] = *reinterpret_cast<const uint16_t*>(&hi);
    planes[n + i] = *reinterpret_cast<const uint16_t*>(&mid);
    planes[2 * n + i] = *reinterpret_cast<const uint16_t*>(&lo);
}

struct Params {
    int T, d, E, bn, ksplit;
    float* z_part;      // [ksplit][T][E]
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
logits_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    Smem& s = *reinterpret_cast<Smem*>(base + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int t0 = blockIdx.x * BM;
    const int n0 = blockIdx.y * BN_MAX;
    const int bn = min(p.bn, p.E - n0);                  // multiple of 16
    const int kblocks = p.d / BK;
    const int nchunks = 3 * kblocks;
    const int per = (nchunks + p.ksplit - 1) / p.ksplit;
    const int c0 = blockIdx.z * per;
    const int c1 = min(nchunks, c0 + per);
    uint32_t ncols = 32;
    while (ncols < static_cast<uint32_t>(bn)) ncols <<= 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
        mbar_init(&s.done, 1);
        s.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;
    const uint32_t tx_bytes = A_BYTES + static_cast<uint32_t>(bn) * BK * 2;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int c = c0; c < c1; ++c, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs)) break;
                const int kb = c / 3, term = c - 3 * kb;
                mbar_expect_tx(&s.full[st], tx_bytes);
                tma_load_2d(sA + st * A_BYTES, &tmX, &s.full[st], kb * BK, t0);
                tma_load_2d(sB + st * B_BYTES, &tmW, &s.full[st], kb * BK, term * p.E + n0);
            }
            if (*abort) {
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = make_idesc(BM, static_cast<uint32_t>(bn), 1);
            uint32_t it = 0;
            for (int c = c0; c < c1; ++c, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(&s.full[st], ph, abort, kWaitLimitNs)) break;
                tc_fence_after();
                const uint64_t ad = sw128_desc(smem_addr(sA + st * A_BYTES));
                const uint64_t bd = sw128_desc(smem_addr(sB + st * B_BYTES));
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
                tc_commit(&s.empty[st]);
            }
            tc_commit(&s.done);
            mbar_wait(&s.done, 0, nullptr, kWaitLimitNs);   // no MMA in flight when TMEM is freed
        }
    } else {
        // warps 2..5: TMEM lane quadrant = warp % 4
        const int q = warp & 3;
        const int row = t0 + q * 32 + static_cast<int>(lane);
        const bool ok = mbar_wait(&s.done, 0, abort, kWaitLimitNs);
        tc_fence_after();
        if (ok) {
            float* dst = p.z_part + (static_cast<int64_t>(blockIdx.z) * p.T + row) * p.E + n0;
            for (int c = 0; c < bn; c += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, v);
                tmem_ld_wait();
                tmem_reg_fence(v);
                if (row < p.T) {
                    const int nv = min(32, bn - c);
                    if (nv == 32) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            reinterpret_cast<float4*>(dst + c)[i] =
                                make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < nv) dst[c + i] = __uint_as_float(v[i]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

}  // namespace rtc
}  // namespace moe
