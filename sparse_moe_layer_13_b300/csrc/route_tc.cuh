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
// kernel sums the K-split partials in a fixed order. This split path serves
// batches too small to fill the GPU with one CTA per token tile; larger ones
// take the fused kernel below.
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
#ifndef MOE_ROUTE_MAX_CHUNKS
#define MOE_ROUTE_MAX_CHUNKS 24
#endif
constexpr int kMaxChunksPerSplit = MOE_ROUTE_MAX_CHUNKS;   // chunks of 64 accumulated per TMEM K split

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
    int* splits;        // workspace word: split count of the stored logits
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
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) *p.splits = p.ksplit;
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

#include "route.cuh"

namespace moe {
namespace rtc {

// ---------------------------------------------------------------------------
// Fused router: logits, K-split sums and selection in one kernel, one CTA per
// 128-token tile with all E <= 256 experts, so only the choice (and the
// summed logits, 1/ksplit of the partials' bytes) ever reaches HBM.
//
//   warp 0      TMA: x (128x64 bf16) and one weight term (Ex64 bf16) per chunk
//   warp 1      MMA: the chunks of K split s accumulate in TMEM buffer s % 2
//               (2 x 256 columns); the split's last commit hands it over
//   warps 2..9  sum the splits in registers in split order (the first split
//               assigned, each later one added: the same FP32 additions the
//               split-path selection makes), 128 logits per thread: lane
//               quadrant = warp % 4, column half = (warp - 2) / 4
// Then the sums go to shared memory (the operand ring, idle by then) and to
// z [T][E] in the workspace, and all ten warps run the warp-per-token
// selection on them. With the same split count the results equal the split
// path's bit for bit.
constexpr int F_THREADS = 320;
constexpr int F_WARPS = F_THREADS / 32;
constexpr int F_LD = BN_MAX + 4;                    // staged logit row stride (floats), 16-byte rows
constexpr uint32_t F_TMEM_COLS = 2 * BN_MAX;
constexpr size_t F_LOGIT_BYTES = static_cast<size_t>(BM) * F_LD * sizeof(float);
constexpr size_t F_SEL_BYTES = static_cast<size_t>(F_WARPS) * 2 * BN_MAX * sizeof(float);
static_assert(F_LOGIT_BYTES + F_SEL_BYTES <= static_cast<size_t>(STAGES) * STAGE_BYTES,
              "staged logits and selection rows must fit in the operand ring");

struct FSmem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t F_SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + sizeof(FSmem);

struct FParams {
    int T, d, E, ksplit, G, M, K, gk;
    const float* offset;     // per-expert logit offset or nullptr
    const float* bias;       // selection bias [E]
    int32_t* topk_idx;       // [T][K]
    float* topk_gate;        // [T][K]
    float* z;                // summed logits [T][E]
    int* splits;             // workspace word: split count of the stored logits (1 here)
};

template <int EPL, int MAXGK>
__global__ void __launch_bounds__(F_THREADS, 1)
fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, FParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    FSmem& s = *reinterpret_cast<FSmem*>(base + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int t0 = blockIdx.x * BM;
    const int E = p.E;                                   // <= 256, multiple of 16
    const int nchunks = 3 * (p.d / BK);
    const int per = (nchunks + p.ksplit - 1) / p.ksplit;
    const int nsplit = (nchunks + per - 1) / per;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&s.tfull[i], 1); mbar_init(&s.tempty[i], 8); }
        mbar_init(&s.done, 1);
        s.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (blockIdx.x == 0) *p.splits = 1;
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, F_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;
    const uint32_t tx_bytes = A_BYTES + static_cast<uint32_t>(E) * BK * 2;

    float acc[128];                                      // summing warps: this thread's 128 logits
    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int c = 0; c < nchunks; ++c, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs)) break;
                const int kb = c / 3, term = c - 3 * kb;
                mbar_expect_tx(&s.full[st], tx_bytes);
                tma_load_2d(sA + st * A_BYTES, &tmX, &s.full[st], kb * BK, t0);
                tma_load_2d(sB + st * B_BYTES, &tmW, &s.full[st], kb * BK, term * E);
            }
            if (*abort) {      // let every issued copy land before the CTA moves on
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = make_idesc(BM, static_cast<uint32_t>(E), 1);
            uint32_t it = 0;
            bool ok = true;
            for (int sp = 0; sp < nsplit && ok; ++sp) {
                const uint32_t b = sp & 1, bph = (sp >> 1) & 1;
                if (!mbar_wait(&s.tempty[b], bph ^ 1u, abort, kWaitLimitNs)) break;
                const int c0 = sp * per, c1 = min(nchunks, c0 + per);
                for (int c = c0; c < c1; ++c, ++it) {
                    const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(&s.full[st], ph, abort, kWaitLimitNs)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_addr(sA + st * A_BYTES));
                    const uint64_t bd = sw128_desc(smem_addr(sB + st * B_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16(tmem + b * BN_MAX, ad + 2 * k, bd + 2 * k, idesc, (c > c0 || k > 0) ? 1u : 0u);
                    tc_commit(&s.empty[st]);
                }
                if (ok) tc_commit(&s.tfull[b]);
            }
            tc_commit(&s.done);
            mbar_wait(&s.done, 0, nullptr, kWaitLimitNs);   // no MMA in flight when TMEM is freed
        }
    } else {
        const int q = warp & 3;                          // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;                // column half
        for (int sp = 0; sp < nsplit; ++sp) {
            const uint32_t b = sp & 1, bph = (sp >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[b], bph, abort, kWaitLimitNs))) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN_MAX + half * 128;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint32_t v[32];
                tmem_ld32(taddr + r * 32, v);
                tmem_ld_wait();
                tmem_reg_fence(v);
                if (r == 3) {                            // the buffer is in registers: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.tempty[b]);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    acc[r * 32 + i] = sp == 0 ? __uint_as_float(v[i]) : acc[r * 32 + i] + __uint_as_float(v[i]);
            }
        }
    }
    __syncthreads();                                     // every MMA done, the operand ring idle
    const bool ok = *abort == 0;
    float* zs = reinterpret_cast<float*>(base);          // staged logits [BM][F_LD]
    float* sel = zs + BM * F_LD;                         // per-warp selection rows [F_WARPS][2][E]
    if (ok && warp >= 2) {
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int row = q * 32 + static_cast<int>(lane);
        const uint32_t dst = smem_addr(zs + row * F_LD + half * 128);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (half * 128 + 4 * i < E)
                st_shared_v4(dst + 16 * i, acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
    }
    __syncthreads();
    if (ok) {
        const int rows = min(BM, p.T - t0);
        // summed logits to the workspace (router backward, balance statistics), a row per warp step
        for (int r = warp; r < rows; r += F_WARPS) {
            const float4* src = reinterpret_cast<const float4*>(zs + r * F_LD);
            float4* dst = reinterpret_cast<float4*>(p.z + static_cast<int64_t>(t0 + r) * E);
            for (int c = static_cast<int>(lane); c < E / 4; c += 32) dst[c] = src[c];
        }
        float* spw = sel + static_cast<size_t>(warp) * 2 * E;
        for (int r = warp; r < rows; r += F_WARPS) {
            float zz[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = static_cast<int>(lane) + 32 * i;
                zz[i] = e < E ? zs[r * F_LD + e] : 0.0f;
            }
            route::select_token<EPL, MAXGK>(zz, static_cast<int64_t>(t0 + r), E, p.G, p.M, p.K, p.gk, p.offset,
                                            p.bias, spw, spw + E, p.topk_idx, p.topk_gate);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, F_TMEM_COLS);
    }
}

}  // namespace rtc
}  // namespace moe
