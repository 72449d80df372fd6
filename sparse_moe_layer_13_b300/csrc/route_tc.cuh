// Router logits on the 5th-generation tensor cores, and the fused router.
//
// z[t][e] = sum_j x[t][j] * Wr[e][j] with x in bf16 (exact) and the FP32
// router weight split into three bf16 terms hi + mid + lo whose sum is Wr
// exactly (24 significand bits = 3 x 8). The GEMM runs over a contraction
// of length 3d in chunks c = (k block of 64, term) on bf16 tensor cores with
// FP32 accumulation in TMEM.
//
// Accuracy: the tensor core's accumulation of a long run of chunks drifts
// from the correctly rounded sum (measured on the B300 at d = 7168 against
// FP64: mean |error| 1.4e-6 with runs of 24 chunks, 3.0e-7 with runs of 3),
// and the selection compares affinities to 1e-6. So a CTA accumulates runs
// ("sub-splits") of at most kMaxChunksPerSplit chunks in one of two TMEM
// buffers (2 x 256 columns) and its summing warps add the runs in order in
// FP32 registers while the tensor core fills the other buffer.
//
// One CTA per (128-token tile, <=256-expert tile, K slice); a K slice is a
// contiguous range of sub-splits, more than one only to fill the SMs when
// the batch is small:
//   warp 0      TMA: x (128x64 bf16) and one weight term (BNx64 bf16) per chunk
//   warp 1      MMA: 4 x tcgen05.mma.kind::f16 (K=16) per chunk
//   warps 2..9  sum the sub-splits, 128 logits per thread (lane quadrant =
//               warp % 4, column half = (warp - 2) / 4)
// Then, with SELECT (one slice, all E <= 256 experts in the CTA), the sums go
// to shared memory (the operand ring, idle by then) and to z [T][E], and all
// ten warps run the warp-per-token selection on them: only the choice and
// the summed logits reach HBM. Without SELECT the slice sums go to
// z_part[slice][T][E] and route::select_kernel adds the slices in order;
// with one slice both give the same bits.
#pragma once

#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace rtc {

constexpr int BM = 128;
constexpr int BK = 64;                 // bf16 elements per 128-byte row
constexpr int BN_MAX = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_MAX * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
#ifndef MOE_ROUTE_MAX_CHUNKS
#define MOE_ROUTE_MAX_CHUNKS 3
#endif
constexpr int kMaxChunksPerSplit = MOE_ROUTE_MAX_CHUNKS;   // chunks of 64 per TMEM accumulation run
constexpr int kMaxSlices = 16;                              // K slices across CTAs (small batches)

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

struct FParams {
    int T, d, E, G, M, K, gk;
    int subs_per_slice;      // sub-splits of kMaxChunksPerSplit chunks per K slice (gridDim.z slices)
    const float* offset;     // per-expert logit offset or nullptr (SELECT)
    const float* bias;       // selection bias [E] (SELECT)
    int32_t* topk_idx;       // [T][K] (SELECT)
    float* topk_gate;        // [T][K] (SELECT)
    float* z;                // SELECT: summed logits [T][E]; else slice sums [gridDim.z][T][E]
    int* splits;             // workspace word: slice planes of the stored logits
};

template <bool SELECT, int EPL, int MAXGK>
__global__ void __launch_bounds__(F_THREADS, 1)
route_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, FParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    FSmem& s = *reinterpret_cast<FSmem*>(base + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int t0 = blockIdx.x * BM;
    const int n0 = blockIdx.y * BN_MAX;
    const int E = p.E;
    const int bn = min(BN_MAX, E - n0);                  // multiple of 16
    const int nchunks = 3 * (p.d / BK);
    const int c_begin = blockIdx.z * p.subs_per_slice * kMaxChunksPerSplit;
    const int c_end = min(nchunks, c_begin + p.subs_per_slice * kMaxChunksPerSplit);
    const int nsub = (c_end - c_begin + kMaxChunksPerSplit - 1) / kMaxChunksPerSplit;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&s.tfull[i], 1); mbar_init(&s.tempty[i], 8); }
        mbar_init(&s.done, 1);
        s.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            *p.splits = SELECT ? 1 : static_cast<int>(gridDim.z);
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
    // the weight box is min(E, 256) rows for every expert tile (a last tile narrower
    // than the box still receives, and counts, the whole box)
    const uint32_t tx_bytes = A_BYTES + static_cast<uint32_t>(min(E, BN_MAX)) * BK * 2;

    float acc[128];                                      // summing warps: this thread's 128 logits
    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int c = c_begin; c < c_end; ++c, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs)) break;
                const int kb = c / 3, term = c - 3 * kb;
                mbar_expect_tx(&s.full[st], tx_bytes);
                tma_load_2d(sA + st * A_BYTES, &tmX, &s.full[st], kb * BK, t0);
                tma_load_2d(sB + st * B_BYTES, &tmW, &s.full[st], kb * BK, term * E + n0);
            }
            if (*abort) {      // let every issued copy land before the CTA moves on
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = make_idesc(BM, static_cast<uint32_t>(bn), 1);
            uint32_t it = 0;
            bool ok = true;
            for (int sp = 0; sp < nsub && ok; ++sp) {
                const uint32_t b = sp & 1, bph = (sp >> 1) & 1;
                if (!mbar_wait(&s.tempty[b], bph ^ 1u, abort, kWaitLimitNs)) break;
                const int c0 = c_begin + sp * kMaxChunksPerSplit, c1 = min(c_end, c0 + kMaxChunksPerSplit);
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
        for (int sp = 0; sp < nsub; ++sp) {
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
    if constexpr (!SELECT) {
        // this slice's sums to z_part[slice][t][n0 + col]
        if (ok && warp >= 2) {
            const int q = warp & 3, half = (warp - 2) >> 2;
            const int row = t0 + q * 32 + static_cast<int>(lane);
            if (row < p.T) {
                float* dst = p.z + (static_cast<int64_t>(blockIdx.z) * p.T + row) * E + n0 + half * 128;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (half * 128 + 4 * i < bn)
                        reinterpret_cast<float4*>(dst)[i] =
                            make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
            }
        }
    } else {
        float* zs = reinterpret_cast<float*>(base);      // staged logits [BM][F_LD]
        float* sel = zs + BM * F_LD;                     // per-warp selection rows [F_WARPS][2][E]
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
