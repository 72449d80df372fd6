// Weight-gradient GEMM of the backward pass: per group g,
//   D_g[m][n] = sum over the 128-token chunks kc of g's rows of
//               saT[kc][m] * sbT[kc][n] * sum_{r in kc} AT[m][r] BT[n][r]
// with both operands E4M3, transposed (tokens contiguous) and scaled per 128
// tokens x 1 channel ("DeepSeek-V3的MoE架构设计革新" §2 FP8 training: the
// activation rule taken along the contracted dimension, which for a weight
// gradient is the tokens), partial sums promoted to FP32 at every chunk.
// Group g's rows are chunks chunk0_g .. chunk0_g + ceil(m_g/128) - 1 of the
// transposed operands (quant_128x1_kernel's layout); D is FP32 [groups][M][N].
//
// Same warp roles as the grouped forward GEMM: warp 0 TMA producer (operand
// tiles 128x128 and 256x128 into a 3-stage ring; the chunk's 128 + 256 scale
// values by bulk copy into a 4-slot scale ring), warp 1 MMA issuer
// (tcgen05.mma M128 N256 K32 into two TMEM chunk accumulators), warps 4..11
// epilogue (row rit of the tile, 128 columns: acc += partial * sa[rit] * sb[n];
// the finished tile leaves through shared memory by TMA stores of 32x32 boxes,
// since direct stores of 32 rows per warp instruction tie up L1).
// Tiles: groups in reverse order (the shared expert, last and largest, first),
// then row tile, then column tile; CTA c takes tiles c, c + gridDim.x, ...
// A group with no rows gets zero tiles.
#pragma once

#include "common.cuh"
#include "gemm_fp8.cuh"

namespace moe {
namespace wgrad {

using gemm::BK;
using gemm::BM;
using gemm::BN;
using gemm::A_BYTES;
using gemm::B_BYTES;
using gemm::STAGE_BYTES;
using gemm::NUM_THREADS;
using gemm::kRegsEpilogue;
using gemm::kRegsProducer;
using gemm::TMEM_COLS;
using gemm::IDESC;
constexpr int STAGES = 3;                 // operand ring (few K chunks per tile; room for the store staging)
constexpr int SSLOTS = 4;                 // scale ring
constexpr int OUT_BOX = 32;               // output box: 32 rows x 32 FP32 columns, 128-byte swizzle
constexpr int OUT_BOX_BYTES = OUT_BOX * OUT_BOX * 4;
constexpr int OUT_STAGE_BYTES = 8 * 2 * OUT_BOX_BYTES;   // two boxes per epilogue warp
constexpr int MAX_GROUPS = 1025;
constexpr uint32_t SCALE_BYTES = (BM + BN) * sizeof(float);

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[4];                // chunk it's TMEM buffer read out (index it % 4, one arrive per epilogue warp)
    uint64_t sfull[SSLOTS];
    uint64_t sempty[SSLOTS];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    int bad;
    int chunk0[MAX_GROUPS + 1];        // exclusive prefix of ceil(m_g / 128)
    alignas(16) float sa[SSLOTS][BM];
    alignas(16) float sb[SSLOTS][BN];
};

constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OUT_STAGE_BYTES + sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may have");

struct Params {
    const int32_t* offsets;   // [groups + 1] row offsets of the groups
    int32_t groups;
    int64_t rows;             // offsets[groups] <= rows
    int64_t chunks;           // 128-token chunks the transposed operands hold (width / 128)
    int32_t M;
    int32_t N;
    const float* saT;         // [chunks][M]
    const float* sbT;         // [chunks][N]
    float* out;               // [groups][M][N]
};

__device__ __forceinline__ void decode(int tile, int groups, int mtn, int ntn, int& g, int& mt, int& nt) {
    const int per = mtn * ntn;
    const int q = tile / per;
    g = groups - 1 - q;
    const int rem = tile - q * per;
    mt = rem / ntn;
    nt = rem - mt * ntn;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_wgrad_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmOut, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    uint8_t* sOut = base + STAGES * STAGE_BYTES;                    // 1024-byte aligned
    Smem& s = *reinterpret_cast<Smem*>(sOut + OUT_STAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int groups = p.groups;
    const int mtn = p.M / BM, ntn = p.N / BN;
    const int total = groups * mtn * ntn;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
        for (int i = 0; i < 2; ++i) mbar_init(&s.tfull[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&s.tempty[i], 8);
        for (int i = 0; i < SSLOTS; ++i) { mbar_init(&s.sfull[i], 1); mbar_init(&s.sempty[i], 8); }
        mbar_init(&s.mma_done, 1);
        s.abort = 0;
        s.bad = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    if (warp == 2) {
        int carry = 0;
        for (int b0 = 0; b0 < groups; b0 += 32) {
            const int g = b0 + static_cast<int>(lane);
            int v = 0;
            if (g < groups) {
                const int a = __ldg(p.offsets + g), b = __ldg(p.offsets + g + 1);
                if (a < 0 || b < a || static_cast<int64_t>(b) > p.rows) s.bad = 1;
                else v = (b - a + BM - 1) / BM;
            }
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (static_cast<int>(lane) >= o) incl += t;
            }
            if (g < groups) s.chunk0[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            s.chunk0[groups] = carry;
            if (carry > p.chunks) s.bad = 1;     // the operands are narrower than the rows need
        }
        __syncwarp();
        if (lane == 0 && s.bad && blockIdx.x == 0) set_status(MOE_ERR_DEVICE_CHECK);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;
    const bool run = !s.bad;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
      if (warp == 0 && lane == 0 && run) {
        // ---------------------------------------------------- TMA producer ----
        uint32_t it = 0, n_sc = 0;        // operand stages and scale slots issued
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            int g, mt, nt;
            decode(tile, groups, mtn, ntn, g, mt, nt);
            const int c0 = s.chunk0[g], nk = s.chunk0[g + 1] - c0;
            for (int kc = 0; kc < nk; ++kc) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                const uint32_t ss = it % SSLOTS, sph = (it / SSLOTS) & 1u;
                if (!(ok = mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs))) break;
                mbar_expect_tx(&s.full[st], STAGE_BYTES);
                tma_load_2d(sA + st * A_BYTES, &tmA, &s.full[st], (c0 + kc) * BK, mt * BM);
                tma_load_2d(sB + st * B_BYTES, &tmB, &s.full[st], (c0 + kc) * BK, nt * BN);
                ++it;
                if (!(ok = mbar_wait(&s.sempty[ss], sph ^ 1u, abort, kWaitLimitNs))) break;
                mbar_expect_tx(&s.sfull[ss], SCALE_BYTES);
                const int64_t chunk = c0 + kc;
                bulk_load(s.sa[ss], p.saT + chunk * p.M + mt * BM, BM * sizeof(float), &s.sfull[ss]);
                bulk_load(s.sb[ss], p.sbT + chunk * p.N + nt * BN, BN * sizeof(float), &s.sfull[ss]);
                ++n_sc;
            }
        }
        if (*abort) {
            // let every issued copy land before the CTA exits
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
            for (uint32_t j = n_sc > SSLOTS ? n_sc - SSLOTS : 0; j < n_sc; ++j)
                mbar_wait(&s.sfull[j % SSLOTS], (j / SSLOTS) & 1u, nullptr, kWaitLimitNs);
        }
      } else if (warp == 1 && lane == 0 && run) {
        // ------------------------------------------------------ MMA issuer ----
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
            int g, mt, nt;
            decode(tile, groups, mtn, ntn, g, mt, nt);
            const int nk = s.chunk0[g + 1] - s.chunk0[g];
            bool ok = true;
            for (int kc = 0; kc < nk; ++kc, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                const uint32_t b = it & 1u;
                // buffer b is free once chunk it - 2 has been read out
                if (it >= 2 && !(ok = mbar_wait(&s.tempty[(it - 2) & 3u], ((it - 2) >> 2) & 1u, abort, kWaitLimitNs)))
                    break;
                if (!(ok = mbar_wait(&s.full[st], ph, abort, kWaitLimitNs))) break;
                tc_fence_after();
                const uint64_t ad = sw128_desc(smem_addr(sA + st * A_BYTES));
                const uint64_t bd = sw128_desc(smem_addr(sB + st * B_BYTES));
#pragma unroll
                for (int k = 0; k < BK / 32; ++k)
                    mma_e4m3(tmem + b * BN, ad + 2 * k, bd + 2 * k, IDESC, k > 0 ? 1u : 0u);
                tc_commit(&s.empty[st]);
                tc_commit(&s.tfull[b]);
            }
            if (!ok) break;
        }
        // no MMA may be in flight when TMEM is released
        tc_commit(&s.mma_done);
        mbar_wait(&s.mma_done, 0, nullptr, kWaitLimitNs);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
        // -------------------------------------------------------- epilogue ----
        const int ew = warp - 4;             // 0..7
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int half = ew >> 2;            // column half of the 256-wide tile
        const int rit = q * 32 + static_cast<int>(lane);
        uint32_t it = 0, nbox = 0;
        bool ok = run;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            int g, mt, nt;
            decode(tile, groups, mtn, ntn, g, mt, nt);
            const int nk = s.chunk0[g + 1] - s.chunk0[g];
            float2 acc2[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.0f, 0.0f);
            for (int kc = 0; kc < nk; ++kc, ++it) {
                const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
                const uint32_t ss = it % SSLOTS, sph = (it / SSLOTS) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&s.sfull[ss], sph, abort, kWaitLimitNs))) { ok = false; break; }
                const float sav = s.sa[ss][rit];
                if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[b], bph, abort, kWaitLimitNs))) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN + half * 128;
                const float2 sa2 = make_float2(sav, sav);
                // four steps of 32 columns (half * 128 + r * 32 ..): fewer live registers than two of 64
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    uint32_t v[32];
                    tmem_ld32(taddr + r * 32, v);
                    tmem_ld_wait();
                    tmem_reg_fence(v);
                    if (r == 3) {                // every value of the chunk is in registers now
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&s.tempty[it & 3u]);
                    }
                    const float4* sbp = reinterpret_cast<const float4*>(&s.sb[ss][half * 128 + r * 32]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 w = sbp[i];
                        float2* a = &acc2[r * 16 + 2 * i];
                        a[0] = __ffma2_rn(__fmul2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                                                     make_float2(w.x, w.y)), sa2, a[0]);
                        a[1] = __ffma2_rn(__fmul2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                                                     make_float2(w.z, w.w)), sa2, a[1]);
                    }
                }
                // every scale of this chunk has been read
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.sempty[ss]);
            }
            if (!ok) break;
            float* acc = reinterpret_cast<float*>(acc2);
            // 4 boxes of 32 columns: the warp's 32 rows go to shared memory in the 128-byte
            // swizzled box layout (16-byte chunk c of row r at chunk c ^ (r % 8): a quarter warp
            // covers all banks), then one lane stores the box with TMA. Two boxes alternate; a box
            // is rewritten only after the store issued two boxes earlier has read it.
            const int y = g * p.M + mt * BM + q * 32;
#pragma unroll
            for (int j = 0; j < 4; ++j, ++nbox) {
                uint8_t* buf = sOut + (ew * 2 + (nbox & 1u)) * OUT_BOX_BYTES;
                if (nbox >= 2) {
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                }
                const uint32_t row = smem_addr(buf) + lane * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(row + ((c ^ (lane & 7)) << 4), acc[32 * j + 4 * c], acc[32 * j + 4 * c + 1],
                                 acc[32 * j + 4 * c + 2], acc[32 * j + 4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmOut, buf, nt * BN + half * 128 + j * 32, y);
                    bulk_commit();
                }
            }
        }
        // every store has finished with shared memory (and written its box) before the CTA exits
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace wgrad
}  // namespace moe
