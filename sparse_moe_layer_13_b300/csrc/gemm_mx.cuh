// Block-scaled grouped FP8 GEMM: the power-of-two scale variant of the
// grouped GEMM ("DeepSeek-V3的MoE架构设计革新" §2 items 1-2 with every 1x128 /
// 128x128 scale a power of two, see moe_scale_rule).
//
// With power-of-two scales the per-chunk promotion sa * sb * partial is a
// scaling by 2^(ea + eb), which tcgen05.mma.kind::mxf8f6f4.block_scale
// applies inside the tensor core from 8-bit exponent codes (UE8M0) held in
// TMEM. One accumulator then collects the whole K reduction of a tile, and
// the epilogue runs once per tile instead of once per 128-element chunk.
//
// Persistent, warp-specialised, one CTA per SM, 384 threads:
//   warp 0      TMA producer: A tile 128x128 and B tile 256x128 per K chunk
//               into a 4-stage ring (128-byte swizzle), as in the FP32-scale
//               kernel.
//   warp 1      MMA issuer: per chunk, three tcgen05.cp 32x128b.warpx4 copy the
//               chunk's scale factors from shared memory into TMEM, then four
//               block-scaled MMAs (M=128, N=256, K=32) accumulate into the
//               tile accumulator (TMEM columns 0..255).
//   warps 2,3   scale staging: turn the chunk's FP32 power-of-two scales into
//               UE8M0 words in the layout the copy expects (below), a group of
//               four chunks ahead in registers, across tile boundaries.
//   warps 4-11  epilogue: per tile, read the accumulator (128 values per
//               thread), release it, then store as the FP32-scale kernel does.
//
// Scale factors in TMEM (scale_vec::1X, one per row of A / per column of D
// for each K=32 step): every 32-lane quadrant holds a full copy; A's row
// 32j + l sits at column j, lane l (4 columns) and B's row n = 32j + l at
// column j, lane l (8 columns); byte i of each 32-bit cell serves scale
// factor id i (all four bytes equal here: the scale is constant over the
// 128-element chunk). In shared memory one 32x128b block is 32 rows of 16
// bytes (row l = columns 0..3 of lane l), 512 bytes: SFA, then SFB columns
// 0-3, then SFB columns 4-7.
#pragma once

#include "gemm_fp8.cuh"

namespace moe {
namespace gemm_mx {

using gemm::A_BYTES;
using gemm::B_BYTES;
using gemm::BK;
using gemm::BM;
using gemm::BN;
using gemm::MAX_GROUPS;
using gemm::NUM_THREADS;
using gemm::Params;
using gemm::STAGE_BYTES;
using gemm::STAGES;
using gemm::TILE_TAB;
using gemm::TileInfo;
using gemm::TMEM_COLS;

// Register split: 128 x 56 + 256 x 224 = 7168 + 57344 = 64512 = 384 x 168.
constexpr uint32_t kRegsProducer = 56;
constexpr uint32_t kRegsEpilogue = 224;
constexpr int SF_WORDS = 3 * 128;              // per stage: SFA block + two SFB blocks, 512 bytes each
constexpr uint32_t SF_TMEM_COL = 256;          // stage st's scale factors: TMEM columns 256 + 12 st ..
// kind::mxf8f6f4 instruction descriptor: E4M3 A and B (format 0), both K-major,
// N >> 3 at bit 17, UE8M0 scale type (bit 23), M >> 4 at bit 24, scale-factor
// ids 0 (bits 4-5 for B, 29-30 for A).
constexpr uint32_t IDESC_MX = (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                              (static_cast<uint32_t>(BM >> 4) << 24);

struct Smem {
    uint64_t full[STAGES];            // TMA bytes (producer's arrive) + one arrive per staging warp
    uint64_t empty[STAGES];
    uint64_t tfull;                   // accumulator holds a finished tile
    uint64_t tempty;                  // accumulator read out (one arrive per epilogue warp)
    uint64_t mma_done;
    uint64_t pair[4];                 // SwiGLU amax exchange between the two warps of a lane quadrant
    uint32_t tmem_base;
    int abort;
    int bad;
    int mtiles_total;
    int row_start[MAX_GROUPS + 1];
    int mtile_prefix[MAX_GROUPS + 1];
    float amax_x[2][8][32];
    uint2 tile_tab[TILE_TAB];
    alignas(128) uint32_t sf[STAGES][SF_WORDS];
};

constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may have");
static_assert(SF_TMEM_COL + STAGES * 12 <= TMEM_COLS, "scale factor columns outside the allocation");

// UE8M0 code (the biased exponent) of an FP32 power-of-two scale. A zero scale
// (all-zero tile, codes 0) takes code 0 (2^-127). Anything else that is not a
// positive power of two sets `bad`.
__device__ __forceinline__ uint32_t ue8m0(float sc, bool& bad) {
    const uint32_t b = __float_as_uint(sc);
    const uint32_t e = (b >> 23) & 0xFFu;
    if ((b & 0x807FFFFFu) != 0 || e == 0xFFu) bad = true;
    return e;
}

// the codes of four chunks, chunk c in byte c
__device__ __forceinline__ uint32_t ue8m0_x4(float s0, float s1, float s2, float s3, bool& bad) {
    return ue8m0(s0, bad) | (ue8m0(s1, bad) << 8) | (ue8m0(s2, bad) << 16) | (ue8m0(s3, bad) << 24);
}

// chunk c's code of a packed group, in all four bytes of a word (one byte per scale-factor id)
__device__ __forceinline__ uint32_t code_word(uint32_t packed, int c) {
    return ((packed >> (8 * c)) & 0xFFu) * 0x01010101u;
}

// shared-memory descriptor of one 32x128b scale block for tcgen05.cp: no
// swizzle, 8-row x 16-byte core matrices, 128 bytes apart along the rows
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// D[tmem] (+)= (A * 2^sfa) x (B * 2^sfb)^T, E4M3 x E4M3 -> FP32, one K=32 step
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// UE8M0 codes of four consecutive chunks (byte c: chunk 4 grp + c) for one staging
// thread: its two A rows and the tile's two weight blocks (B rows [0,128) and
// [128,256) of the column tile).
struct ScaleGroup {
    uint32_t a0, a1, b0, b1;
};

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    Smem& s = *reinterpret_cast<Smem*>(base + STAGES * STAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int groups = p.groups;
    const int ntiles = p.N / BN;
    const int nkc = p.Kdim / BK;

    // ---- set-up: barriers, TMEM, per-group row tiles, this CTA's tile table ----
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 3); mbar_init(&s.empty[i], 1); }
        mbar_init(&s.tfull, 1);
        mbar_init(&s.tempty, 8);
        mbar_init(&s.mma_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&s.pair[i], 64);
        s.abort = 0;
        s.bad = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    for (int g = threadIdx.x; g <= groups; g += NUM_THREADS) s.row_start[g] = __ldg(p.offsets + g);
    __syncthreads();
    for (int g = threadIdx.x; g < groups; g += NUM_THREADS) {
        const int a = s.row_start[g], b = s.row_start[g + 1];
        if (a < 0 || b < a || static_cast<int64_t>(b) > p.rows) s.bad = 1;
    }
    __syncthreads();
    if (warp == 2) {
        int carry = 0;
        for (int b0 = 0; b0 < groups; b0 += 32) {
            const int g = b0 + static_cast<int>(lane);
            int v = 0;
            if (g < groups && !s.bad) v = (s.row_start[g + 1] - s.row_start[g] + BM - 1) / BM;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (static_cast<int>(lane) >= o) incl += t;
            }
            if (g < groups) s.mtile_prefix[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            s.mtile_prefix[groups] = carry;
            s.mtiles_total = carry;
            if (s.bad && blockIdx.x == 0) set_status(MOE_ERR_DEVICE_CHECK);
        }
    }
    __syncthreads();
    const int total = s.mtiles_total * ntiles;
    for (int k = threadIdx.x; k < TILE_TAB; k += NUM_THREADS) {
        const int tile = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        if (tile >= total) break;
        const TileInfo t = gemm::tile_info_search(s, groups, ntiles, tile);
        s.tile_tab[k] = make_uint2(static_cast<uint32_t>(t.g) | (static_cast<uint32_t>(t.nt) << 11) |
                                       (static_cast<uint32_t>(t.m_valid) << 19),
                                   static_cast<uint32_t>(t.row0));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;
    const int nbn = p.N / 128;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
      if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x, k = 0; tile < total && !*abort; tile += gridDim.x, ++k) {
                const TileInfo t = gemm::tile_info(s, groups, ntiles, k, tile);
                const int brow = t.g * p.N + t.nt * BN;
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs)) break;
                    mbar_expect_tx(&s.full[st], STAGE_BYTES);
                    tma_load_2d(sA + st * A_BYTES, &tmA, &s.full[st], kc * BK, t.row0);
                    tma_load_2d(sB + st * B_BYTES, &tmB, &s.full[st], kc * BK, brow);
                }
            }
            if (*abort) {
                // let every issued copy land before the CTA exits
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer ----
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x, ++tc) {
                // the epilogue has read out the previous tile
                if (!mbar_wait(&s.tempty, (tc & 1u) ^ 1u, abort, kWaitLimitNs)) break;
                tc_fence_after();
                bool ok = true;
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(&s.full[st], ph, abort, kWaitLimitNs)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sft = tmem + SF_TMEM_COL + st * 12;
                    const uint32_t sfs = smem_addr(&s.sf[st][0]);
                    tc_cp_sf(sft, sf_desc(sfs));               // A's scales: columns 0-3
                    tc_cp_sf(sft + 4, sf_desc(sfs + 512));     // B's scales: columns 0-3 ...
                    tc_cp_sf(sft + 8, sf_desc(sfs + 1024));    // ... and 4-7
                    const uint64_t ad = sw128_desc(smem_addr(sA + st * A_BYTES));
                    const uint64_t bd = sw128_desc(smem_addr(sB + st * B_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_mx(tmem, ad + 2 * k, bd + 2 * k, IDESC_MX, sft, sft + 4, (kc > 0 || k > 0) ? 1u : 0u);
                    tc_commit(&s.empty[st]);
                }
                if (!ok) break;
                tc_commit(&s.tfull);
            }
            // no MMA may be in flight when TMEM is released
            tc_commit(&s.mma_done);
            mbar_wait(&s.mma_done, 0, nullptr, kWaitLimitNs);
        }
      } else {
        // -------------------------------------------------- scale staging ----
        // Thread t64 (0..63) writes A's scale words for tile rows t64 and t64 + 64 and the
        // B words of lane t64 % 32 of B block t64 / 32 (columns 4 (t64 / 32) .. + 3).
        const int t64 = (warp - 2) * 32 + static_cast<int>(lane);
        const bool vec = (nkc % 4) == 0 && (reinterpret_cast<uintptr_t>(p.sa) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.sb) & 15u) == 0;
        const int ngrp = (nkc + 3) / 4;
        // loads the four-chunk group `grp` of the k-th tile of this CTA
        bool bad = false, ok = true;
        auto load_group = [&](int k, int tile, int grp, ScaleGroup& sg) {
            const TileInfo t = gemm::tile_info(s, groups, ntiles, k, tile);
            const int64_t r0 = t64 < t.m_valid ? static_cast<int64_t>(t.row0) + t64 : 0;
            const int64_t r1 = t64 + 64 < t.m_valid ? static_cast<int64_t>(t.row0) + t64 + 64 : 0;
            const float* a0 = p.sa + r0 * nkc + grp * 4;
            const float* a1 = p.sa + r1 * nkc + grp * 4;
            const float* b0 = p.sb + (static_cast<int64_t>(t.g) * nbn + 2 * t.nt) * nkc + grp * 4;
            const float* b1 = b0 + nkc;
            if (vec) {
                const float4 va0 = __ldg(reinterpret_cast<const float4*>(a0));
                const float4 va1 = __ldg(reinterpret_cast<const float4*>(a1));
                const float4 vb0 = __ldg(reinterpret_cast<const float4*>(b0));
                const float4 vb1 = __ldg(reinterpret_cast<const float4*>(b1));
                sg.a0 = ue8m0_x4(va0.x, va0.y, va0.z, va0.w, bad);
                sg.a1 = ue8m0_x4(va1.x, va1.y, va1.z, va1.w, bad);
                sg.b0 = ue8m0_x4(vb0.x, vb0.y, vb0.z, vb0.w, bad);
                sg.b1 = ue8m0_x4(vb1.x, vb1.y, vb1.z, vb1.w, bad);
            } else {
                sg.a0 = sg.a1 = sg.b0 = sg.b1 = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (grp * 4 + c < nkc) {
                        sg.a0 |= ue8m0(__ldg(a0 + c), bad) << (8 * c);
                        sg.a1 |= ue8m0(__ldg(a1 + c), bad) << (8 * c);
                        sg.b0 |= ue8m0(__ldg(b0 + c), bad) << (8 * c);
                        sg.b1 |= ue8m0(__ldg(b1 + c), bad) << (8 * c);
                    }
                }
            }
        };
        // position of the next group to load: (k-th tile, group)
        int nk = 0, ntile = blockIdx.x, ngr = 0;
        auto advance = [&]() {
            if (++ngr == ngrp) { ngr = 0; ++nk; ntile += gridDim.x; }
        };
        ScaleGroup cur{0, 0, 0, 0}, nxt{0, 0, 0, 0};
        if (ntile < total) { load_group(nk, ntile, ngr, nxt); advance(); }
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            for (int kc = 0; kc < nkc; ++kc, ++it) {
                const int c = kc & 3;
                if (c == 0) {
                    cur = nxt;
                    if (ntile < total) { load_group(nk, ntile, ngr, nxt); advance(); }
                }
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs))) {
                    ok = false;
                    break;
                }
                uint32_t* sf = s.sf[st];
                // A: row r at word 4 (r % 32) + r / 32
                sf[4 * (t64 & 31) + (t64 >> 5)] = code_word(cur.a0, c);
                sf[4 * (t64 & 31) + ((t64 + 64) >> 5)] = code_word(cur.a1, c);
                // B: column j covers tile columns 32j .. 32j+31. SwiGLU tiles interleave
                // gate / up rows in 64-row blocks (columns 0,1,4,5: gate block; 2,3,6,7: up);
                // otherwise columns 0-3 use block 2 nt, columns 4-7 block 2 nt + 1
                const uint32_t wb0 = code_word(cur.b0, c), wb1 = code_word(cur.b1, c);
                const int blk = t64 >> 5;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = 4 * blk + j;
                    const bool second = (EPI == MOE_EPI_SWIGLU_FP8) ? ((col >> 1) & 1) != 0 : col >= 4;
                    sf[128 + 128 * blk + 4 * (t64 & 31) + j] = second ? wb1 : wb0;
                }
                // the words are read by tcgen05.cp (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.full[st]);
            }
        }
        if (bad) set_status(MOE_ERR_DEVICE_CHECK);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
        // -------------------------------------------------------- epilogue ----
        const int ew = warp - 4;             // 0..7
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int half = ew >> 2;            // column half of the 256-wide tile
        const int rit = q * 32 + static_cast<int>(lane);
        const int last_start = s.row_start[groups - 1];
        uint32_t tcount = 0;
        for (int tile = blockIdx.x, k = 0; tile < total; tile += gridDim.x, ++k, ++tcount) {
            const TileInfo t = gemm::tile_info(s, groups, ntiles, k, tile);
            if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull, tcount & 1u, abort, kWaitLimitNs))) break;
            tc_fence_after();
            float acc[128];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * 128;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint32_t v[32];
                tmem_ld32(taddr + r * 32, v);
                tmem_ld_wait();
                tmem_reg_fence(v);
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[r * 32 + i] = __uint_as_float(v[i]);
            }
            // the accumulator is free for the next tile's MMAs
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty);
            if (!gemm::store_tile<EPI, true>(acc, p, s, t, groups, last_start, rit, half, ew, q, lane, tcount, abort))
                break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace gemm_mx
}  // namespace moe
