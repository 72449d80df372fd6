// Grouped FP8 GEMM with fine-grained scales on the 5th-generation tensor
// cores ("DeepSeek-V3的MoE架构设计革新" §2 FP8 training: activations scaled per
// 1x128 tile, weights per 128x128 block, partial sums promoted to FP32 at
// every 128-element K chunk).
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: A tile 128x128 and B tile 256x128 (E4M3,
//               128-byte swizzle) per K chunk into a 4-stage ring.
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=32) per chunk
//               into one of two TMEM chunk accumulators (2 x 256 columns).
//   warps 2,3   idle (they complete the first warpgroup, which gives its
//               registers to the epilogue warpgroups via setmaxnreg)
//   warps 4..11 epilogue: per chunk, tcgen05.ld the 128x256 FP32 partial,
//               multiply by sa[row][kc] * sb[group][n/128][kc] and add to
//               the FP32 tile accumulator kept in registers (128 values per
//               thread: lane quadrant = warp % 4, column half = (warp-4)/4).
//               After the last chunk: bf16 store, or SwiGLU + 1x128 E4M3
//               requantisation of h.
// The chunk accumulator is released as soon as its last TMEM load lands
// (before the second half of the promotion FMAs), so the tensor cores run up
// to two chunks ahead of the promotion arithmetic; the release barriers are
// indexed by chunk position mod 4, so the issuer of chunk c waits on exactly
// the release of chunk c - 2. The chunk scales reach the epilogue either from
// registers (activation scales, 16-byte loads a group of four chunks ahead)
// and a per-warp shared row of the tile's weight scales staged once per tile
// (VSC), or through a per-chunk shared-memory ring; both form the same
// products.
//
// Tiles: for each group, ceil(m_g / 128) row tiles x N/256 column tiles,
// numbered group by group with the column tile fastest; CTA c takes tiles
// c, c + gridDim.x, ... A rows past a group's end belong to the next group
// (or are TMA zero fill past the last row); their results are never stored.
#pragma once

#include "common.cuh"

namespace moe {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
static_assert(BM == 32 * 4, "gather mode: one gather4 (four rows) per producer lane");
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 384;
// Register split: launch budget 384 x 168 = 64512. The producer warpgroup
// drops to 40 per thread (128 x 40 = 5120), the two epilogue warpgroups
// rise to 232 (256 x 232 = 59392); 5120 + 59392 = 64512.
constexpr uint32_t kRegsProducer = 40;
constexpr uint32_t kRegsEpilogue = 232;
constexpr int MAX_GROUPS = 1025;
constexpr int TILE_TAB = 1024;          // tiles per CTA decoded in the prologue (later ones: binary search)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = make_idesc(BM, BN, 0);


struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[4];               // chunk it's TMEM buffer read out (index it % 4, one arrive per epilogue warp)
    uint64_t mma_done;
    uint64_t pair[4];                 // SwiGLU amax exchange between the two warps of a lane quadrant
    uint32_t tmem_base;
    int abort;
    int bad;
    int mtiles_total;
    int row_start[MAX_GROUPS + 1];    // offsets[g]
    int mtile_prefix[MAX_GROUPS + 1]; // exclusive prefix of ceil(m_g / BM)
    float amax_x[2][8][32];
    uint2 tile_tab[TILE_TAB];         // this CTA's tiles in order: {g | nt << 11 | min(m_valid,128) << 19, row0}
    alignas(16) float ring_sa[4][256];  // per-thread activation scale of chunks kc .. kc+3; VSC: per-warp weight scales
    float ring_sb[4][8][2];           // per-warp weight scales (two 128-column blocks)
};

constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "more shared memory than a CTA may have");

// The all-FP32 epilogues (the backward pass's data-gradient and recomputation GEMMs) send
// their tiles out through shared memory by TMA stores: per epilogue warp two 2 KB boxes of
// 32 rows x 16 FP32 (64-byte swizzle), which takes a 3-stage operand ring to fit.
constexpr int OUT_BOX_COLS = 16;
constexpr int OUT_BOX_BYTES = 32 * OUT_BOX_COLS * 4;
constexpr int OUT_STAGE_BYTES = 8 * 2 * OUT_BOX_BYTES;
template <int EPI>
struct EpiCfg {
    static constexpr bool kTmaOut = EPI == MOE_EPI_F32 || EPI == MOE_EPI_GATEUP_F32;
    static constexpr int kStages = kTmaOut ? 3 : STAGES;
    static constexpr int kOutBytes = kTmaOut ? OUT_STAGE_BYTES : 0;
    static constexpr size_t kSmem = 1024 + kStages * STAGE_BYTES + kOutBytes + sizeof(Smem);
};
static_assert(EpiCfg<MOE_EPI_F32>::kSmem <= 227 * 1024, "more shared memory than a CTA may have");

struct Params {
    const int32_t* offsets;
    int32_t groups;
    int64_t rows;
    int32_t N;
    int32_t Kdim;
    const float* sa;
    const float* sb;
    void* out;
    float* out_aux;      // SwiGLU: h scales; BF16_F32_LAST: FP32 output of the last group
    const int32_t* row_index;   // gather mode: grouped row r reads A and sa row row_index[r]
    int64_t a_rows;             // gather mode: rows of A
};

// tile -> (group, row tile inside the group, column tile)
template <typename SmemT>
__device__ __forceinline__ void decode_tile(const SmemT& s, int groups, int ntiles, int tile, int& g, int& mt, int& nt) {
    const int mtg = tile / ntiles;
    nt = tile - mtg * ntiles;
    int lo = 0, hi = groups - 1;           // last g with mtile_prefix[g] <= mtg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.mtile_prefix[mid] <= mtg) lo = mid; else hi = mid - 1;
    }
    g = lo;
    mt = mtg - s.mtile_prefix[g];
}

// One tile's place: group, column tile, first grouped row, and valid rows
// (m_valid, clipped to BM).
struct TileInfo {
    int g, nt, row0, m_valid;
};

template <typename SmemT>
__device__ __forceinline__ TileInfo tile_info_search(const SmemT& s, int groups, int ntiles, int tile) {
    int g, mt, nt;
    decode_tile(s, groups, ntiles, tile, g, mt, nt);
    const int row0 = s.row_start[g] + mt * BM;
    return TileInfo{g, nt, row0, min(s.row_start[g + 1] - row0, BM)};
}

// k-th tile of this CTA (tile = blockIdx.x + k * gridDim.x): one shared-memory
// load from the prologue's table (a binary search over the group prefix would
// be nine dependent loads, slow while TMA and the tensor cores keep shared
// memory busy)
template <typename SmemT>
__device__ __forceinline__ TileInfo tile_info(const SmemT& s, int groups, int ntiles, int k, int tile) {
    if (k < TILE_TAB) {
        const uint2 e = s.tile_tab[k];
        return TileInfo{static_cast<int>(e.x & 2047u), static_cast<int>((e.x >> 11) & 255u), static_cast<int>(e.y),
                        static_cast<int>(e.x >> 19)};
    }
    return tile_info_search(s, groups, ntiles, tile);
}

// The finished FP32 tile accumulator of this thread (row `rit` of the tile, 128 columns
// of column half `half`) to the output: FP32 rows, bf16 rows, or SwiGLU + 1x128 E4M3
// requantisation of h (scale rule POW2 or FP32). Returns false if the amax exchange with
// the partner warp timed out.
template <int EPI, bool POW2, typename SmemT>
__device__ __forceinline__ bool store_tile(float* acc, const Params& p, SmemT& s, const TileInfo& t, int groups,
                                           int last_start, int rit, int half, int ew, int q, uint32_t lane,
                                           uint32_t tcount, volatile int* abort) {
    const int g = t.g, nt = t.nt;
    const bool valid = rit < t.m_valid;
    const int64_t row = static_cast<int64_t>(t.row0) + rit;
        const bool f32_out = (EPI == MOE_EPI_F32) || (EPI == MOE_EPI_GATEUP_F32) ||
                             (EPI == MOE_EPI_BF16_F32_LAST && g == groups - 1);
        if (f32_out) {
            if (valid) {
                float* dst = (EPI != MOE_EPI_BF16_F32_LAST)
                                 ? static_cast<float*>(p.out) + row * p.N + nt * BN + half * 128
                                 : p.out_aux + (row - last_start) * p.N + nt * BN + half * 128;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    st_v8_b32(dst + 8 * i, __float_as_uint(acc[8 * i]), __float_as_uint(acc[8 * i + 1]),
                              __float_as_uint(acc[8 * i + 2]), __float_as_uint(acc[8 * i + 3]),
                              __float_as_uint(acc[8 * i + 4]), __float_as_uint(acc[8 * i + 5]),
                              __float_as_uint(acc[8 * i + 6]), __float_as_uint(acc[8 * i + 7]));
            }
        } else if (EPI == MOE_EPI_BF16 || EPI == MOE_EPI_BF16_F32_LAST) {
            if (valid) {
                uint16_t* dst = static_cast<uint16_t*>(p.out) + row * p.N + nt * BN + half * 128;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_v8_b32(dst + 16 * i, pack_bf16x2(acc[16 * i + 0], acc[16 * i + 1]),
                              pack_bf16x2(acc[16 * i + 2], acc[16 * i + 3]),
                              pack_bf16x2(acc[16 * i + 4], acc[16 * i + 5]),
                              pack_bf16x2(acc[16 * i + 6], acc[16 * i + 7]),
                              pack_bf16x2(acc[16 * i + 8], acc[16 * i + 9]),
                              pack_bf16x2(acc[16 * i + 10], acc[16 * i + 11]),
                              pack_bf16x2(acc[16 * i + 12], acc[16 * i + 13]),
                              pack_bf16x2(acc[16 * i + 14], acc[16 * i + 15]));
            }
        } else {
            // h = SiLU(gate) * up for this thread's 64 columns; gate in acc[0,64), up in acc[64,128)
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float gte = acc[c];
                const float h = __fdividef(gte * acc[64 + c], 1.0f + __expf(-gte));
                acc[c] = h;
                amax = fmaxf(amax, fabsf(h));
            }
            // the partner warp (same quadrant, other half) holds the other 64 columns
            s.amax_x[tcount & 1u][ew][lane] = amax;
            mbar_arrive(&s.pair[q]);
            if (!__all_sync(0xffffffffu, mbar_wait(&s.pair[q], tcount & 1u, abort, kWaitLimitNs))) return false;
            amax = fmaxf(amax, s.amax_x[tcount & 1u][ew ^ 4][lane]);
            const float sc = tile_scale<POW2>(amax);
            // h is multiplied by the correctly rounded reciprocal of the scale (exact for
            // a power of two; otherwise one rounding more than the quotient, enough for an
            // E4M3 code)
            const float rs = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
            if (valid) {
                const int I = p.N / 2;
                uint8_t* dst = static_cast<uint8_t*>(p.out) + row * I + nt * 128 + half * 64;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 w;
                    w.x = e4m3x4(rs * acc[16 * i + 0], rs * acc[16 * i + 1],
                                 rs * acc[16 * i + 2], rs * acc[16 * i + 3]);
                    w.y = e4m3x4(rs * acc[16 * i + 4], rs * acc[16 * i + 5],
                                 rs * acc[16 * i + 6], rs * acc[16 * i + 7]);
                    w.z = e4m3x4(rs * acc[16 * i + 8], rs * acc[16 * i + 9],
                                 rs * acc[16 * i + 10], rs * acc[16 * i + 11]);
                    w.w = e4m3x4(rs * acc[16 * i + 12], rs * acc[16 * i + 13],
                                 rs * acc[16 * i + 14], rs * acc[16 * i + 15]);
                    reinterpret_cast<uint4*>(dst)[i] = w;
                }
                if (half == 0) p.out_aux[row * (I / 128) + nt] = sc;
            }
        }
    return true;
}

// The finished FP32 tile accumulator of this thread (row rit of the tile, 128 columns of
// column half `half`) to the FP32 output through shared memory: the warp's 32 rows go out
// as 8 TMA boxes of 32 rows x 16 columns, written into one of the warp's two staging
// buffers in the 64-byte swizzled layout (16-byte chunk c of row r at chunk c ^ ((r/2) % 4),
// which spreads a quarter warp over all banks). A buffer is rewritten only after the store
// issued two boxes earlier has read it. A warp whose 32 rows are not all in the tile's
// group stores its valid rows directly (a box would overwrite the next group's rows).
__device__ __forceinline__ void store_tile_tma(const float* acc, const Params& p, const CUtensorMap* tmOut,
                                               uint8_t* sOut, const TileInfo& t, int rit, int half, int ew, int q,
                                               uint32_t lane, uint32_t& nbox) {
    const int64_t row0 = static_cast<int64_t>(t.row0) + q * 32;
    const int col0 = t.nt * BN + half * 128;
    if (q * 32 + 32 > t.m_valid) {                       // warp-uniform
        if (rit < t.m_valid) {
            float* dst = static_cast<float*>(p.out) + (row0 + lane) * p.N + col0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                st_v8_b32(dst + 8 * i, __float_as_uint(acc[8 * i]), __float_as_uint(acc[8 * i + 1]),
                          __float_as_uint(acc[8 * i + 2]), __float_as_uint(acc[8 * i + 3]),
                          __float_as_uint(acc[8 * i + 4]), __float_as_uint(acc[8 * i + 5]),
                          __float_as_uint(acc[8 * i + 6]), __float_as_uint(acc[8 * i + 7]));
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 128 / OUT_BOX_COLS; ++j, ++nbox) {
        uint8_t* buf = sOut + (ew * 2 + (nbox & 1u)) * OUT_BOX_BYTES;
        if (nbox >= 2) {
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
        }
        const uint32_t row = smem_addr(buf) + lane * (OUT_BOX_COLS * 4);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            st_shared_v4(row + ((c ^ ((lane >> 1) & 3u)) << 4), acc[16 * j + 4 * c], acc[16 * j + 4 * c + 1],
                         acc[16 * j + 4 * c + 2], acc[16 * j + 4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmOut, buf, col0 + OUT_BOX_COLS * j, static_cast<int32_t>(row0));
            bulk_commit();
        }
    }
}

// GATHER: A rows are fetched by index (TMA gather4, four rows per copy)
// instead of as one 128-row tile.
// VSC: the activation scales go straight from global memory into registers and a tile's
// weight scales are staged once per tile (Kdim / 128 a multiple of 4 and at most 64, sa
// and sb 16-byte aligned) instead of streaming both through the per-chunk shared-memory
// ring.
template <int EPI, bool GATHER, bool VSC>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, Params p) {
    constexpr int STAGES = EpiCfg<EPI>::kStages;     // operand ring of this epilogue
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + STAGES * A_BYTES;
    uint8_t* sOut = base + STAGES * STAGE_BYTES;     // TMA-store staging (all-FP32 epilogues)
    Smem& s = *reinterpret_cast<Smem*>(sOut + EpiCfg<EPI>::kOutBytes);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const int groups = p.groups;
    const int ntiles = p.N / BN;
    const int nkc = p.Kdim / BK;

    // ---- set-up: barriers, TMEM, per-group row tiles -------------------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
        for (int i = 0; i < 2; ++i) mbar_init(&s.tfull[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&s.tempty[i], 8);
        mbar_init(&s.mma_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&s.pair[i], 64);
        s.abort = 0;
        s.bad = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (EpiCfg<EPI>::kTmaOut) tma_prefetch_desc(&tmOut);
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
        const TileInfo t = tile_info_search(s, groups, ntiles, tile);
        s.tile_tab[k] = make_uint2(static_cast<uint32_t>(t.g) | (static_cast<uint32_t>(t.nt) << 11) |
                                       (static_cast<uint32_t>(t.m_valid) << 19),
                                   static_cast<uint32_t>(t.row0));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
      if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        // Lane 0 waits for a free stage and arms its barrier; in gather mode
        // every lane then issues one gather4 (rows 4*lane .. 4*lane+3 of the
        // tile, indices held in registers for the whole tile).
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x, k = 0; tile < total; tile += gridDim.x, ++k) {
            const TileInfo t = tile_info(s, groups, ntiles, k, tile);
            const int row0 = t.row0;
            const int brow = t.g * p.N + t.nt * BN;
            int src[4] = {0, 0, 0, 0};
            if (GATHER) {
                // rows past the group's end read row 0 (their results are dropped)
                const int end = row0 + t.m_valid;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = row0 + 4 * static_cast<int>(lane) + q;
                    int v = r < end ? __ldg(p.row_index + r) : 0;
                    if (v < 0 || v >= p.a_rows) { set_status(MOE_ERR_DEVICE_CHECK); v = 0; }
                    src[q] = v;
                }
            }
            for (int kc = 0; kc < nkc; ++kc, ++it) {
                const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                if (lane == 0) {
                    ok = mbar_wait(&s.empty[st], ph ^ 1u, abort, kWaitLimitNs);
                    if (ok) mbar_expect_tx(&s.full[st], STAGE_BYTES);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
                if (GATHER)
                    tma_gather4_2d(sA + st * A_BYTES + lane * 4 * BK, &tmA, &s.full[st], kc * BK, src[0], src[1],
                                   src[2], src[3]);
                else if (lane == 0)
                    tma_load_2d(sA + st * A_BYTES, &tmA, &s.full[st], kc * BK, row0);
                if (lane == 0) tma_load_2d(sB + st * B_BYTES, &tmB, &s.full[st], kc * BK, brow);
            }
            if (!ok || __shfl_sync(0xffffffffu, *abort, 0)) break;
        }
        if (lane == 0 && *abort) {
            // let every issued copy land before the CTA exits
            const uint32_t first = it > STAGES ? it - STAGES : 0;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait(&s.full[j % STAGES], (j / STAGES) & 1u, nullptr, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer ----
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it & 1u;
                    // buffer b is free once chunk it - 2 has been read out
                    if (it >= 2 && !mbar_wait(&s.tempty[(it - 2) & 3u], ((it - 2) >> 2) & 1u, abort, kWaitLimitNs))
                        break;
                    if (!mbar_wait(&s.full[st], ph, abort, kWaitLimitNs)) break;
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_addr(sA + st * A_BYTES));
                    const uint64_t bd = sw128_desc(smem_addr(sB + st * B_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_e4m3(tmem + b * BN, ad + 2 * k, bd + 2 * k, IDESC, k > 0 ? 1u : 0u);
                    tc_commit(&s.empty[st]);
                    tc_commit(&s.tfull[b]);
                }
            }
            // no MMA may be in flight when TMEM is released
            tc_commit(&s.mma_done);
            mbar_wait(&s.mma_done, 0, nullptr, kWaitLimitNs);
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
        // -------------------------------------------------------- epilogue ----
        const int ew = warp - 4;             // 0..7
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int half = ew >> 2;            // column half of the 256-wide tile
        const int rit = q * 32 + static_cast<int>(lane);
        const int et = ew * 32 + static_cast<int>(lane);
        const int nbn = p.N / 128;
        // Chunk scales stream through a 4-slot shared-memory ring indexed by the chunk's
        // position `it` in this CTA's sequence of chunks, copied (cp.async) three positions
        // ahead. The look-ahead continues into the next tile, so a tile's first scales are in
        // flight while the previous tile finishes; with fewer than three K chunks it would
        // have to skip tiles, so each tile then starts its own copies.
        struct ScaleRows { uint32_t sa; uint32_t sb; };   // element offsets of a tile's scale rows
        constexpr bool kSwigluLayout = EPI == MOE_EPI_SWIGLU_FP8 || EPI == MOE_EPI_GATEUP_F32;
        auto scale_rows = [&](const TileInfo& t) {
            const int g = t.g, nt = t.nt;
            int64_t src_row = rit < t.m_valid ? static_cast<int64_t>(t.row0) + rit : 0;
            if (GATHER && rit < t.m_valid) {
                src_row = __ldg(p.row_index + src_row);
                if (src_row < 0 || src_row >= p.a_rows) src_row = 0;      // reported by the producer
            }
            // weight scale rows: SwiGLU layout -> gate block 2*nt (up block 2*nt+1 is nkc further on);
            // otherwise block 2*nt+half. Offsets stay below 2^32 (checked at launch).
            const int64_t sb0 = (static_cast<int64_t>(g) * nbn + 2 * nt + (kSwigluLayout ? 0 : half)) * nkc;
            return ScaleRows{static_cast<uint32_t>(src_row * nkc), static_cast<uint32_t>(sb0)};
        };
        // copies the scales of K chunk kc of the tile at `rows` into ring slot `slot`, as one group
        auto copy_scales = [&](const ScaleRows& rows, int kc, uint32_t slot) {
            cp_async_4(&s.ring_sa[slot][et], p.sa + rows.sa + kc);
            if (lane == 0) {
                cp_async_4(&s.ring_sb[slot][ew][0], p.sb + rows.sb + kc);
                cp_async_4(&s.ring_sb[slot][ew][1], p.sb + rows.sb + (kSwigluLayout ? nkc : 0) + kc);
            }
        };
        // tells the MMA issuer that chunk position `it` has been read out of its TMEM buffer,
        // once this warp's loads from it have completed (before the last half of the promotion
        // arithmetic, which runs on registers)
        auto release = [&](uint32_t it_done) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty[it_done & 3u]);
        };
        // VSC: the activation scales of this thread's row for K chunks 4j .. 4j+3 are one
        // 16-byte load, issued one group of four chunks ahead (into the next tile at a tile's
        // last group). A tile's weight scales (the warp's gate-block and up-block rows) are
        // copied once per tile into a per-warp shared-memory row, while the previous tile is
        // stored: SwiGLU layout interleaved, one 8-byte broadcast load per chunk; otherwise
        // one 16-byte load per four chunks, a group ahead. Each per-chunk shared or shuffle
        // instruction costs the epilogue warps beside the TMA and MMA warps about 40 cycles a
        // chunk, so the number of such reads is what was minimised (per-chunk copies through the
        // ring, shuffles from lane-held rows, separate gate and up loads, 16-byte register
        // loads of the weight scales and, for the SwiGLU layout, 16-byte loads a pair of
        // chunks ahead all measured slower).
        auto a_row = [&](const TileInfo& t) -> const float* {
            int64_t src_row = rit < t.m_valid ? static_cast<int64_t>(t.row0) + rit : 0;
            if (GATHER && rit < t.m_valid) {
                src_row = __ldg(p.row_index + src_row);
                if (src_row < 0 || src_row >= p.a_rows) src_row = 0;      // reported by the producer
            }
            return p.sa + src_row * nkc;
        };
        // this warp's weight scales of the tile: SwiGLU layout (gate, up) of chunk kc at
        // [2 kc, 2 kc + 1]; otherwise chunk kc at [kc]
        float* wsb = &s.ring_sa[0][0] + ew * 128;
        auto load_wscales = [&](const TileInfo& t) {
            const float* g0 = p.sb + (static_cast<int64_t>(t.g) * nbn + 2 * t.nt + (kSwigluLayout ? 0 : half)) * nkc;
            const int l = static_cast<int>(lane);
            __syncwarp();
            if (kSwigluLayout) {
                for (int e = l; e < 2 * nkc; e += 32) cp_async_4(wsb + e, g0 + (e & 1) * nkc + (e >> 1));
            } else if (4 * l < nkc) {
                cp_async_16(wsb + 4 * l, g0 + 4 * l);
            }
            cp_async_commit();
        };
        float4 a_cur = make_float4(0.0f, 0.0f, 0.0f, 0.0f), a_nxt = a_cur;
        const float* arow_carry = p.sa;
        // (the all-FP32 store epilogue keeps per-tile copies: the look-ahead state makes it spill)
        const bool ahead = !VSC && EPI != MOE_EPI_F32 && EPI != MOE_EPI_GATEUP_F32 && nkc >= 3;
        uint32_t it = 0, tcount = 0, nbox = 0;
        bool ok = true;
        ScaleRows cur{0, 0}, nxt{0, 0};
        if (ahead && static_cast<int>(blockIdx.x) < total) {
            cur = scale_rows(tile_info(s, groups, ntiles, 0, blockIdx.x));
            for (int j = 0; j < 3; ++j) {
                copy_scales(cur, j, static_cast<uint32_t>(j));
                cp_async_commit();
            }
        }
        // the first row of the last group (FP32 output rows of MOE_EPI_BF16_F32_LAST count from it)
        const int last_start = s.row_start[groups - 1];
        TileInfo tnext = static_cast<int>(blockIdx.x) < total ? tile_info(s, groups, ntiles, 0, blockIdx.x)
                                                              : TileInfo{0, 0, 0, 0};
        if (VSC && static_cast<int>(blockIdx.x) < total) {
            arow_carry = a_row(tnext);
            a_nxt = __ldg(reinterpret_cast<const float4*>(arow_carry));
            load_wscales(tnext);
        }
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tcount) {
            const TileInfo t = tnext;
            const int g = t.g, nt = t.nt;
            const bool valid = rit < t.m_valid;
            const int64_t row = static_cast<int64_t>(t.row0) + rit;
            const int next = tile + static_cast<int>(gridDim.x);
            const bool has_next = next < total;
            if (has_next) tnext = tile_info(s, groups, ntiles, static_cast<int>(tcount) + 1, next);
            const float* arow = arow_carry;                       // VSC: this tile's activation scales
            const float* arow_next = arow;
            if (VSC && has_next) arow_next = a_row(tnext);
            if (!VSC && !ahead) {
                cur = scale_rows(t);
                for (int j = 0; j < 3; ++j) {
                    if (j < nkc) copy_scales(cur, j, (it + j) & 3u);
                    cp_async_commit();
                }
            }
            if (ahead && has_next) nxt = scale_rows(tnext);
            float2 acc2[64];             // FP32 tile accumulator, column pairs
#pragma unroll
            for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.0f, 0.0f);
            float4 wcur = make_float4(0.0f, 0.0f, 0.0f, 0.0f), wnxt = wcur;
            if (VSC) {
                cp_async_wait<0>();      // this tile's weight scales
                __syncwarp();
                if (!kSwigluLayout) wnxt = *reinterpret_cast<const float4*>(wsb);
            }
            for (int kc = 0; kc < nkc; ++kc, ++it) {
                const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
                float f0, f1;
                if constexpr (VSC) {
                    if ((kc & 3) == 0) {
                        a_cur = a_nxt;
                        const float* src = kc + 4 < nkc ? arow + kc + 4 : arow_next;
                        a_nxt = __ldg(reinterpret_cast<const float4*>(src));
                    }
                    const int j = kc & 3;
                    const float sav = j == 0 ? a_cur.x : j == 1 ? a_cur.y : j == 2 ? a_cur.z : a_cur.w;
                    if (kSwigluLayout) {          // (gate, up) of this chunk in one 8-byte load
                        const float2 w = *reinterpret_cast<const float2*>(wsb + 2 * kc);
                        f0 = sav * w.x;
                        f1 = sav * w.y;
                    } else {                      // chunks kc .. kc + 3 in one 16-byte load, a group ahead
                        if (j == 0) {
                            wcur = wnxt;
                            if (kc + 4 < nkc) wnxt = *reinterpret_cast<const float4*>(wsb + kc + 4);
                        }
                        f0 = sav * (j == 0 ? wcur.x : j == 1 ? wcur.y : j == 2 ? wcur.z : wcur.w);
                        f1 = f0;
                    }
                } else {
                    cp_async_wait<2>();      // this position's copies were the oldest of three groups
                    __syncwarp();
                    const uint32_t slot = it & 3u;
                    const float sav = s.ring_sa[slot][et];
                    f0 = sav * s.ring_sb[slot][ew][0];
                    f1 = sav * s.ring_sb[slot][ew][1];
                    // three positions ahead: this tile, else (look-ahead) the next one
                    const int k3 = kc + 3;
                    if (k3 < nkc)
                        copy_scales(cur, k3, (it + 3) & 3u);
                    else if (ahead && has_next)
                        copy_scales(nxt, k3 - nkc, (it + 3) & 3u);
                    cp_async_commit();
                }
                // warp-uniform outcome: every lane leaves together (warp syncs follow)
                if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[b], bph, abort, kWaitLimitNs))) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * BN + half * 128;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(taddr + r * 64, v0);
                    tmem_ld32(taddr + r * 64 + 32, v1);
                    tmem_ld_wait();
                    tmem_reg_fence(v0);
                    tmem_reg_fence(v1);
                    if (r == 1) release(it);   // every value of the chunk is in registers now
                    const float2 ff = make_float2((r == 0) ? f0 : f1, (r == 0) ? f0 : f1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        acc2[r * 32 + i] = __ffma2_rn(make_float2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1])),
                                                      ff, acc2[r * 32 + i]);
                        acc2[r * 32 + 16 + i] = __ffma2_rn(make_float2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1])),
                                                           ff, acc2[r * 32 + 16 + i]);
                    }
                }
            }
            float* acc = reinterpret_cast<float*>(acc2);
            if (!ok) break;
            if (VSC && has_next) load_wscales(tnext);              // landed while the tile is stored
            arow_carry = arow_next;
            if constexpr (EpiCfg<EPI>::kTmaOut)
                store_tile_tma(acc, p, &tmOut, sOut, t, rit, half, ew, q, lane, nbox);
            else if (!store_tile<EPI, false>(acc, p, s, t, groups, last_start, rit, half, ew, q, lane, tcount, abort))
                break;
            cur = nxt;
        }
        cp_async_wait<0>();          // no scale copy may still target shared memory at exit
        if (EpiCfg<EPI>::kTmaOut) {  // every box store has read its buffer and landed
            if (lane == 0) bulk_wait<0>();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace moe
