// C ABI of the B300 DeepSeekMoE layer forward: argument checks, launch
// planning and kernel launches. Declarations and contracts: moe_b300.h.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "backward.cuh"
#include "common.cuh"
#include "ep.cuh"
#include "gemm_fp8.cuh"
#include "gemm_wgrad.cuh"
#include "gemm_mx.cuh"
#include "misc.cuh"
#include "permute.cuh"
#include "quant.cuh"
#include "route.cuh"
#include "route_tc.cuh"

namespace {

using namespace moe;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

moe_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status check_config(const moe_config* c) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->d < 128 || c->I < 128 || c->d % 128 || c->I % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->E < 16 || c->E > 1024 || c->E % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->G < 1 || c->G > 32 || c->E % c->G) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->M < 1 || c->M > c->G) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int n = c->E / c->G;
    if (c->gk < 1 || c->gk > n || c->gk > route::kMaxGK) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->K < 1 || c->K > 16 || c->K > c->M * n) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(c->T) * (c->K + 1) > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// Raises the dynamic shared-memory limit of kernel `fn` to `bytes` once per
// device: the attribute belongs to the device's context, so each device that
// launches the kernel needs its own call. `done` holds one bit per device
// ordinal (< 64); setting the attribute twice from racing threads is harmless.
moe_status smem_attr(const void* fn, size_t bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return MOE_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
        return MOE_ERR_CUDA;
    done.fetch_or(bit, std::memory_order_release);
    return MOE_OK;
}

// SM count of the current device (queried per call: a cheap attribute read,
// correct when a process drives devices of different sizes).
int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    return sms;
}

// Router geometry. A CTA accumulates sub-splits of rtc::kMaxChunksPerSplit
// chunks (the accuracy bound); its K slice is a run of sub-splits. Slices
// across CTAs exist only to fill the SMs when the token tiles x expert tiles
// leave them idle (at most rtc::kMaxSlices), each slice non-empty.
int route_nsub(const moe_config* c) {
    const int nchunks = 3 * (c->d / rtc::BK);
    return (nchunks + rtc::kMaxChunksPerSplit - 1) / rtc::kMaxChunksPerSplit;
}

int route_subs_per_slice(const moe_config* c, int slices) {
    return (route_nsub(c) + slices - 1) / slices;
}

int route_slices(const moe_config* c) {
    const int64_t ctas = ceil_div(c->T, rtc::BM) * ceil_div(c->E, rtc::BN_MAX);
    const int want = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(rtc::kMaxSlices, num_sms() / std::max<int64_t>(ctas, 1))));
    const int per = route_subs_per_slice(c, std::min(want, route_nsub(c)));
    return (route_nsub(c) + per - 1) / per;
}

// The fused router (selection inside the logits kernel) serves E <= 256 when
// its one CTA per 128-token tile covers at least half the SMs; smaller
// batches take the sliced logits kernel and the selection kernel, whose extra
// CTAs fill the GPU.
bool route_fused_auto(const moe_config* c) {
    return c->E <= rtc::BN_MAX && 2 * ceil_div(c->T, rtc::BM) >= num_sms();
}

// Workspace layout: [header: slice count of the stored router logits, i32,
// written by the router kernels][router logit slice sums f32 slices*T*E (the
// fused router stores the whole sums in the first T*E)][router weight planes bf16
// 3*E*d][per-block counts i32 nblk*E][per-block bases i32 nblk*E][offsets
// scratch i32 E+2][balance chunk sums f32, i32 (T/32)*E each]
struct WsLayout {
    size_t header, logits, planes, blk_counts, blk_base, offsets, balance, total;
};

WsLayout ws_layout(const moe_config* c) {
    WsLayout w{};
    const int64_t nblk = ceil_div(c->T, perm::kTokPerBlk);
    w.header = 0;
    w.logits = 256;
    w.planes = w.logits + align_up(static_cast<size_t>(route_slices(c)) * c->T * c->E * sizeof(float), 256);
    w.blk_counts = w.planes + align_up(static_cast<size_t>(3) * c->E * c->d * sizeof(uint16_t), 256);
    w.blk_base = w.blk_counts + align_up(static_cast<size_t>(nblk) * c->E * sizeof(int32_t), 256);
    w.offsets = w.blk_base + align_up(static_cast<size_t>(nblk) * c->E * sizeof(int32_t), 256);
    w.balance = w.offsets + align_up(static_cast<size_t>(c->E + 2) * sizeof(int32_t), 256);
    // balance statistics: per-32-token-chunk sums, f32 [T/32][E] then i32 [T/32][E]
    w.total = w.balance + 2 * align_up(static_cast<size_t>(ceil_div(c->T, 32)) * c->E * sizeof(float), 256);
    return w;
}

// ----------------------------------------------------------- tensor maps ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D K-major byte matrix [outer][inner], box [box_outer][128 bytes], 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D FP32 matrix [outer][inner] for TMA stores of boxes of 32 rows x box_cols elements:
// box_cols 32 (128 bytes, 128-byte swizzle) or 16 (64 bytes, 64-byte swizzle).
bool make_map_f32_box(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {box_cols, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D K-major bf16 matrix [outer][inner], box [box_outer][64 elements], 128-byte swizzle.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPL, int MAXGK>
void launch_select_t(const moe_config* c, const float* z, int ks, const float* off, const float* bias, int32_t* idx,
                     float* gate, int grid, size_t smem, cudaStream_t st) {
    route::select_kernel<EPL, MAXGK><<<grid, route::kSelWarps * 32, smem, st>>>(z, ks, c->T, c->E, c->G, c->M, c->K,
                                                                               c->gk, off, bias, idx, gate);
}

template <int EPL>
void launch_select_e(const moe_config* c, const float* z, int ks, const float* off, const float* bias, int32_t* idx,
                     float* gate, int grid, size_t smem, cudaStream_t st) {
    if (c->gk <= 2) launch_select_t<EPL, 2>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else if (c->gk <= 4) launch_select_t<EPL, 4>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else launch_select_t<EPL, route::kMaxGK>(c, z, ks, off, bias, idx, gate, grid, smem, st);
}

void launch_select(const moe_config* c, const float* z, int ks, const float* off, const float* bias, int32_t* idx,
                   float* gate, int grid, size_t smem, cudaStream_t st) {
    const int epl = (c->E + 31) / 32;
    if (epl <= 1) launch_select_e<1>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else if (epl <= 2) launch_select_e<2>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else if (epl <= 4) launch_select_e<4>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else if (epl <= 8) launch_select_e<8>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else if (epl <= 16) launch_select_e<16>(c, z, ks, off, bias, idx, gate, grid, smem, st);
    else launch_select_e<32>(c, z, ks, off, bias, idx, gate, grid, smem, st);
}

template <bool SELECT, int EPL, int MAXGK>
moe_status launch_route_t(const moe_config* c, const CUtensorMap& tx, const CUtensorMap& tw, int slices,
                          const float* off, const float* bias, int32_t* idx, float* gate, float* z, int* splits,
                          cudaStream_t st) {
    static std::atomic<uint64_t> attr_done{0};
    if (smem_attr(reinterpret_cast<const void*>(rtc::route_kernel<SELECT, EPL, MAXGK>), rtc::F_SMEM_BYTES,
                  attr_done) != MOE_OK)
        return MOE_ERR_CUDA;
    rtc::FParams fp{c->T, c->d, c->E, c->G, c->M, c->K, c->gk, route_subs_per_slice(c, slices),
                    off, bias, idx, gate, z, splits};
    const dim3 grid(static_cast<unsigned>(ceil_div(c->T, rtc::BM)),
                    SELECT ? 1u : static_cast<unsigned>(ceil_div(c->E, rtc::BN_MAX)), static_cast<unsigned>(slices));
    rtc::route_kernel<SELECT, EPL, MAXGK><<<grid, rtc::F_THREADS, rtc::F_SMEM_BYTES, st>>>(tx, tw, fp);
    return launch_status();
}

template <int EPL>
moe_status launch_fused_e(const moe_config* c, const CUtensorMap& tx, const CUtensorMap& tw, const float* off,
                          const float* bias, int32_t* idx, float* gate, float* z, int* splits, cudaStream_t st) {
    if (c->gk <= 2) return launch_route_t<true, EPL, 2>(c, tx, tw, 1, off, bias, idx, gate, z, splits, st);
    if (c->gk <= 4) return launch_route_t<true, EPL, 4>(c, tx, tw, 1, off, bias, idx, gate, z, splits, st);
    return launch_route_t<true, EPL, route::kMaxGK>(c, tx, tw, 1, off, bias, idx, gate, z, splits, st);
}

// The fused router: one K slice, selection in the kernel (E <= 256: at most 8 experts per lane).
moe_status launch_fused(const moe_config* c, const CUtensorMap& tx, const CUtensorMap& tw, const float* off,
                        const float* bias, int32_t* idx, float* gate, float* z, int* splits, cudaStream_t st) {
    const int epl = (c->E + 31) / 32;
    if (epl <= 1) return launch_fused_e<1>(c, tx, tw, off, bias, idx, gate, z, splits, st);
    if (epl <= 2) return launch_fused_e<2>(c, tx, tw, off, bias, idx, gate, z, splits, st);
    if (epl <= 4) return launch_fused_e<4>(c, tx, tw, off, bias, idx, gate, z, splits, st);
    return launch_fused_e<8>(c, tx, tw, off, bias, idx, gate, z, splits, st);
}

// to: the FP32 output's tensor map for the all-FP32 epilogues (unused by the others)
template <int EPI, bool GATHER, bool VSC>
moe_status launch_gemm_v(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const gemm::Params& p,
                         int64_t tiles_max, cudaStream_t st) {
    constexpr size_t smem = gemm::EpiCfg<EPI>::kSmem;
    static std::atomic<uint64_t> attr_done{0};
    const void* fn = reinterpret_cast<const void*>(gemm::grouped_gemm_fp8_kernel<EPI, GATHER, VSC>);
    if (smem_attr(fn, smem, attr_done) != MOE_OK) return MOE_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), std::max<int64_t>(tiles_max, 1)));
    gemm::grouped_gemm_fp8_kernel<EPI, GATHER, VSC><<<grid, gemm::NUM_THREADS, smem, st>>>(ta, tb, to, p);
    return launch_status();
}

// Chunk scales in registers (VSC) where the kernel supports it: K/128 a multiple of 4 and
// at most 64, 16-byte aligned scale arrays.
template <int EPI, bool GATHER>
moe_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const gemm::Params& p,
                       int64_t tiles_max, cudaStream_t st) {
    const int nkc = p.Kdim / gemm::BK;
    if (nkc % 4 == 0 && nkc <= 64 && aligned16(p.sa) && aligned16(p.sb))
        return launch_gemm_v<EPI, GATHER, true>(ta, tb, to, p, tiles_max, st);
    return launch_gemm_v<EPI, GATHER, false>(ta, tb, to, p, tiles_max, st);
}

template <bool GATHER>
moe_status launch_gemm_epi(int32_t epilogue, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                           const gemm::Params& p, int64_t tiles_max, cudaStream_t st) {
    if (epilogue == MOE_EPI_BF16) return launch_gemm<MOE_EPI_BF16, GATHER>(ta, tb, to, p, tiles_max, st);
    if (epilogue == MOE_EPI_F32) return launch_gemm<MOE_EPI_F32, GATHER>(ta, tb, to, p, tiles_max, st);
    if (epilogue == MOE_EPI_BF16_F32_LAST)
        return launch_gemm<MOE_EPI_BF16_F32_LAST, GATHER>(ta, tb, to, p, tiles_max, st);
    if (epilogue == MOE_EPI_GATEUP_F32) return launch_gemm<MOE_EPI_GATEUP_F32, GATHER>(ta, tb, to, p, tiles_max, st);
    return launch_gemm<MOE_EPI_SWIGLU_FP8, GATHER>(ta, tb, to, p, tiles_max, st);
}

template <int EPI>
moe_status launch_gemm_mx(const CUtensorMap& ta, const CUtensorMap& tb, const gemm::Params& p, int64_t tiles_max,
                          cudaStream_t st) {
    static std::atomic<uint64_t> attr_done{0};
    if (smem_attr(reinterpret_cast<const void*>(gemm_mx::grouped_gemm_mx_kernel<EPI>), gemm_mx::SMEM_BYTES,
                  attr_done) != MOE_OK)
        return MOE_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), std::max<int64_t>(tiles_max, 1)));
    gemm_mx::grouped_gemm_mx_kernel<EPI><<<grid, gemm::NUM_THREADS, gemm_mx::SMEM_BYTES, st>>>(ta, tb, p);
    return launch_status();
}

// Shared checks and launch of the grouped GEMM; row_index == nullptr: A is in grouped row order.
moe_status grouped_gemm(int32_t groups, const int32_t* offsets, int64_t rows, int32_t N, int32_t Kdim,
                        const uint8_t* A, const float* sa, int64_t a_rows, const int32_t* row_index,
                        const uint8_t* B, const float* sb, int32_t epilogue, void* out, float* out_aux,
                        cudaStream_t st, bool block_scaled = false) {
    if (!offsets || !A || !sa || !B || !sb || !out || rows < 0 || a_rows < 0 || groups < 1 || N < 0 || Kdim < 0)
        return MOE_ERR_INVALID_ARG;
    if (epilogue != MOE_EPI_BF16 && epilogue != MOE_EPI_SWIGLU_FP8 && epilogue != MOE_EPI_F32 &&
        epilogue != MOE_EPI_BF16_F32_LAST && epilogue != MOE_EPI_GATEUP_F32)
        return MOE_ERR_INVALID_ARG;
    if (epilogue == MOE_EPI_GATEUP_F32 && block_scaled) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((epilogue == MOE_EPI_SWIGLU_FP8 || epilogue == MOE_EPI_BF16_F32_LAST) && !out_aux) return MOE_ERR_INVALID_ARG;
    if (epilogue == MOE_EPI_BF16_F32_LAST && !aligned16(out_aux)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if (groups > gemm::MAX_GROUPS || N % gemm::BN || N == 0 || Kdim % gemm::BK || Kdim == 0 || rows >= INT32_MAX ||
        a_rows >= INT32_MAX)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(groups) * N >= INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (N / gemm::BN > 256) return MOE_ERR_UNSUPPORTED_SHAPE;   // column tile index packed in 8 bits
    // the kernel addresses the scale arrays with 32-bit element offsets
    if ((row_index != nullptr ? a_rows : rows) * (Kdim / gemm::BK) >= UINT32_MAX ||
        static_cast<int64_t>(groups) * (N / 128) * (Kdim / gemm::BK) >= UINT32_MAX)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (row_index != nullptr && a_rows == 0) return MOE_ERR_INVALID_ARG;
    CUtensorMap ta, tb;
    const bool gather = row_index != nullptr;
    if (!make_map_u8(&ta, A, static_cast<uint64_t>(Kdim), static_cast<uint64_t>(gather ? a_rows : rows),
                     gather ? 1u : static_cast<uint32_t>(gemm::BM)))
        return MOE_ERR_CUDA;
    if (!make_map_u8(&tb, B, static_cast<uint64_t>(Kdim), static_cast<uint64_t>(groups) * N, gemm::BN))
        return MOE_ERR_CUDA;
    gemm::Params p{offsets, groups, rows, N, Kdim, sa, sb, out, out_aux, row_index, a_rows};
    const int64_t tiles_max = (ceil_div(rows, gemm::BM) + groups) * (N / gemm::BN);
    if (block_scaled) {
        if (epilogue == MOE_EPI_BF16) return launch_gemm_mx<MOE_EPI_BF16>(ta, tb, p, tiles_max, st);
        if (epilogue == MOE_EPI_F32) return launch_gemm_mx<MOE_EPI_F32>(ta, tb, p, tiles_max, st);
        if (epilogue == MOE_EPI_BF16_F32_LAST) return launch_gemm_mx<MOE_EPI_BF16_F32_LAST>(ta, tb, p, tiles_max, st);
        return launch_gemm_mx<MOE_EPI_SWIGLU_FP8>(ta, tb, p, tiles_max, st);
    }
    CUtensorMap to = ta;       // a placeholder for the epilogues that store directly
    if (epilogue == MOE_EPI_F32 || epilogue == MOE_EPI_GATEUP_F32) {
        if (!make_map_f32_box(&to, out, static_cast<uint64_t>(N), static_cast<uint64_t>(rows), gemm::OUT_BOX_COLS))
            return MOE_ERR_CUDA;
    }
    if (gather) return launch_gemm_epi<true>(epilogue, ta, tb, to, p, tiles_max, st);
    return launch_gemm_epi<false>(epilogue, ta, tb, to, p, tiles_max, st);
}

const char* kStatusNames[] = {
    "MOE_OK",
    "MOE_ERR_INVALID_ARG: null or misaligned pointer, negative size or bad enum",
    "MOE_ERR_UNSUPPORTED_SHAPE: shape outside the supported set",
    "MOE_ERR_WORKSPACE: workspace missing or too small",
    "MOE_ERR_CUDA: a CUDA runtime call failed",
    "MOE_ERR_TIMEOUT: a bounded device wait ran out",
    "MOE_ERR_DEVICE_CHECK: a device-side index or offset check failed",
    "MOE_ERR_NO_DEVICE: no usable sm_103 device",
};

// ---------------------------------------------------------------------------
// Static scratch of moe_permute_noalloc: the per-block expert counts and
// per-block starting rows (2 * nblk * E int32) live in this file-scope device
// array instead of a caller workspace. Every device that loads the library
// holds it until the process exits.
constexpr size_t kPermuteScratchInts = 256 * 1024;   // 1 MiB
static __device__ __align__(256) int32_t g_permute_scratch[kPermuteScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is asked of the
// runtime once per device (with that device current) and cached.
moe_status permute_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

template <int EPL>
void launch_balance_partial(const float* z, const int* splits, const moe_config* c, const float* offset,
                            const int32_t* idx, float* p_part, int32_t* c_part, cudaStream_t st) {
    const int nchunk = c->T / 32;
    const int grid = static_cast<int>(std::min<int64_t>(ceil_div(nchunk, 4), static_cast<int64_t>(num_sms()) * 8));
    route::balance_partial_kernel<EPL><<<grid, 128, 0, st>>>(z, splits, c->T, c->E, c->K, offset, idx, p_part,
                                                             c_part);
}

// Checks shared by the 128x1 grouped quantisers; returns MOE_OK to launch.
moe_status check_q1(int32_t groups, const int32_t* offsets, int64_t rows, int32_t cols, int32_t rule,
                    const uint8_t* qT, int64_t ldq, const float* sT) {
    if (!offsets || !qT || !sT || groups < 1 || rows < 0 || cols < 0 || ldq < 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(qT) || !aligned16(sT) || ldq % 16) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    if (groups > bwd::kQ1MaxGroups || cols % 128 || rows >= INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

template <int SRC>
moe_status launch_q1(const bwd::QSrc& src, int32_t groups, const int32_t* offsets, int64_t rows, int32_t cols,
                     int32_t rule, uint8_t* qT, int64_t ldq, float* sT, cudaStream_t st) {
    if (rows == 0 || cols == 0) return MOE_OK;
    const size_t smem = 128 * 129 * sizeof(float) + static_cast<size_t>(groups + 1) * sizeof(int);
    static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};
    const int ri = rule == MOE_SCALE_POW2 ? 1 : 0;
    const void* fn = rule == MOE_SCALE_POW2 ? reinterpret_cast<const void*>(bwd::quant_128x1_kernel<SRC, true>)
                                            : reinterpret_cast<const void*>(bwd::quant_128x1_kernel<SRC, false>);
    if (smem_attr(fn, 128 * 129 * sizeof(float) + (bwd::kQ1MaxGroups + 1) * sizeof(int), attr_done[ri]) != MOE_OK)
        return MOE_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>(ceil_div(rows, 128) + groups), static_cast<unsigned>(cols / 128));
    if (rule == MOE_SCALE_POW2)
        bwd::quant_128x1_kernel<SRC, true><<<grid, 256, smem, st>>>(src, rows, cols, groups, offsets, qT, ldq, sT);
    else
        bwd::quant_128x1_kernel<SRC, false><<<grid, 256, smem, st>>>(src, rows, cols, groups, offsets, qT, ldq, sT);
    return launch_status();
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    if (static_cast<int>(s) < 0 || static_cast<int>(s) >= static_cast<int>(sizeof(kStatusNames) / sizeof(kStatusNames[0])))
        return "MOE_ERR_UNKNOWN";
    return kStatusNames[s];
}

const char* moe_version(void) { return "moe_b300 1.0 (sm_103a)"; }

moe_status moe_check_device_status(void* stream) {
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, moe::g_status, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(moe::g_status, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    return static_cast<moe_status>(v);
}

size_t moe_workspace_size(const moe_config* cfg) {
    if (check_config(cfg) != MOE_OK) return 0;
    return ws_layout(cfg).total;
}

moe_status moe_router_planes(const float* Wr, int32_t E, int32_t d, uint16_t* planes, void* stream) {
    if (!Wr || !planes || E < 1 || d < 1) return MOE_ERR_INVALID_ARG;
    const int64_t nw = static_cast<int64_t>(E) * d;
    rtc::split_kernel<<<static_cast<unsigned>(ceil_div(nw, 256)), 256, 0, as_stream(stream)>>>(Wr, nw, planes);
    return launch_status();
}

moe_status moe_route_planes(const moe_config* cfg, const uint16_t* x, const uint16_t* planes,
                            const float* logit_offset, const float* bias, int32_t* topk_idx, float* topk_gate,
                            int32_t* counts, int32_t path, void* workspace, size_t workspace_bytes, void* stream) {
    const moe_status cs = check_config(cfg);
    if (cs != MOE_OK) return cs;
    if (!x || !planes || !bias || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(planes) || !aligned16(topk_idx) || !aligned16(topk_gate))
        return MOE_ERR_INVALID_ARG;
    if (path != MOE_ROUTE_AUTO && path != MOE_ROUTE_FUSED && path != MOE_ROUTE_SPLIT) return MOE_ERR_INVALID_ARG;
    if (path == MOE_ROUTE_FUSED && cfg->E > rtc::BN_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout wl = ws_layout(cfg);
    if (workspace == nullptr || workspace_bytes < wl.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    const bool fused = path == MOE_ROUTE_FUSED || (path == MOE_ROUTE_AUTO && route_fused_auto(cfg));
    cudaStream_t st = as_stream(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* splits = reinterpret_cast<int*>(ws + wl.header);
    float* z = reinterpret_cast<float*>(ws + wl.logits);
    const int bn = std::min(cfg->E, rtc::BN_MAX);
    CUtensorMap tx, tw;
    if (!make_map_bf16(&tx, x, static_cast<uint64_t>(cfg->d), static_cast<uint64_t>(cfg->T), rtc::BM)) return MOE_ERR_CUDA;
    if (!make_map_bf16(&tw, planes, static_cast<uint64_t>(cfg->d), static_cast<uint64_t>(3) * cfg->E,
                       static_cast<uint32_t>(bn)))
        return MOE_ERR_CUDA;
    if (fused) {
        if (launch_fused(cfg, tx, tw, logit_offset, bias, topk_idx, topk_gate, z, splits, st) != MOE_OK)
            return MOE_ERR_CUDA;
    } else {
        const int ks = route_slices(cfg);
        if (launch_route_t<false, 1, 2>(cfg, tx, tw, ks, nullptr, nullptr, nullptr, nullptr, z, splits, st) != MOE_OK)
            return MOE_ERR_CUDA;
        const size_t sel_smem = static_cast<size_t>(route::kSelWarps) * 2 * cfg->E * sizeof(float);
        const int sel_grid = static_cast<int>(std::min<int64_t>(ceil_div(cfg->T, route::kSelWarps), 65535));
        launch_select(cfg, z, ks, logit_offset, bias, topk_idx, topk_gate, sel_grid, sel_smem, st);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    if (counts != nullptr) {
        const int nblk = static_cast<int>(ceil_div(cfg->T, perm::kTokPerBlk));
        int32_t* blk_counts = reinterpret_cast<int32_t*>(ws + wl.blk_counts);
        int32_t* blk_base = reinterpret_cast<int32_t*>(ws + wl.blk_base);
        const size_t hsm = static_cast<size_t>(perm::kWarps) * cfg->E * sizeof(int);
        const int64_t npairs = static_cast<int64_t>(cfg->T) * cfg->K;
        perm::hist_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(perm::KeyExpert{topk_idx, cfg->E}, npairs, cfg->K,
                                                                 cfg->E, blk_counts);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
        int32_t* offs = reinterpret_cast<int32_t*>(ws + wl.offsets);
        perm::scan_kernel<<<1, 1024, 0, st>>>(blk_counts, nblk, cfg->E, cfg->T, cfg->K, blk_base, offs, counts);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const uint16_t* x, const float* Wr, const float* logit_offset,
                     const float* bias, int32_t* topk_idx, float* topk_gate, int32_t* counts, void* workspace,
                     size_t workspace_bytes, void* stream) {
    const moe_status cs = check_config(cfg);
    if (cs != MOE_OK) return cs;
    if (!Wr || !aligned16(Wr)) return MOE_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(cfg);
    if (workspace == nullptr || workspace_bytes < wl.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    uint16_t* planes = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + wl.planes);
    const moe_status ps = moe_router_planes(Wr, cfg->E, cfg->d, planes, stream);
    if (ps != MOE_OK) return ps;
    return moe_route_planes(cfg, x, planes, logit_offset, bias, topk_idx, topk_gate, counts, MOE_ROUTE_AUTO,
                            workspace, workspace_bytes, stream);
}

moe_status moe_quant_fp8_1x128_rule(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int32_t rule,
                                    uint8_t* q, float* scale, void* stream) {
    if (!x || !q || !scale || rows < 0 || cols < 0 || ld < cols) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale) || ld % 8) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    if (cols % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || cols == 0) return MOE_OK;
    const int64_t tiles = rows * (cols / 128);
    // 8 warps per CTA, four tiles per warp step, two steps in flight per thread
    const int grid = static_cast<int>(std::min<int64_t>(ceil_div(tiles, 64), static_cast<int64_t>(num_sms()) * 16));
    if (rule == MOE_SCALE_POW2)
        quant_1x128_kernel<false, true><<<grid, 256, 0, as_stream(stream)>>>(x, rows, cols, ld, q, scale, nullptr, 0);
    else
        quant_1x128_kernel<false, false><<<grid, 256, 0, as_stream(stream)>>>(x, rows, cols, ld, q, scale, nullptr, 0);
    return launch_status();
}

moe_status moe_quant_fp8_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q, float* scale,
                               void* stream) {
    return moe_quant_fp8_1x128_rule(x, rows, cols, ld, MOE_SCALE_FP32, q, scale, stream);
}

moe_status moe_quant_fp8_1x128_scatter_rule(const moe_config* cfg, const uint16_t* x, const int32_t* row_of,
                                            int32_t rule, uint8_t* xq_perm, float* xs_perm, void* stream) {
    if (const moe_status st = check_config(cfg); st != MOE_OK) return st;
    if (!x || !row_of || !xq_perm || !xs_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq_perm)) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    const int64_t tiles = static_cast<int64_t>(cfg->T) * (cfg->d / 128);
    const int grid = static_cast<int>(std::min<int64_t>(ceil_div(tiles, 64), static_cast<int64_t>(num_sms()) * 16));
    if (rule == MOE_SCALE_POW2)
        quant_1x128_kernel<true, true><<<grid, 256, 0, as_stream(stream)>>>(x, cfg->T, cfg->d, cfg->d, xq_perm,
                                                                          xs_perm, row_of, cfg->K);
    else
        quant_1x128_kernel<true, false><<<grid, 256, 0, as_stream(stream)>>>(x, cfg->T, cfg->d, cfg->d, xq_perm,
                                                                           xs_perm, row_of, cfg->K);
    return launch_status();
}

moe_status moe_quant_fp8_1x128_scatter(const moe_config* cfg, const uint16_t* x, const int32_t* row_of,
                                       uint8_t* xq_perm, float* xs_perm, void* stream) {
    return moe_quant_fp8_1x128_scatter_rule(cfg, x, row_of, MOE_SCALE_FP32, xq_perm, xs_perm, stream);
}

moe_status moe_quant_fp8_128x128_rule(const float* w, int64_t batch, int64_t rows, int64_t cols, int32_t rule,
                                      uint8_t* q, float* scale, void* stream) {
    if (!w || !q || !scale || batch < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(scale)) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t blocks = batch * (rows / 128) * (cols / 128);
    if (blocks == 0) return MOE_OK;
    if (blocks > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rule == MOE_SCALE_POW2)
        quant_128x128_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, as_stream(stream)>>>(w, rows, cols, q, scale);
    else
        quant_128x128_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, as_stream(stream)>>>(w, rows, cols, q, scale);
    return launch_status();
}

moe_status moe_quant_fp8_128x128(const float* w, int64_t batch, int64_t rows, int64_t cols, uint8_t* q, float* scale,
                                 void* stream) {
    return moe_quant_fp8_128x128_rule(w, batch, rows, cols, MOE_SCALE_FP32, q, scale, stream);
}

moe_status moe_pack_w13(const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3, int64_t batch,
                        int64_t I, int64_t d, uint8_t* q13, float* s13, void* stream) {
    if (!q1 || !s1 || !q3 || !s3 || !q13 || !s13 || batch < 0 || I < 0 || d < 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(q1) || !aligned16(q3) || !aligned16(q13)) return MOE_ERR_INVALID_ARG;
    if (I % 128 || d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (batch == 0 || I == 0 || d == 0) return MOE_OK;
    cudaStream_t st = as_stream(stream);
    const int64_t rows = batch * 2 * I;
    pack_w13_kernel<<<static_cast<unsigned>(ceil_div(rows * 32, 256)), 256, 0, st>>>(q1, q3, batch, I, d, q13);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    const int64_t ns = batch * 2 * (I / 128) * (d / 128);
    pack_w13_scale_kernel<<<static_cast<unsigned>(ceil_div(ns, 256)), 256, 0, st>>>(s1, s3, batch, I / 128, d / 128, s13);
    return launch_status();
}

moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx, const uint8_t* xq, const float* xs,
                       int32_t* offsets, int32_t* counts, int32_t* sorted_token, int32_t* row_of, uint8_t* xq_perm,
                       float* xs_perm, void* workspace, size_t workspace_bytes, void* stream) {
    const moe_status cs = check_config(cfg);
    if (cs != MOE_OK) return cs;
    if (!topk_idx || !offsets || !sorted_token || !row_of) return MOE_ERR_INVALID_ARG;
    const bool gather_rows = xq_perm != nullptr || xs_perm != nullptr;
    if (gather_rows && (!xq || !xs || !xq_perm || !xs_perm)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(topk_idx) || (gather_rows && (!aligned16(xq) || !aligned16(xq_perm)))) return MOE_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(cfg);
    if (workspace == nullptr || workspace_bytes < wl.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* blk_counts = reinterpret_cast<int32_t*>(ws + wl.blk_counts);
    int32_t* blk_base = reinterpret_cast<int32_t*>(ws + wl.blk_base);
    const int nblk = static_cast<int>(ceil_div(cfg->T, perm::kTokPerBlk));
    const int64_t npairs = static_cast<int64_t>(cfg->T) * cfg->K;
    const size_t hsm = static_cast<size_t>(perm::kWarps) * cfg->E * sizeof(int);
    perm::hist_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(perm::KeyExpert{topk_idx, cfg->E}, npairs, cfg->K,
                                                                 cfg->E, blk_counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scan_kernel<<<1, 1024, 0, st>>>(blk_counts, nblk, cfg->E, cfg->T, cfg->K, blk_base, offsets, counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scatter_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(perm::KeyExpert{topk_idx, cfg->E}, npairs, cfg->K,
                                                               cfg->E, blk_base, row_of, sorted_token);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (!gather_rows) return MOE_OK;
    const int64_t rows = npairs + cfg->T;
    perm::gather_kernel<<<static_cast<unsigned>(ceil_div(rows * 32, 256)), 256, 0, st>>>(
        sorted_token, cfg->T, cfg->K, cfg->d, xq, xs, xq_perm, xs_perm);
    return launch_status();
}

moe_status moe_balance_loss(const moe_config* cfg, const float* logit_offset, const int32_t* topk_idx,
                            int32_t seq_len, float alpha, float* f, float* P, float* loss, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (const moe_status st = check_config(cfg); st != MOE_OK) return st;
    if (!topk_idx || !loss || !workspace) return MOE_ERR_INVALID_ARG;
    if (seq_len < 32 || seq_len % 32 || cfg->T % seq_len) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WsLayout w = ws_layout(cfg);
    if (workspace_bytes < w.total) return MOE_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const float* z = reinterpret_cast<const float*>(ws + w.logits);
    const int* splits = reinterpret_cast<const int*>(ws + w.header);
    float* p_part = reinterpret_cast<float*>(ws + w.balance);
    int32_t* c_part = reinterpret_cast<int32_t*>(
        ws + w.balance + align_up(static_cast<size_t>(ceil_div(cfg->T, 32)) * cfg->E * sizeof(float), 256));
    const cudaStream_t st = as_stream(stream);
    const int epl = (cfg->E + 31) / 32;
    if (epl <= 8)
        launch_balance_partial<8>(z, splits, cfg, logit_offset, topk_idx, p_part, c_part, st);
    else if (epl <= 16)
        launch_balance_partial<16>(z, splits, cfg, logit_offset, topk_idx, p_part, c_part, st);
    else
        launch_balance_partial<32>(z, splits, cfg, logit_offset, topk_idx, p_part, c_part, st);
    const int nseq = cfg->T / seq_len;
    route::balance_final_kernel<<<ceil_div(nseq, 4), 128, 0, st>>>(p_part, c_part, nseq, seq_len, cfg->E, cfg->K,
                                                                   alpha, f, P, loss);
    return launch_status();
}

moe_status moe_permute_noalloc(const moe_config* cfg, const int32_t* topk_idx, const uint8_t* xq, const float* xs,
                               int32_t* offsets, int32_t* counts, int32_t* sorted_token, int32_t* row_of,
                               uint8_t* xq_perm, float* xs_perm, void* stream) {
    const moe_status cs = check_config(cfg);
    if (cs != MOE_OK) return cs;
    const int64_t nblk = ceil_div(cfg->T, perm::kTokPerBlk);
    if (2 * nblk * cfg->E > static_cast<int64_t>(kPermuteScratchInts)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!topk_idx || !offsets || !sorted_token || !row_of) return MOE_ERR_INVALID_ARG;
    const bool gather_rows = xq_perm != nullptr || xs_perm != nullptr;
    if (gather_rows && (!xq || !xs || !xq_perm || !xs_perm)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(topk_idx) || (gather_rows && (!aligned16(xq) || !aligned16(xq_perm)))) return MOE_ERR_INVALID_ARG;
    int32_t* scratch = nullptr;
    const moe_status ss = permute_scratch(&scratch);
    if (ss != MOE_OK) return ss;
    // every scratch entry is written by the histogram and scan kernels before
    // it is read, so nothing left by an earlier call needs clearing
    int32_t* blk_counts = scratch;
    int32_t* blk_base = scratch + nblk * cfg->E;
    cudaStream_t st = as_stream(stream);
    const int64_t npairs = static_cast<int64_t>(cfg->T) * cfg->K;
    const size_t hsm = static_cast<size_t>(perm::kWarps) * cfg->E * sizeof(int);
    perm::hist_kernel<<<static_cast<unsigned>(nblk), perm::kWarps * 32, hsm, st>>>(
        perm::KeyExpert{topk_idx, cfg->E}, npairs, cfg->K, cfg->E, blk_counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scan_kernel<<<1, 1024, 0, st>>>(blk_counts, static_cast<int>(nblk), cfg->E, cfg->T, cfg->K, blk_base,
                                          offsets, counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scatter_kernel<<<static_cast<unsigned>(nblk), perm::kWarps * 32, hsm, st>>>(
        perm::KeyExpert{topk_idx, cfg->E}, npairs, cfg->K, cfg->E, blk_base, row_of, sorted_token);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (!gather_rows) return MOE_OK;
    const int64_t rows = npairs + cfg->T;
    perm::gather_kernel<<<static_cast<unsigned>(ceil_div(rows * 32, 256)), 256, 0, st>>>(
        sorted_token, cfg->T, cfg->K, cfg->d, xq, xs, xq_perm, xs_perm);
    return launch_status();
}

moe_status moe_grouped_gemm_fp8(int32_t groups, const int32_t* offsets, int64_t rows, int32_t N, int32_t Kdim,
                                const uint8_t* A, const float* sa, const uint8_t* B, const float* sb, int32_t epilogue,
                                void* out, float* out_aux, void* stream) {
    return grouped_gemm(groups, offsets, rows, N, Kdim, A, sa, rows, nullptr, B, sb, epilogue, out, out_aux,
                        as_stream(stream));
}

moe_status moe_grouped_gemm_fp8_mx(int32_t groups, const int32_t* offsets, int64_t rows, int32_t N, int32_t Kdim,
                                   const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                                   int32_t epilogue, void* out, float* out_aux, void* stream) {
    return grouped_gemm(groups, offsets, rows, N, Kdim, A, sa, rows, nullptr, B, sb, epilogue, out, out_aux,
                        as_stream(stream), true);
}

moe_status moe_grouped_gemm_fp8_gather(int32_t groups, const int32_t* offsets, int64_t rows, int32_t N, int32_t Kdim,
                                       const uint8_t* A, const float* sa, int64_t a_rows, const int32_t* row_index,
                                       const uint8_t* B, const float* sb, int32_t epilogue, void* out, float* out_aux,
                                       void* stream) {
    if (!row_index) return MOE_ERR_INVALID_ARG;
    return grouped_gemm(groups, offsets, rows, N, Kdim, A, sa, a_rows, row_index, B, sb, epilogue, out, out_aux,
                        as_stream(stream));
}

moe_status moe_combine(const moe_config* cfg, const uint16_t* routed_out, const float* shared_out,
                       const int32_t* row_of, const float* topk_gate, const uint16_t* residual, uint16_t* y,
                       void* stream) {
    const moe_status cs = check_config(cfg);
    if (cs != MOE_OK) return cs;
    if (!routed_out || !shared_out || !row_of || !topk_gate || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(routed_out) || !aligned16(shared_out) || !aligned16(y) || (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    combine_kernel<<<cfg->T, 256, 0, as_stream(stream)>>>(routed_out, shared_out, row_of, topk_gate, residual, cfg->T,
                                                          cfg->K, cfg->d, y);
    return launch_status();
}

moe_status moe_bias_update(int32_t E, int32_t T, int32_t K, const int32_t* counts, float gamma, float* bias,
                           void* stream) {
    if (!counts || !bias || E < 1 || T < 0 || K < 1) return MOE_ERR_INVALID_ARG;
    bias_update_kernel<<<static_cast<unsigned>(ceil_div(E, 256)), 256, 0, as_stream(stream)>>>(E, T, K, counts, gamma,
                                                                                              bias);
    return launch_status();
}

// ------------------------------------------------------------- backward ----
moe_status moe_transpose_fp8_blocks(const uint8_t* q, const float* scale, int64_t batch, int64_t rows, int64_t cols,
                                    uint8_t* qT, float* scaleT, int64_t ldT, int64_t colsT, void* stream) {
    if (!q || !scale || !qT || !scaleT || batch < 0 || rows < 0 || cols < 0 || ldT < rows || colsT < cols)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qT) || ldT % 16) return MOE_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128 || ldT % 128 || colsT % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t blocks = batch * (rows / 128) * (cols / 128);
    if (blocks == 0) return MOE_OK;
    if (blocks > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    bwd::transpose_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, as_stream(stream)>>>(q, scale, rows, cols, qT,
                                                                                              scaleT, ldT, colsT);
    return launch_status();
}

moe_status moe_combine_backward(const moe_config* cfg, const uint16_t* dy, const uint16_t* routed_out,
                                const int32_t* row_of, const float* topk_gate, int32_t rule, uint8_t* dOq, float* dOs,
                                float* row_gate, float* dgate, void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (!dy || !routed_out || !row_of || !topk_gate || !dOq || !dOs || !row_gate || !dgate) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(routed_out) || !aligned16(dOq)) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (rule == MOE_SCALE_POW2)
        bwd::combine_backward_kernel<true><<<cfg->T, 256, 0, st>>>(dy, routed_out, row_of, topk_gate, cfg->T, cfg->K,
                                                                   cfg->d, dOq, dOs, row_gate, dgate);
    else
        bwd::combine_backward_kernel<false><<<cfg->T, 256, 0, st>>>(dy, routed_out, row_of, topk_gate, cfg->T, cfg->K,
                                                                    cfg->d, dOq, dOs, row_gate, dgate);
    return launch_status();
}

moe_status moe_route_backward(const moe_config* cfg, const float* logit_offset, const int32_t* topk_idx,
                              const float* dgate, float* dz, void* workspace, size_t workspace_bytes, void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (!topk_idx || !dgate || !dz) return MOE_ERR_INVALID_ARG;
    const WsLayout wl = ws_layout(cfg);
    if (workspace == nullptr || workspace_bytes < wl.total) return MOE_ERR_WORKSPACE;
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    const float* z = reinterpret_cast<const float*>(ws + wl.logits);
    const int* splits = reinterpret_cast<const int*>(ws + wl.header);
    bwd::route_backward_kernel<<<static_cast<unsigned>(ceil_div(cfg->T, 4)), 128, 0, as_stream(stream)>>>(
        z, splits, cfg->T, cfg->E, cfg->K, logit_offset, topk_idx, dgate, dz);
    return launch_status();
}

moe_status moe_router_wgrad(const moe_config* cfg, const uint16_t* x, const int32_t* offsets,
                            const int32_t* sorted_token, const int32_t* row_of, const float* dz, float* dWr,
                            void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (!x || !offsets || !sorted_token || !row_of || !dz || !dWr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(dWr)) return MOE_ERR_INVALID_ARG;
    const dim3 grid(static_cast<unsigned>(cfg->E), static_cast<unsigned>(ceil_div(cfg->d, 512)));
    bwd::router_wgrad_kernel<<<grid, 256, 0, as_stream(stream)>>>(x, cfg->T, cfg->K, cfg->d, offsets, sorted_token,
                                                                  row_of, dz, dWr);
    return launch_status();
}

moe_status moe_swiglu_backward(int64_t rows, int32_t I, float* ab, const float* dh, int64_t ld_dh, int32_t rule,
                               uint8_t* dab_q, float* dab_s, void* stream) {
    if (!ab || !dh || !dab_q || !dab_s || rows < 0 || I < 0 || ld_dh < I) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ab) || !aligned16(dh) || !aligned16(dab_q) || ld_dh % 4) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_SCALE_FP32 && rule != MOE_SCALE_POW2) return MOE_ERR_INVALID_ARG;
    if (I % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || I == 0) return MOE_OK;
    const int64_t warps = rows * (I / 128);
    const int grid = static_cast<int>(std::min<int64_t>(ceil_div(warps, 8), static_cast<int64_t>(num_sms()) * 32));
    if (rule == MOE_SCALE_POW2)
        bwd::swiglu_backward_kernel<true><<<grid, 256, 0, as_stream(stream)>>>(ab, dh, ld_dh, rows, I, dab_q, dab_s);
    else
        bwd::swiglu_backward_kernel<false><<<grid, 256, 0, as_stream(stream)>>>(ab, dh, ld_dh, rows, I, dab_q, dab_s);
    return launch_status();
}

moe_status moe_dx_combine(const moe_config* cfg, const uint16_t* dx_routed, const float* dx_shared,
                          const int32_t* row_of, const int32_t* topk_idx, const float* dz, const float* Wr, uint16_t* dx,
                          void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (!dx_routed || !dx_shared || !row_of || !topk_idx || !dz || !Wr || !dx) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dx_routed) || !aligned16(dx_shared) || !aligned16(Wr) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
    bwd::dx_combine_kernel<<<cfg->T, 256, 0, as_stream(stream)>>>(dx_routed, dx_shared, row_of, topk_idx, dz, Wr,
                                                                 cfg->T, cfg->K, cfg->d, cfg->E, dx);
    return launch_status();
}

moe_status moe_quant_fp8_128x1_f32(const float* v, int64_t ld, int32_t groups, const int32_t* offsets, int64_t rows,
                                   int32_t cols, int32_t rule, uint8_t* qT, int64_t ldq, float* sT, void* stream) {
    if (const moe_status cs = check_q1(groups, offsets, rows, cols, rule, qT, ldq, sT); cs != MOE_OK) return cs;
    if (!v || !aligned16(v) || ld < cols || ld % 4) return MOE_ERR_INVALID_ARG;
    bwd::QSrc src{};
    src.f32 = v;
    src.ld = ld;
    return launch_q1<bwd::SRC_F32>(src, groups, offsets, rows, cols, rule, qT, ldq, sT, as_stream(stream));
}

moe_status moe_quant_fp8_128x1_fp8(const uint8_t* q, const float* scale, int64_t ld, int32_t groups,
                                   const int32_t* offsets, int64_t rows, int32_t cols, int32_t rule, uint8_t* qT,
                                   int64_t ldq, float* sT, void* stream) {
    if (const moe_status cs = check_q1(groups, offsets, rows, cols, rule, qT, ldq, sT); cs != MOE_OK) return cs;
    if (!q || !scale || !aligned16(q) || ld < cols || ld % 128) return MOE_ERR_INVALID_ARG;
    bwd::QSrc src{};
    src.q8 = q;
    src.s8 = scale;
    src.ld = ld;
    src.ld_s = ld / 128;
    return launch_q1<bwd::SRC_FP8>(src, groups, offsets, rows, cols, rule, qT, ldq, sT, as_stream(stream));
}

moe_status moe_quant_fp8_128x1_bf16_rows(const uint16_t* x, int64_t x_rows, int64_t ld, const int32_t* row_map,
                                         const float* row_mult, int32_t groups, const int32_t* offsets, int64_t rows,
                                         int32_t cols, int32_t rule, uint8_t* qT, int64_t ldq, float* sT,
                                         void* stream) {
    if (const moe_status cs = check_q1(groups, offsets, rows, cols, rule, qT, ldq, sT); cs != MOE_OK) return cs;
    if (!x || !row_map || !aligned16(x) || ld < cols || ld % 8 || x_rows < 0) return MOE_ERR_INVALID_ARG;
    bwd::QSrc src{};
    src.bf16 = x;
    src.map = row_map;
    src.mult = row_mult;
    src.ld = ld;
    src.src_rows = x_rows;
    return launch_q1<bwd::SRC_BF16_ROWS>(src, groups, offsets, rows, cols, rule, qT, ldq, sT, as_stream(stream));
}

moe_status moe_grouped_wgrad_fp8(int32_t groups, const int32_t* offsets, int64_t rows, int64_t width, int32_t M,
                                 int32_t N, const uint8_t* AT, const float* saT, const uint8_t* BT, const float* sbT,
                                 float* out, void* stream) {
    if (!offsets || !AT || !saT || !BT || !sbT || !out || groups < 1 || rows < 0 || width < 0 || M < 0 || N < 0)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(AT) || !aligned16(BT) || !aligned16(saT) || !aligned16(sbT) ||
        (reinterpret_cast<uintptr_t>(out) & 31u) != 0)      // 32-byte vector stores
        return MOE_ERR_INVALID_ARG;
    if (groups > wgrad::MAX_GROUPS || M % gemm::BM || N % gemm::BN || width % 128 || M == 0 || N == 0 ||
        rows >= INT32_MAX || width >= INT32_MAX)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(groups) * (M / gemm::BM) * (N / gemm::BN) >= INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (width == 0) {
        // no rows at all: every gradient is zero
        return cudaMemsetAsync(out, 0, static_cast<size_t>(groups) * M * N * sizeof(float), as_stream(stream)) ==
                       cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    CUtensorMap ta, tb, to;
    if (!make_map_u8(&ta, AT, static_cast<uint64_t>(width), static_cast<uint64_t>(M), gemm::BM)) return MOE_ERR_CUDA;
    if (!make_map_u8(&tb, BT, static_cast<uint64_t>(width), static_cast<uint64_t>(N), gemm::BN)) return MOE_ERR_CUDA;
    if (!make_map_f32_box(&to, out, static_cast<uint64_t>(N), static_cast<uint64_t>(groups) * M, 32)) return MOE_ERR_CUDA;
    static std::atomic<uint64_t> attr_done{0};
    if (smem_attr(reinterpret_cast<const void*>(wgrad::grouped_wgrad_fp8_kernel), wgrad::SMEM_BYTES, attr_done) !=
        MOE_OK)
        return MOE_ERR_CUDA;
    wgrad::Params p{offsets, groups, rows, width / 128, M, N, saT, sbT, out};
    const int64_t tiles = static_cast<int64_t>(groups) * (M / gemm::BM) * (N / gemm::BN);
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), tiles));
    wgrad::grouped_wgrad_fp8_kernel<<<grid, gemm::NUM_THREADS, wgrad::SMEM_BYTES, as_stream(stream)>>>(ta, tb, to, p);
    return launch_status();
}

// ------------------------------------------------------ expert parallel ----
int64_t moe_ep_row_bytes(int32_t d, int32_t K) {
    if (d < 128 || d % 128 || K < 1 || K > 16) return 0;
    return ep::row_bytes(d, K);
}

size_t moe_ep_workspace_size(const moe_config* cfg, int32_t R, int64_t rows) {
    if (check_config(cfg) != MOE_OK || R < 1 || R > cfg->E || cfg->E % R || rows < 0) return 0;
    const int64_t keys = std::max<int64_t>(R, cfg->E / R);
    return 2 * align_up(static_cast<size_t>(ceil_div(std::max<int64_t>(rows, 1), perm::kTokPerBlk)) * keys * 4, 256);
}

moe_status moe_ep_dispatch(const moe_config* cfg, int32_t R, const int32_t* topk_idx, const float* topk_gate,
                           const uint8_t* xq, const float* xs, int32_t* send_counts, int32_t* send_offsets,
                           int32_t* send_row_of, int32_t* send_token, uint8_t* send_buf, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (R < 1 || R > cfg->E || cfg->E % R) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!topk_idx || !topk_gate || !xq || !xs || !send_offsets || !send_row_of || !send_token || !send_buf)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(send_buf) || !aligned16(topk_idx)) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_ep_workspace_size(cfg, R, cfg->T);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    const int nblk = static_cast<int>(ceil_div(cfg->T, perm::kTokPerBlk));
    int32_t* blk_counts = static_cast<int32_t*>(workspace);
    int32_t* blk_base = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + need / 2);
    const cudaStream_t st = as_stream(stream);
    const int64_t npairs = static_cast<int64_t>(cfg->T) * cfg->K;
    const perm::KeyDest key{topk_idx, cfg->E, cfg->E / R};
    const size_t hsm = static_cast<size_t>(perm::kWarps) * R * sizeof(int);
    perm::hist_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(key, npairs, cfg->K, R, blk_counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scan_kernel<<<1, 1024, 0, st>>>(blk_counts, nblk, R, cfg->T, cfg->K, blk_base, send_offsets, send_counts,
                                          false);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scatter_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(key, npairs, cfg->K, R, blk_base, send_row_of,
                                                               send_token, false);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    // at most min(K, R) send rows per token; warps past the total stop at once
    const int64_t cap = static_cast<int64_t>(cfg->T) * std::min(cfg->K, R);
    ep::pack_kernel<<<static_cast<unsigned>(ceil_div(cap * 32, 256)), 256, 0, st>>>(
        send_offsets + R, send_token, cap, cfg->T, cfg->d, cfg->K, xq, xs, topk_idx, topk_gate, send_buf);
    return launch_status();
}

moe_status moe_ep_receive(const moe_config* cfg, int32_t R, int32_t rank, int64_t n_recv, const uint8_t* recv_buf,
                          int32_t* local_offsets, int32_t* local_counts, int32_t* sorted_row, int32_t* row_of,
                          uint8_t* xq_local, float* xs_local, void* workspace, size_t workspace_bytes,
                          void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (R < 1 || R > cfg->E || cfg->E % R || rank < 0 || rank >= R || n_recv < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (n_recv * cfg->K >= INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!local_offsets || !sorted_row || !row_of || !xq_local || !xs_local || (n_recv > 0 && !recv_buf))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(xq_local) || (recv_buf && !aligned16(recv_buf))) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_ep_workspace_size(cfg, R, n_recv);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    const int n_local = cfg->E / R;
    const int nblk = static_cast<int>(ceil_div(std::max<int64_t>(n_recv, 1), perm::kTokPerBlk));
    int32_t* blk_counts = static_cast<int32_t*>(workspace);
    int32_t* blk_base = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + need / 2);
    const cudaStream_t st = as_stream(stream);
    const int64_t npairs = n_recv * cfg->K;
    const int64_t rb = ep::row_bytes(cfg->d, cfg->K);
    const int32_t* ridx =
        recv_buf != nullptr ? reinterpret_cast<const int32_t*>(recv_buf + cfg->d + 4 * (cfg->d / 128)) : nullptr;
    const perm::KeyWindow key{ridx, rb / 4, cfg->E, rank * n_local, n_local};
    const size_t hsm = static_cast<size_t>(perm::kWarps) * n_local * sizeof(int);
    perm::hist_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(key, npairs, cfg->K, n_local, blk_counts);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    perm::scan_kernel<<<1, 1024, 0, st>>>(blk_counts, nblk, n_local, static_cast<int>(n_recv), cfg->K, blk_base,
                                          local_offsets, local_counts, false);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (n_recv == 0) return MOE_OK;
    perm::scatter_kernel<<<nblk, perm::kWarps * 32, hsm, st>>>(key, npairs, cfg->K, n_local, blk_base, row_of,
                                                               sorted_row, false);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    ep::gather_kernel<<<static_cast<unsigned>(ceil_div(npairs * 32, 256)), 256, 0, st>>>(
        local_offsets, n_local, sorted_row, n_recv, recv_buf, cfg->d, cfg->K, xq_local, xs_local);
    return launch_status();
}

moe_status moe_ep_partial(const moe_config* cfg, int64_t n_recv, const uint8_t* recv_buf, const int32_t* row_of,
                          const uint16_t* routed_out, int64_t out_rows, float* partial, void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (n_recv < 0 || out_rows < 0 || n_recv > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (n_recv == 0) return MOE_OK;
    if (!recv_buf || !row_of || !routed_out || !partial) return MOE_ERR_INVALID_ARG;
    if (!aligned16(recv_buf) || !aligned16(routed_out) || !aligned16(partial)) return MOE_ERR_INVALID_ARG;
    ep::partial_kernel<<<static_cast<unsigned>(n_recv), 256, 0, as_stream(stream)>>>(recv_buf, cfg->d, cfg->K, row_of,
                                                                                     out_rows, routed_out, partial);
    return launch_status();
}

moe_status moe_ep_combine(const moe_config* cfg, const float* shared_out, const float* returned, int64_t S,
                          const int32_t* send_row_of, const uint16_t* residual, uint16_t* y, void* stream) {
    if (const moe_status cs = check_config(cfg); cs != MOE_OK) return cs;
    if (!shared_out || !send_row_of || !y || S < 0 || (S > 0 && !returned)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(shared_out) || !aligned16(y) || (returned && !aligned16(returned)) ||
        (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    ep::combine_kernel<<<cfg->T, 256, 0, as_stream(stream)>>>(shared_out, returned, send_row_of, S, residual, cfg->T,
                                                              cfg->K, cfg->d, y);
    return launch_status();
}

moe_status moe_selftest_wait_timeout(uint32_t limit_us, void* stream) {
    selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(static_cast<uint64_t>(limit_us) * 1000ull);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    return moe_check_device_status(stream);
}

}  // extern "C"
