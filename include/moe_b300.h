/*
 * moe_b300.h -- C ABI of the B300 (sm_103a) DeepSeekMoE layer forward.
 *
 * The layer (《DeepSeek-V3 Technical Report》深度解读报告, §2.2 DeepSeekMoE):
 *     y = [u +] FFN_shared(u) + sum_{k<K} g_k * FFN_{e_k}(u)
 * with sigmoid affinities, aux-loss-free biased top-K choice (§2.3),
 * group-limited routing (§2.4), and expert FFNs run as FP8 (E4M3) GEMMs
 * with activations scaled per 1x128 tile, weights per 128x128 block and
 * partial sums promoted to FP32 every 128-element K chunk ("DeepSeek-V3的
 * MoE架构设计革新", §2 FP8 training, items 1-2).
 *
 * Conventions for every call:
 *  - The caller owns all memory. Pointers named as device pointers must be
 *    device memory of the current CUDA device; the library never
 *    allocates. Calls that need scratch take a caller-provided workspace of
 *    at least moe_workspace_size() bytes.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) except where stated. Calls never print, never
 *    throw and never abort.
 *  - Errors found on the host (null pointer, bad size, misalignment, too
 *    small workspace) return a non-zero status before anything is launched.
 *    Errors found on the device (corrupt routing indices or offsets, a
 *    bounded wait that ran out) set a device status word that
 *    moe_check_device_status() reads and clears.
 *  - bf16 tensors are passed as uint16_t bit patterns. Matrices are
 *    row-major with the last index contiguous unless stated.
 *  - Device pointers must be 16-byte aligned.
 *
 * Shapes (moe_config): T tokens, d hidden, E routed experts, I expert
 * intermediate size (the shared expert has the same I), K experts per
 * token, G expert groups (contiguous blocks of E/G experts standing in for
 * nodes), M groups a token may reach, gk highest affinities summed into a
 * group's score. Supported: T >= 1; d, I multiples of 128; 16 <= E <= 1024,
 * E % 16 == 0, E % G == 0, G <= 32; 1 <= M <= G; 1 <= gk <= E/G;
 * 1 <= K <= min(16, M*E/G). Anything else is MOE_ERR_UNSUPPORTED_SHAPE.
 *
 * Grouped rows: the routed (token, slot) pairs are grouped by expert
 * (ascending expert, then ascending token) into rows [0, T*K); the shared
 * expert's rows T*K + t (t < T) follow, so the whole layer runs as one
 * grouped GEMM over E + 1 groups.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null or misaligned pointer, negative size, bad enum */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above */
    MOE_ERR_WORKSPACE = 3,         /* workspace missing or smaller than required */
    MOE_ERR_CUDA = 4,              /* a CUDA runtime call failed (see cudaGetLastError) */
    MOE_ERR_TIMEOUT = 5,           /* a bounded device wait ran out; kernel returned early */
    MOE_ERR_DEVICE_CHECK = 6,      /* a device-side check of indices or offsets failed */
    MOE_ERR_NO_DEVICE = 7          /* no usable sm_103 device is current */
} moe_status;

typedef struct moe_config {
    int32_t T, d, E, I, K, G, M, gk;
} moe_config;

/* Epilogues of the grouped FP8 GEMM. */
typedef enum moe_epilogue {
    /* out: bf16 [rows][N]. */
    MOE_EPI_BF16 = 0,
    /* SwiGLU + 1x128 requantisation. B holds gate (W1) and up (W3) rows
     * interleaved as moe_pack_w13 writes them; out: E4M3 [rows][N/2],
     * out_scale: f32 [rows][N/256]. */
    MOE_EPI_SWIGLU_FP8 = 1,
    /* out: f32 [rows][N]. */
    MOE_EPI_F32 = 2,
    /* out: bf16 [rows][N] for every group but the last; out_aux: f32
     * [offsets[groups] - offsets[groups-1]][N] for the last group (the
     * shared expert, whose output enters the layer output with gate 1). */
    MOE_EPI_BF16_F32_LAST = 3,
    /* The SwiGLU pre-activations, unreduced: B laid out as for
     * MOE_EPI_SWIGLU_FP8; out: f32 [rows][N] in that tile layout (for I-block
     * j, columns 256j.. hold gate[128j..+64), up[128j..+64), gate[128j+64..
     * +128), up[128j+64..+128)). The backward pass recomputes them with this
     * epilogue; the values equal those the SwiGLU epilogue reduces. */
    MOE_EPI_GATEUP_F32 = 4
} moe_epilogue;

/* Human-readable name of a status. Never NULL. */
const char* moe_status_string(moe_status s);

/* Version string of the library build. */
const char* moe_version(void);

/* Synchronises `stream`, then returns and clears the device status word
 * (MOE_OK if no device-side check failed since the last call). Blocking. */
moe_status moe_check_device_status(void* stream);

/* Bytes of workspace moe_route and moe_permute need for `cfg` (the larger
 * of the two). 0 for an unsupported cfg. Host only, no device access. */
size_t moe_workspace_size(const moe_config* cfg);

/* Router: affinity, aux-loss-free group-limited top-K and gates.
 * 《DeepSeek-V3 Technical Report》深度解读报告 §2.2 (s_e = sigmoid(x . Wr_e),
 * gates = s over the chosen experts renormalised to 1), §2.3 (b_e added to
 * s_e only to choose experts), §2.4 (at most M groups per token, groups
 * ranked by the sum of their gk highest biased affinities).
 *   x            device bf16 [T][d]
 *   Wr           device f32  [E][d]
 *   logit_offset device f32  [E] or NULL: added to x . Wr_e before the sigmoid
 *                (a synthetic knob that skews expert popularity)
 *   bias         device f32  [E] selection bias b
 *   topk_idx     device i32  [T][K] out: chosen experts, by descending s + b
 *                (equal values: lower expert index first)
 *   topk_gate    device f32  [T][K] out: s_e / sum of s over the chosen experts
 *   counts       device i32  [E] out or NULL: pairs routed to each expert
 *   workspace    device, >= moe_workspace_size(cfg) bytes
 * Logits are computed on the tensor cores from x (bf16, exact) times Wr
 * split into three bf16 terms whose sum is Wr exactly, accumulated in FP32.
 * Equivalent to moe_router_planes into the workspace followed by
 * moe_route_planes(..., MOE_ROUTE_AUTO, ...). The logits stay in the
 * workspace for moe_route_backward and moe_balance_loss. */
moe_status moe_route(const moe_config* cfg, const uint16_t* x, const float* Wr,
                     const float* logit_offset, const float* bias,
                     int32_t* topk_idx, float* topk_gate, int32_t* counts,
                     void* workspace, size_t workspace_bytes, void* stream);

/* The router weight as three bf16 planes for moe_route_planes: planes[0] =
 * bf16(Wr), planes[1] = bf16(Wr - planes[0]), planes[2] = bf16(Wr - planes[0]
 * - planes[1]), whose sum is Wr exactly (FP32 has 24 significant bits, each
 * bf16 term 8). A set-up step, to be redone whenever Wr changes.
 *   Wr      device f32  [E][d]
 *   planes  device bf16 [3][E][d] out, 16-byte aligned, caller-owned */
moe_status moe_router_planes(const float* Wr, int32_t E, int32_t d, uint16_t* planes, void* stream);

/* Which router kernels moe_route_planes runs. */
typedef enum {
    /* the fused kernel when E <= 256 and ceil(T/128) reaches half the SM
     * count, otherwise the K-split kernels */
    MOE_ROUTE_AUTO = 0,
    /* one kernel, one CTA per 128-token tile: logits accumulated in TMEM in
     * K splits of at most 24 chunks of 64, the splits summed in registers in
     * order, the selection run from shared memory; E <= 256 (else
     * MOE_ERR_UNSUPPORTED_SHAPE) */
    MOE_ROUTE_FUSED = 1,
    /* a logits kernel that writes FP32 K-split partials to the workspace,
     * then a selection kernel that sums them in split order; any E, and the
     * SMs stay busy for small T */
    MOE_ROUTE_SPLIT = 2
} moe_route_path;

/* moe_route with the router weight given as planes (moe_router_planes) and
 * the kernel path chosen by `path` (moe_route_path; else
 * MOE_ERR_INVALID_ARG). When both paths use the same number of K splits
 * (whenever ceil(T/128) * ceil(E/256) alone covers the SMs) they add the
 * same FP32 partials in the same order and give bit-identical logits,
 * choices and gates. Other arguments as moe_route; planes 16-byte aligned. */
moe_status moe_route_planes(const moe_config* cfg, const uint16_t* x, const uint16_t* planes,
                            const float* logit_offset, const float* bias,
                            int32_t* topk_idx, float* topk_gate, int32_t* counts, int32_t path,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Activation quantisation per 1x128 tile ("DeepSeek-V3的MoE架构设计革新" §2
 * item 1; E4M3 largest finite value 448 from "DeepSeek-V3技术解析" §6.2):
 *   scale = fl32(amax / 448); q = E4M3_RNE_SATFINITE(fl32(x / scale)),
 *   scale 0 and codes 0x00/0x80 (by sign) for an all-zero tile.
 *   x     device bf16 [rows][ld] (the first cols of each row are used)
 *   q     device u8   [rows][cols]
 *   scale device f32  [rows][cols/128]
 * cols % 128 == 0, ld >= cols, ld % 8 == 0. */
moe_status moe_quant_fp8_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                               uint8_t* q, float* scale, void* stream);

/* moe_quant_fp8_1x128 of the T tokens x [T][d] (bf16, contiguous), with
 * each token's codes and scales written straight into grouped order: to
 * rows row_of[t][0..K) (as returned by moe_permute) and to the shared
 * expert's row T*K + t. Same values as moe_quant_fp8_1x128 followed by the
 * row gather of moe_permute, without the unpermuted copy.
 *   row_of   device i32 [T][K], values in [0, T*K) (else MOE_ERR_DEVICE_CHECK
 *            and that copy is not written)
 *   xq_perm  device u8  [T*K + T][d] out
 *   xs_perm  device f32 [T*K + T][d/128] out */
moe_status moe_quant_fp8_1x128_scatter(const moe_config* cfg, const uint16_t* x, const int32_t* row_of,
                                       uint8_t* xq_perm, float* xs_perm, void* stream);

/* Scale rule of the FP8 quantisers below.
 *   MOE_SCALE_FP32  scale = fl32(amax / 448), as above (the layer the pages
 *                   describe; the default of the calls without a rule).
 *   MOE_SCALE_POW2  scale = the smallest power of two s with 448 * s >= amax,
 *                   at least 2^-126; 0 for an all-zero tile. Every scale is
 *                   then an 8-bit exponent code, which the block-scaled
 *                   GEMM (moe_grouped_gemm_fp8_mx) applies in the tensor
 *                   core. The pages fix the tile shapes and the 448 bound
 *                   ("DeepSeek-V3的MoE架构设计革新" §2 item 1, "DeepSeek-V3技术
 *                   解析" §6.2) but not the scale's format; this is the
 *                   second reading. v / s is exact and |v / s| <= 448. */
typedef enum { MOE_SCALE_FP32 = 0, MOE_SCALE_POW2 = 1 } moe_scale_rule;

/* moe_quant_fp8_1x128 with a scale rule (moe_scale_rule; else MOE_ERR_INVALID_ARG). */
moe_status moe_quant_fp8_1x128_rule(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int32_t rule,
                                    uint8_t* q, float* scale, void* stream);

/* moe_quant_fp8_1x128_scatter with a scale rule. */
moe_status moe_quant_fp8_1x128_scatter_rule(const moe_config* cfg, const uint16_t* x, const int32_t* row_of,
                                            int32_t rule, uint8_t* xq_perm, float* xs_perm, void* stream);

/* moe_quant_fp8_128x128 with a scale rule. */
moe_status moe_quant_fp8_128x128_rule(const float* w, int64_t batch, int64_t rows, int64_t cols, int32_t rule,
                                      uint8_t* q, float* scale, void* stream);

/* Weight quantisation per 128x128 block, same rule as above with amax over
 * the block (same page, same item). Set-up only; `batch` independent
 * matrices stored back to back.
 *   w     device f32 [batch][rows][cols]
 *   q     device u8  [batch][rows][cols]
 *   scale device f32 [batch][rows/128][cols/128]
 * rows % 128 == 0, cols % 128 == 0. */
moe_status moe_quant_fp8_128x128(const float* w, int64_t batch, int64_t rows, int64_t cols,
                                 uint8_t* q, float* scale, void* stream);

/* Lays out quantised gate (W1) and up (W3) projections for the SwiGLU
 * epilogue. For each 128-row block j of I, rows 256j + [0,64) of W13 are
 * W1 rows 128j + [0,64), then W3 rows 128j + [0,64), then W1 rows
 * 128j + [64,128), then W3 rows 128j + [64,128). Scales: block 2j of the
 * output is W1's block j, block 2j + 1 is W3's block j.
 *   q1, q3   device u8  [batch][I][d];  s1, s3 device f32 [batch][I/128][d/128]
 *   q13      device u8  [batch][2I][d]; s13    device f32 [batch][2I/128][d/128]
 * Set-up only. */
moe_status moe_pack_w13(const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3,
                        int64_t batch, int64_t I, int64_t d,
                        uint8_t* q13, float* s13, void* stream);

/* Sequence-wise balance statistics and loss ("《DeepSeek-V3 Technical Report》
 * 深度解读报告" §2.3: beside the auxiliary-loss-free bias, a balance loss L_Bal
 * of very small weight alpha keeps a single sequence from extreme imbalance;
 * the page gives no formula, this is the plainest reading). Tokens form
 * sequences of seq_len consecutive tokens; for sequence q:
 *   f[q][i] = E / (K * seq_len) * (number of its tokens that chose expert i)
 *   P[q][i] = mean over its tokens t of s[t][i] / sum_j s[t][j]
 *   loss[q] = alpha * sum_i f[q][i] * P[q][i]
 * with s the unbiased affinities (sigmoid of the logits plus logit_offset).
 * Call after moe_route on the same workspace and stream: the router logits it
 * left there are read back, so logit_offset must be the one moe_route got.
 *   topk_idx  device i32 [T][K], moe_route's output
 *   seq_len   multiple of 32 dividing T (else MOE_ERR_UNSUPPORTED_SHAPE)
 *   f, P      device f32 [T/seq_len][E] out, or NULL
 *   loss      device f32 [T/seq_len] out
 * Deterministic (fixed summation order, no atomics). */
moe_status moe_balance_loss(const moe_config* cfg, const float* logit_offset, const int32_t* topk_idx,
                            int32_t seq_len, float alpha, float* f, float* P, float* loss, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Token permutation by expert (expert histogram, exclusive prefix sum and a
 * stable scatter, all without atomics), then a gather of the quantised
 * rows into grouped order. Rows are ordered by (expert, token); the shared
 * expert's rows T*K + t follow.
 *   topk_idx     device i32 [T][K] (values in [0, E); else MOE_ERR_DEVICE_CHECK)
 *   xq, xs       device u8 [T][d], f32 [T][d/128] (moe_quant_fp8_1x128 of x)
 *   offsets      device i32 [E+2] out: group g holds rows [offsets[g], offsets[g+1]);
 *                group E is the shared expert (offsets[E] = T*K, offsets[E+1] = T*K + T)
 *   counts       device i32 [E] out or NULL: histogram of topk_idx
 *   sorted_token device i32 [T*K + T] out: token of each grouped row (the
 *                shared expert's rows T*K + t hold t)
 *   row_of       device i32 [T][K] out: grouped row of each (token, slot)
 *   xq_perm      device u8  [T*K + T][d] out, or NULL together with xs_perm to
 *                skip the row gather (xq, xs are then not read)
 *   xs_perm      device f32 [T*K + T][d/128] out or NULL
 *   workspace    device, >= moe_workspace_size(cfg) bytes */
moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx,
                       const uint8_t* xq, const float* xs,
                       int32_t* offsets, int32_t* counts, int32_t* sorted_token, int32_t* row_of,
                       uint8_t* xq_perm, float* xs_perm,
                       void* workspace, size_t workspace_bytes, void* stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory: for example a host framework that owns every allocation and hands
 * this library only the input and output buffers of a call, or a serving
 * loop that forbids allocation after start-up. The pages have no
 * counterpart; this is a packaging variant of moe_permute with the same
 * arguments (minus the workspace) and bit-identical results.
 * Scratch: a file-scope device array of 1 MiB (262144 int32) inside the
 * library, held by every device that loads the library until the process
 * exits. It bounds the shape: 2 * ceil(T / 256) * E must not exceed 262144
 * (e.g. T <= 131072 tokens for E = 256), otherwise MOE_ERR_UNSUPPORTED_SHAPE
 * and nothing is launched. Allocates nothing and calls no allocating
 * routine.
 * The first call on each device looks up the array's device address with
 * cudaGetSymbolAddress (that device must be current) and caches it; make that
 * first call before any stream capture. The cache assumes the device's
 * primary context lives as long as the process: after cudaDeviceReset (or
 * any teardown of the primary context) the cached address may be stale, so
 * a process that resets a device must not call this entry point afterwards.
 * All calls share the one array: two calls that overlap on the GPU (e.g. on
 * different streams without ordering between them) race and give wrong
 * results. Each call writes every scratch entry it reads, so what an
 * earlier call left behind never matters. */
moe_status moe_permute_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                               const uint8_t* xq, const float* xs,
                               int32_t* offsets, int32_t* counts, int32_t* sorted_token, int32_t* row_of,
                               uint8_t* xq_perm, float* xs_perm, void* stream);

/* Grouped FP8 GEMM with per-chunk scale promotion
 * ("DeepSeek-V3的MoE架构设计革新" §2 items 1-2): for each group g and row r in
 * [offsets[g], offsets[g+1]),
 *   D[r][n] = sum_kc sa[r][kc] * sb[g][n/128][kc] * sum_{k in chunk kc} A[r][k] * B[g][n][k]
 * with E4M3 A and B, FP32 accumulation, kc over Kdim/128 chunks.
 *   groups    number of groups (<= 1025)
 *   offsets   device i32 [groups+1], non-decreasing, offsets[groups] <= rows
 *             (checked on the device: MOE_ERR_DEVICE_CHECK, nothing written)
 *   rows      rows of A and of the output
 *   A, sa     device u8 [rows][Kdim], f32 [rows][Kdim/128]
 *   B, sb     device u8 [groups][N][Kdim], f32 [groups][N/128][Kdim/128]
 *   epilogue  moe_epilogue; out / out_aux as described there
 * The SwiGLU epilogue computes h = SiLU(gate) * up in FP32 with the fast
 * exponential and division and quantises it per 1x128 tile with the scale
 * rule above, multiplying by the correctly rounded reciprocal of the scale;
 * h therefore matches an exact evaluation to a few FP32 ulps, not bit for
 * bit, and its E4M3 codes match except where that difference crosses a
 * rounding boundary.
 * N % 256 == 0, N <= 65536, Kdim % 128 == 0, rows * Kdim/128 and
 * groups * N/128 * Kdim/128 below 2^32 (else MOE_ERR_UNSUPPORTED_SHAPE).
 * Rows outside every group are not written.
 * Runs on the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA
 * operand loads); no workspace. With Kdim/128 a multiple of 4 and at most
 * 64 and sa, sb 16-byte aligned the chunk scales are read into registers
 * (the faster path); otherwise they stream through shared memory. Both give
 * the same bits. */
moe_status moe_grouped_gemm_fp8(int32_t groups, const int32_t* offsets, int64_t rows,
                                int32_t N, int32_t Kdim,
                                const uint8_t* A, const float* sa,
                                const uint8_t* B, const float* sb,
                                int32_t epilogue, void* out, float* out_aux, void* stream);

/* moe_grouped_gemm_fp8 for power-of-two scales (MOE_SCALE_POW2): the same
 * result, computed by the block-scaled tensor-core MMA
 * (tcgen05.mma.kind::mxf8f6f4.block_scale) that applies each K=32 step's
 * scales 2^ea * 2^eb from 8-bit exponent codes, so the whole K reduction of
 * a tile accumulates in one TMEM accumulator. sa and sb must hold powers of
 * two or zero (as moe_quant_*_rule(MOE_SCALE_POW2) writes them); any other
 * value sets MOE_ERR_DEVICE_CHECK. The SwiGLU epilogue quantises h with the
 * power-of-two rule. Arguments, layouts and other errors as
 * moe_grouped_gemm_fp8. */
moe_status moe_grouped_gemm_fp8_mx(int32_t groups, const int32_t* offsets, int64_t rows, int32_t N, int32_t Kdim,
                                   const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                                   int32_t epilogue, void* out, float* out_aux, void* stream);

/* moe_grouped_gemm_fp8 with the A operand gathered by row: grouped row r
 * reads row row_index[r] of A [a_rows][Kdim] and of sa [a_rows][Kdim/128]
 * (TMA gather, four rows per copy), e.g. the unpermuted quantised tokens with
 * row_index = sorted_token of moe_permute, so the permuted copy of the
 * activations never has to be written. row_index: device i32 [rows], values
 * in [0, a_rows) (else MOE_ERR_DEVICE_CHECK and row 0 is read). Other
 * arguments, layouts and errors as moe_grouped_gemm_fp8. */
moe_status moe_grouped_gemm_fp8_gather(int32_t groups, const int32_t* offsets, int64_t rows,
                                       int32_t N, int32_t Kdim,
                                       const uint8_t* A, const float* sa, int64_t a_rows,
                                       const int32_t* row_index,
                                       const uint8_t* B, const float* sb,
                                       int32_t epilogue, void* out, float* out_aux, void* stream);

/* Gate-weighted un-permute and combine (《DeepSeek-V3 Technical Report》深度解读报告
 * §2.2): y[t] = shared_out[t] + sum_k topk_gate[t][k] * routed_out[row_of[t][k]]
 * (+ residual[t] if residual != NULL), accumulated in FP32 in that order,
 * rounded to bf16.
 *   routed_out device bf16 [T*K][d]; shared_out device f32 [T][d]
 *   (the expert outputs of moe_grouped_gemm_fp8 with MOE_EPI_BF16_F32_LAST)
 *   row_of     device i32 [T][K] (values in [0, T*K), else MOE_ERR_DEVICE_CHECK)
 *   topk_gate  device f32 [T][K]; residual device bf16 [T][d] or NULL
 *   y          device bf16 [T][d] out */
moe_status moe_combine(const moe_config* cfg, const uint16_t* routed_out, const float* shared_out,
                       const int32_t* row_of, const float* topk_gate, const uint16_t* residual,
                       uint16_t* y, void* stream);

/* End-of-step bias update (《DeepSeek-V3 Technical Report》深度解读报告 §2.3):
 *   b_e <- fl32(b_e + gamma * sign(T*K/E - counts[e]))
 * i.e. overloaded experts lose gamma, underloaded experts gain gamma, an
 * expert exactly at the mean load keeps its bias.
 *   counts device i32 [E]; bias device f32 [E] in/out. */
moe_status moe_bias_update(int32_t E, int32_t T, int32_t K, const int32_t* counts,
                           float gamma, float* bias, void* stream);

/* ------------------------------------------------------------------------
 * Backward pass of the layer.
 *
 * The pages frame the FP8 recipe as training ("DeepSeek-V3的MoE架构设计革新"
 * §2 FP8 training) and the bias as acting on expert choice only
 * (《DeepSeek-V3 Technical Report》深度解读报告 §2.3); they print no backward
 * pass. These calls compute the plain one with the chosen experts held
 * fixed: gradients flow through the gates g = s/sum(s), the sigmoid
 * affinities s and the SwiGLU experts, not through the choice or the bias.
 * Each FP8 GEMM quantises along its contracted dimension: the data
 * gradients take 1x128 gradient tiles and the forward's 128x128 weight
 * blocks transposed (moe_transpose_fp8_blocks); the weight gradients take
 * 128-token x 1-channel tiles of both operands (moe_quant_fp8_128x1_*,
 * moe_grouped_wgrad_fp8). Order of calls, after a forward whose workspace
 * is still intact:
 *   moe_combine_backward -> moe_route_backward -> moe_router_wgrad;
 *   moe_grouped_gemm_fp8 (dO x W2^T blocks, MOE_EPI_F32) -> dh;
 *   moe_grouped_gemm_fp8 (x, W13, MOE_EPI_GATEUP_F32) -> a|b;
 *   moe_swiglu_backward; moe_grouped_gemm_fp8 ([dA|dB] x [W1|W3]^T blocks,
 *   MOE_EPI_BF16_F32_LAST); moe_dx_combine;
 *   moe_quant_fp8_128x1_* of dO, h, dA|dB, x; moe_grouped_wgrad_fp8 twice.
 * All calls: caller-owned device memory, asynchronous on `stream`, host
 * checks return before any launch, device checks set the status word.
 * ------------------------------------------------------------------------ */

/* Transposes 128x128-block E4M3 matrices with their scales (a block's codes
 * and scale carry over exactly):
 *   q      device u8 [batch][rows][cols], scale f32 [batch][rows/128][cols/128]
 *   qT     device u8, element (b, c, r) at qT[(b * colsT + c) * ldT + r]
 *   scaleT device f32, block (b, cb, rb) at scaleT[(b * colsT/128 + cb) * (ldT/128) + rb]
 * ldT >= rows lets two matrices share the rows of qT, e.g. W1^T and W3^T side
 * by side as the K order [W1 | W3] of the data gradient of the gate/up
 * projection; colsT >= cols leaves rows cols .. colsT-1 of each transposed
 * matrix untouched (zero padding the caller keeps, e.g. to a GEMM's N tile).
 * rows, cols, ldT, colsT multiples of 128. */
moe_status moe_transpose_fp8_blocks(const uint8_t* q, const float* scale, int64_t batch, int64_t rows, int64_t cols,
                                    uint8_t* qT, float* scaleT, int64_t ldT, int64_t colsT, void* stream);

/* Backward of moe_combine for upstream gradient dy (bf16 [T][d]):
 *   dgate[t][k] = sum_n dy[t][n] * routed_out[row_of[t][k]][n]   (FP32)
 *   the expert-output gradient of each grouped row, quantised per 1x128 tile:
 *   row row_of[t][k] holds g * dy[t] (g = topk_gate[t][k] > 0), shared row
 *   T*K + t holds dy[t]; codes dOq u8 [T*K+T][d], scales dOs f32 [T*K+T][d/128].
 *   MOE_SCALE_FP32: every row of token t takes the codes of dy[t]'s own tile
 *   and scale fl32(g * s) with s = fl32(amax/448) of that tile (the 1x128
 *   quantisation of g * dy, g scaling the tile uniformly);
 *   MOE_SCALE_POW2: fl32(g * dy[t]) quantised row by row (a power-of-two
 *   scale cannot absorb g);
 *   row_gate f32 [T*K+T]: the gate of each grouped row (1 for shared rows).
 * routed_out bf16 [T*K][d] (the forward's routed expert outputs); row_of,
 * topk_gate as in moe_combine. */
moe_status moe_combine_backward(const moe_config* cfg, const uint16_t* dy, const uint16_t* routed_out,
                                const int32_t* row_of, const float* topk_gate, int32_t rule, uint8_t* dOq, float* dOs,
                                float* row_gate, float* dgate, void* stream);

/* Router logit gradient of the chosen experts: with s_k the affinities the
 * forward's moe_route computed (recomputed bit for bit from the logits it
 * left in `workspace`, plus logit_offset if not NULL) and S = sum_k s_k,
 *   dz[t][k] = (dgate[t][k] - sum_j g_j dgate[t][j]) / S * s_k * (1 - s_k),
 * g_j = s_j / S. topk_idx, dgate, dz [T][K]. The workspace must be the one
 * the forward's moe_route used, unchanged since. */
moe_status moe_route_backward(const moe_config* cfg, const float* logit_offset, const int32_t* topk_idx,
                              const float* dgate, float* dz, void* workspace, size_t workspace_bytes, void* stream);

/* Router weight gradient: dWr[e][:] = sum over expert e's grouped rows r of
 * dz[t_r][k_r] * x[t_r][:] (FP32, in row order), with t_r = sorted_token[r]
 * and k_r the slot with row_of[t_r][k_r] == r. x bf16 [T][d]; offsets
 * [E+1] and sorted_token, row_of from moe_permute; dWr f32 [E][d] out. */
moe_status moe_router_wgrad(const moe_config* cfg, const uint16_t* x, const int32_t* offsets,
                            const int32_t* sorted_token, const int32_t* row_of, const float* dz, float* dWr,
                            void* stream);

/* SwiGLU backward of h = SiLU(a) * b, SiLU(a) = a * sigmoid(a):
 *   dA = dh * b * sigmoid(a) * (1 + a * (1 - sigmoid(a))),  dB = dh * SiLU(a).
 *   ab    f32 [rows][2I] in/out: in, a and b in the MOE_EPI_GATEUP_F32 layout;
 *         out, dA and dB in the same places
 *   dh    f32 [rows][ld_dh] (the first I columns are read; ld_dh % 4 == 0)
 *   dab_q u8 [rows][2I], dab_s f32 [rows][2I/128]: 1x128 E4M3 of [dA | dB]
 *         (dA in columns [0, I), dB in [I, 2I)) under scale rule `rule`.
 * I a multiple of 128. */
moe_status moe_swiglu_backward(int64_t rows, int32_t I, float* ab, const float* dh, int64_t ld_dh, int32_t rule,
                               uint8_t* dab_q, float* dab_s, void* stream);

/* Input gradient: dx[t] = dx_shared[t] + sum_k (dx_routed[row_of[t][k]] +
 * dz[t][k] * Wr[topk_idx[t][k]]), FP32 in that order, bf16 result.
 * dx_routed bf16 [T*K][d], dx_shared f32 [T][d] (the data-gradient GEMM's
 * MOE_EPI_BF16_F32_LAST outputs), Wr f32 [E][d], dx bf16 [T][d] out. */
moe_status moe_dx_combine(const moe_config* cfg, const uint16_t* dx_routed, const float* dx_shared,
                          const int32_t* row_of, const int32_t* topk_idx, const float* dz, const float* Wr, uint16_t* dx,
                          void* stream);

/* 128x1 grouped quantisation (the 1x128 rule taken along the rows) of a
 * [rows][cols] operand whose rows are grouped by offsets [groups+1]
 * (device i32, non-decreasing, offsets[groups] <= rows): group g's rows form
 * ceil(m_g/128) tiles of 128 rows (the last zero-padded); the s-th tile over
 * all groups in order becomes columns 128s .. 128s+127 of
 *   qT device u8 [cols][ldq]   (the codes, transposed: row c = channel c)
 *   sT device f32 [*][cols]    (scale of tile s, channel c at sT[s * cols + c])
 * ldq (a multiple of 16) must cover 128 * sum_g ceil(m_g/128), which is at
 * most 128 * (ceil(rows/128) + groups); a narrower ldq sets
 * MOE_ERR_DEVICE_CHECK. Padding codes are 0x00. cols a multiple of 128.
 * The sources differ in where the values come from:
 *   _f32       v f32 [rows][ld]
 *   _fp8       fl32(decode(q) * scale) of E4M3 codes q [rows][ld] with 1x128
 *              scales [rows][ld/128] (ld a multiple of 128): the values an FP8
 *              GEMM of the forward multiplied
 *   _bf16_rows fl32(row_mult[r] * x[row_map[r]][:]) of bf16 x [x_rows][ld]
 *              (row_mult NULL: 1), e.g. the grouped rows of the expert-output
 *              gradient g * dy. row_map values in [0, x_rows) (else
 *              MOE_ERR_DEVICE_CHECK and row 0). */
moe_status moe_quant_fp8_128x1_f32(const float* v, int64_t ld, int32_t groups, const int32_t* offsets, int64_t rows,
                                   int32_t cols, int32_t rule, uint8_t* qT, int64_t ldq, float* sT, void* stream);
moe_status moe_quant_fp8_128x1_fp8(const uint8_t* q, const float* scale, int64_t ld, int32_t groups,
                                   const int32_t* offsets, int64_t rows, int32_t cols, int32_t rule, uint8_t* qT,
                                   int64_t ldq, float* sT, void* stream);
moe_status moe_quant_fp8_128x1_bf16_rows(const uint16_t* x, int64_t x_rows, int64_t ld, const int32_t* row_map,
                                         const float* row_mult, int32_t groups, const int32_t* offsets, int64_t rows,
                                         int32_t cols, int32_t rule, uint8_t* qT, int64_t ldq, float* sT,
                                         void* stream);

/* Grouped weight-gradient GEMM on 5th-generation tensor cores: for each group g,
 *   out[g][m][n] = sum over g's 128-row tiles s of
 *                  saT[s][m] * sbT[s][n] * sum_{j < 128} AT[m][128s+j] * BT[n][128s+j]
 * (E4M3 operands from moe_quant_fp8_128x1_*, FP32 promotion per tile), with
 * g's tiles numbered as moe_quant_fp8_128x1_* numbers them for the same
 * offsets [groups+1] (device). AT u8 [M][width], BT u8 [N][width], saT f32
 * [width/128][M], sbT f32 [width/128][N]; out f32 [groups][M][N] (groups
 * with no rows get zeros). M a multiple of 128, N of 256, width (>= 128 *
 * sum_g ceil(m_g/128), else MOE_ERR_DEVICE_CHECK) of 128; groups <= 1025;
 * out 32-byte aligned. */
moe_status moe_grouped_wgrad_fp8(int32_t groups, const int32_t* offsets, int64_t rows, int64_t width, int32_t M,
                                 int32_t N, const uint8_t* AT, const float* saT, const uint8_t* BT, const float* sbT,
                                 float* out, void* stream);

/* ---------------------------------------------------------------------
 * Expert parallelism with node-limited routing (《DeepSeek-V3 Technical
 * Report》深度解读报告 §2.4: a token reaches at most M nodes, chosen by the
 * sum of their experts' highest affinities; §3.2: tokens cross nodes by
 * all-to-all, experts spread over the GPUs for prefill).
 * R ranks; rank r owns the E/R routed experts [r*E/R, (r+1)*E/R) (E % R ==
 * 0; with R dividing G a rank holds whole groups, so a token reaches at
 * most M ranks); every rank holds the router and the shared expert and
 * routes its own T tokens. A step on one rank:
 *   1. moe_route, moe_quant_fp8_1x128 of its tokens (token order);
 *   2. moe_ep_dispatch: each token's packed row (E4M3 codes, scales, choice,
 *      gates; moe_ep_row_bytes) once per destination rank, ordered by
 *      (rank, token), with per-rank counts (the all-to-all split sizes);
 *   3. all-to-all of the packed rows (the caller's collective);
 *   4. moe_ep_receive: the received pairs on this rank's experts, grouped
 *      by (local expert, received row), codes and scales gathered;
 *   5. moe_grouped_gemm_fp8 over the E/R local experts (gate/up + SwiGLU,
 *      then down with MOE_EPI_BF16), weights of experts r*E/R..;
 *   6. moe_ep_partial: per received row, the gate-weighted sum of its
 *      local expert outputs (FP32);
 *   7. the reverse all-to-all of the partial rows (received order);
 *   8. the shared expert on the rank's own tokens (grouped GEMM with one
 *      group, FP32 output), then moe_ep_combine.
 * The pages have no counterpart for these packing formats; the order of
 * rows is the library's own (stable sorts by rank and by local expert). */

/* Bytes of one packed dispatch row: d code bytes, d/128 FP32 scales, K
 * expert ids (i32), K gates (f32), zero padding to a multiple of 16. 0 for
 * d not a multiple of 128 or K outside 1..16. */
int64_t moe_ep_row_bytes(int32_t d, int32_t K);

/* Workspace bytes of moe_ep_dispatch (rows = cfg->T) and moe_ep_receive
 * (rows = received rows) for R ranks. 0 for an unsupported cfg or R. */
size_t moe_ep_workspace_size(const moe_config* cfg, int32_t R, int64_t rows);

/* Send side of the expert-parallel step.
 *   R            ranks, 1 <= R <= E, E % R == 0 (else MOE_ERR_UNSUPPORTED_SHAPE)
 *   topk_idx     device i32 [T][K], topk_gate f32 [T][K] (moe_route)
 *   xq, xs       device u8 [T][d], f32 [T][d/128] (moe_quant_fp8_1x128)
 *   send_counts  device i32 [R] out or NULL: rows for each rank
 *   send_offsets device i32 [R+1] out: exclusive prefix of send_counts;
 *                send_offsets[R] = S, the number of send rows
 *   send_row_of  device i32 [T][K] out: the send row of the token's first
 *                slot on each destination rank, -1 for later slots on the
 *                same rank
 *   send_token   device i32 [T*min(K,R)] out: token of each send row
 *   send_buf     device u8 [T*min(K,R)][moe_ep_row_bytes(d,K)] out: rows
 *                [0, S) written, ordered by (rank, token)
 *   workspace    device, >= moe_ep_workspace_size(cfg, R, T) bytes
 * Expert ids outside [0, E) set MOE_ERR_DEVICE_CHECK and are skipped. */
moe_status moe_ep_dispatch(const moe_config* cfg, int32_t R, const int32_t* topk_idx, const float* topk_gate,
                           const uint8_t* xq, const float* xs, int32_t* send_counts, int32_t* send_offsets,
                           int32_t* send_row_of, int32_t* send_token, uint8_t* send_buf,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Receive side: groups the received rows' pairs on this rank's experts.
 *   rank          0 <= rank < R; its experts are [rank*E/R, (rank+1)*E/R)
 *   n_recv        received packed rows (any order of source ranks)
 *   recv_buf      device u8 [n_recv][moe_ep_row_bytes(d,K)]
 *   local_offsets device i32 [E/R + 1] out: grouped rows of each local
 *                 expert; local_offsets[E/R] = P, the pairs this rank serves
 *   local_counts  device i32 [E/R] out or NULL
 *   sorted_row    device i32 [n_recv*K] out: received row of grouped row p < P
 *   row_of        device i32 [n_recv][K] out: grouped row of each (row, slot)
 *                 on this rank, -1 for slots served elsewhere
 *   xq_local      device u8 [n_recv*K][d] out, xs_local f32 [n_recv*K][d/128]
 *                 out: rows [0, P) in grouped order
 *   workspace     device, >= moe_ep_workspace_size(cfg, R, n_recv) bytes */
moe_status moe_ep_receive(const moe_config* cfg, int32_t R, int32_t rank, int64_t n_recv, const uint8_t* recv_buf,
                          int32_t* local_offsets, int32_t* local_counts, int32_t* sorted_row, int32_t* row_of,
                          uint8_t* xq_local, float* xs_local, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Per received row i: partial[i] = sum over slots k with row_of[i][k] >= 0,
 * in slot order, of gate[i][k] * routed_out[row_of[i][k]] (FP32 accumulation).
 *   routed_out device bf16 [out_rows][d] (the down GEMM's grouped rows;
 *              row_of values >= out_rows set MOE_ERR_DEVICE_CHECK)
 *   partial    device f32 [n_recv][d] out */
moe_status moe_ep_partial(const moe_config* cfg, int64_t n_recv, const uint8_t* recv_buf, const int32_t* row_of,
                          const uint16_t* routed_out, int64_t out_rows, float* partial, void* stream);

/* y[t] = shared_out[t] + sum over the token's send rows (send_row_of[t][k]
 * >= 0, slot order) of returned[row] (+ residual[t]), FP32 accumulation,
 * bf16 result.
 *   shared_out device f32 [T][d]; returned device f32 [S][d], the partial
 *   rows back from the ranks, in send order; residual bf16 [T][d] or NULL;
 *   y device bf16 [T][d] out */
moe_status moe_ep_combine(const moe_config* cfg, const float* shared_out, const float* returned, int64_t S,
                          const int32_t* send_row_of, const uint16_t* residual, uint16_t* y, void* stream);

/* Failure-detection self test: launches one kernel that waits, with a
 * limit of `limit_us` microseconds, on a barrier nothing will complete, and
 * reports through the device status word. Returns MOE_ERR_TIMEOUT (after a
 * stream synchronisation) when the bounded wait behaves. Blocking. */
moe_status moe_selftest_wait_timeout(uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
