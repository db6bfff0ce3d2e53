/*
 * jetfp8.h — C ABI of the GB300 (sm_103a) mixed-granularity E4M3 linear layer.
 *
 * The operations follow the Jet-RL pages:
 *   [digest]  "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习"
 *             (paper.rainbus.top), sections 前置知识 (FP8 量化 (E4M3 格式);
 *             GEMM 量化布局; Per-group / Per-block 量化粒度), 核心方法 and
 *             方法步骤详情 (steps 1-5).
 *   [summary] "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with
 *             Unified Training and Rollout Precision Flow" (sciencestack.ai),
 *             Figure 5 (the inference graph is a subgraph of the training graph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - E4M3 means the FN encoding (bias 7, no infinities, largest finite 448),
 *    stored one code per uint8_t.  Quantisation of a group:
 *        S = fp32(amax / 448)          (S = 1 when amax = 0)
 *        q = sat_rne_e4m3(fp32(x / S)) (round to nearest even, saturate to ±448,
 *                                       sign of zero kept)
 *    where both quotients are correctly rounded FP32 divisions.
 *  - All tensors are dense, row-major, unit inner stride.  bf16 data is passed
 *    as `const void*` holding IEEE bfloat16.
 *  - Scale arrays are FP32 and "group-index major": the scales of an [R, C]
 *    tensor quantised in 1×128 row groups are stored as S[g][r] with row
 *    stride ld = roundup(R, 4), i.e. an array of (C/128) × ld floats; padding
 *    entries are never read and may be left unwritten.
 *  - Every pointer argument is a DEVICE pointer owned by the caller and must
 *    stay valid until the work on `stream` completes.  bf16 tensors must be
 *    32-byte aligned (they move with 256-bit accesses); E4M3 and FP32 arrays
 *    16-byte aligned (JETFP8_ERR_MISALIGNED otherwise).  The
 *    library allocates no device memory and keeps no pointer after a call
 *    returns.  A null `stream` is the legacy default stream.
 *  - Shapes: every length named K, N, H or I must be a positive multiple of
 *    128.  M (tokens) may be any positive value unless an entry point says
 *    it must be a multiple of 128.
 *  - Calls are asynchronous on `stream`.  The returned status covers argument
 *    validation and the launch.  A kernel whose bounded wait expires records
 *    an error word on the device instead of hanging; read it with
 *    jetfp8_get_last_device_error() after synchronising.
 *  - Outputs must not alias inputs.  No C++ exception crosses this boundary.
 *    NaN or infinite inputs are outside the contract.
 */
#ifndef JETFP8_H_
#define JETFP8_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_H__
typedef struct CUstream_st* cudaStream_t;  /* same type as the CUDA runtime's */
#endif

typedef enum {
  JETFP8_OK = 0,
  JETFP8_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, bad enum */
  JETFP8_ERR_UNSUPPORTED_SHAPE = 2, /* a length violates the multiple-of-128 rules */
  JETFP8_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rule above */
  JETFP8_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  JETFP8_ERR_TIMEOUT = 5,           /* a device-side bounded wait expired */
  JETFP8_ERR_UNSUPPORTED = 6        /* device is not sm_103, or feature not built */
} jetfp8_status;

typedef enum { JETFP8_OUT_BF16 = 0, JETFP8_OUT_FP32 = 1 } jetfp8_out_dtype;

/* Human-readable name of a status code (static string, never null). */
const char* jetfp8_status_string(jetfp8_status st);

/* Synchronises `stream`, returns JETFP8_ERR_TIMEOUT if any kernel of this
 * library on the current device recorded an expired bounded wait since the
 * last call (and clears the record), else JETFP8_OK (or JETFP8_ERR_CUDA). */
jetfp8_status jetfp8_get_last_device_error(cudaStream_t stream);

/* Q1 — 1×128 per-group activation quantisation ([digest] 方法步骤详情, steps 1-2;
 * 前置知识 › Per-group / Per-block 量化粒度).
 *   x  bf16 [M, K]
 *   q  E4M3 [M, K]           (row groups of 128 consecutive elements)
 *   s  fp32 [K/128][roundup(M,4)]
 * M arbitrary, K multiple of 128. */
jetfp8_status jetfp8_quant_act_1x128(const void* x_bf16, int64_t M, int64_t K,
                                     uint8_t* q, float* s, cudaStream_t stream);

/* Q2 — 128×128 per-block weight quantisation ([digest] 方法步骤详情, step 1), with
 * the optional transposed payload that DGrad consumes (step 4: the weight's
 * quantisation is reused between passes, only transposed).
 *   w   bf16 [N, K]
 *   q   E4M3 [N, K]
 *   s   fp32 [N/128][K/128]   (one scale per block; serves q and qT)
 *   qT  E4M3 [K, N] or NULL  (qT[k][n] == q[n][k])
 * N and K multiples of 128. */
jetfp8_status jetfp8_quant_weight_128x128(const void* w_bf16, int64_t N, int64_t K,
                                          uint8_t* q, float* s, uint8_t* qT,
                                          cudaStream_t stream);

/* Q3 — requantise the FP8-saved activation from 1×128 row groups to 128×1
 * column groups, written transposed, for WGrad ([digest] 方法步骤详情, step 4;
 * 技术新颖性).  x̃ = fp32(dec(q)·S_row) (one FP32 multiply), then each column's
 * 128-token group is quantised with its own scale.
 *   q   E4M3 [M, K],  s  fp32 [K/128][M]          (output of Q1 or R1)
 *   qT  E4M3 [K, M],  sT fp32 [M/128][K]
 * M and K multiples of 128. */
jetfp8_status jetfp8_requant_rowgrp_to_colgrp(const uint8_t* q, const float* s,
                                              int64_t M, int64_t K, uint8_t* qT,
                                              float* sT, cudaStream_t stream);

/* Q4 — gradient quantisation from one read of the BF16 ∇Y ([digest]
 * 方法步骤详情, step 4: ∇Y stays BF16; gradients use 1×128 groups):
 *   dy      bf16 [M, N]
 *   q_row   E4M3 [M, N],  s_row  fp32 [N/128][roundup(M,4)]  (groups along N, for DGrad)
 *   qT_col  E4M3 [N, M],  sT_col fp32 [M/128][N]             (128-token groups, transposed,
 *                                                            for WGrad) — both NULL or both set
 * N multiple of 128; M multiple of 128 when qT_col is set, else arbitrary. */
jetfp8_status jetfp8_quant_grad_dual(const void* dy_bf16, int64_t M, int64_t N,
                                     uint8_t* q_row, float* s_row, uint8_t* qT_col,
                                     float* sT_col, cudaStream_t stream);

/* R1 — RMSNorm fused with the 1×128 quantiser ([digest] 方法步骤详情, step 5).
 *   r = 1/sqrt(mean(x²) + eps),  y = bf16((x·r)·γ),  then Q1 on y.
 *   y is evaluated in FP32 and lies within one bf16 ulp of the exact value (rows
 *   up to 8192 wide form RN(RN(x·γ)·r), x·γ exact for |x·γ| in the normal FP32
 *   range); the codes and scales are exactly Q1's on the returned y.
 *   x      bf16 [M, H],  gamma bf16 [H]
 *   q      E4M3 [M, H],  s fp32 [H/128][roundup(M,4)]
 *   rstd   fp32 [M]      (kept for the backward)
 *   y_bf16 bf16 [M, H] or NULL (the normalised output, for checking)
 * H multiple of 128, M arbitrary, eps >= 0. */
jetfp8_status jetfp8_rmsnorm_quant(const void* x_bf16, const void* gamma_bf16, float eps,
                                   int64_t M, int64_t H, uint8_t* q, float* s, float* rstd,
                                   void* y_bf16, cudaStream_t stream);

/* F1 — FProp Y = X̂·Ŵᵀ with (1×128)×(128×128) scales and FP32 accumulation
 * ([digest] 核心方法; 方法步骤详情, step 2; 前置知识 › GEMM 量化布局):
 *   Y[m,n] = Σ_kb sx[kb][m]·sw[n/128][kb]·Σ_{k in kb} dec(xq[m,k])·dec(wq[n,k])
 *   xq E4M3 [M, K], sx fp32 [K/128][roundup(M,4)]
 *   wq E4M3 [N, K], sw fp32 [N/128][K/128]
 *   y  bf16 or fp32 [M, N] per `out_dtype`
 * Used unchanged for rollout (decode-sized M) and training, so both see the
 * same quantised graph ([summary] Figure 5).  M arbitrary. */
jetfp8_status jetfp8_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream);

/* F2 — DGrad ∇X = ∇Ŷ·Ŵ, reusing FProp's configuration with the transposed
 * weight payload ([digest] 核心方法; 方法步骤详情, step 4):
 *   dX[m,k] = Σ_nb sdy[nb][m]·sw[nb][k/128]·Σ_{n in nb} dec(dyq[m,n])·dec(wqT[k,n])
 *   dyq E4M3 [M, N], sdy fp32 [N/128][roundup(M,4)]   (Q4 row output)
 *   wqT E4M3 [K, N], sw  fp32 [N/128][K/128]          (Q2 outputs)
 *   dx  bf16 or fp32 [M, K].  M arbitrary. */
jetfp8_status jetfp8_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT,
                                const float* sw, int64_t M, int64_t N, int64_t K, void* dx,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream);

/* F3 — WGrad ∇W = ∇Ŷᵀ·X̂ with (1×128)×(128×1) scales: the contraction runs
 * over tokens and both operands carry one scale per 128 tokens ([digest]
 * 核心方法; 方法步骤详情, step 4):
 *   dW[n,k] = Σ_tb sdyT[tb][n]·sxT[tb][k]·Σ_{m in tb} dec(dyqT[n,m])·dec(xqT[k,m])
 *   dyqT E4M3 [N, M], sdyT fp32 [M/128][N]   (Q4 column output)
 *   xqT  E4M3 [K, M], sxT  fp32 [M/128][K]   (Q3 output)
 *   dw   bf16 or fp32 [N, K].  M multiple of 128. */
jetfp8_status jetfp8_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                const float* sxT, int64_t M, int64_t N, int64_t K, void* dw,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream);

/* F3 for up to JETFP8_MAX_GROUP linear layers at once (the operation is F3's,
 * [digest] 核心方法; 方法步骤详情, step 4; grouping them is a scheduling choice
 * the pages do not discuss): the WGrads of the linears of one layer (they share
 * the token count M and do not depend on one another) in one persistent launch,
 * so the tiles of one fill the last wave of another.  Problem i is the jetfp8_gemm_wgrad call
 *   (dyqT[i], sdyT[i], xqT[i], sxT[i], M, N[i], K[i], dw[i], out_dtype)
 * and its output equals that call's bit for bit (the same 128-token blocks in
 * the same order for every element).  dyqT, sdyT, xqT, sxT, N, K and dw are
 * HOST arrays of `count` entries; the pointers they hold are device pointers
 * with the layouts and alignment of jetfp8_gemm_wgrad.  Outputs must not
 * overlap one another or any input.  1 <= count <= JETFP8_MAX_GROUP, else
 * JETFP8_ERR_INVALID_ARG; shape errors as jetfp8_gemm_wgrad.  The arrays are
 * read before the call returns; the launch is asynchronous on `stream`. */
#define JETFP8_MAX_GROUP 4
jetfp8_status jetfp8_gemm_wgrad_grouped(int count, const uint8_t* const* dyqT,
                                        const float* const* sdyT, const uint8_t* const* xqT,
                                        const float* const* sxT, int64_t M, const int64_t* N,
                                        const int64_t* K, void* const* dw,
                                        jetfp8_out_dtype out_dtype, cudaStream_t stream);

/* Q2 for up to JETFP8_MAX_GROUP weights at once (the operation is Q2's,
 * [digest] 方法步骤详情, step 1; grouping is a scheduling choice the pages do not
 * discuss): the weights a step quantises together, e.g. the four linears of a
 * layer, in one persistent launch, so the pipeline fills and drains once.
 * Problem i is the jetfp8_quant_weight_128x128 call
 *   (w_bf16[i], N[i], K[i], q[i], s[i], qT ? qT[i] : NULL)
 * and its outputs equal that call's bit for bit.  w_bf16, N, K, q, s and qT are
 * HOST arrays of `count` entries (qT itself may be NULL: no transposes; an
 * entry may be NULL: none for that weight); the pointers they hold are device
 * pointers with the layouts and alignment of jetfp8_quant_weight_128x128.
 * Outputs must not overlap one another or any input.  1 <= count <=
 * JETFP8_MAX_GROUP, else JETFP8_ERR_INVALID_ARG; shape errors as the single
 * call.  The arrays are read before the call returns; the launch is
 * asynchronous on `stream`. */
jetfp8_status jetfp8_quant_weight_grouped(int count, const void* const* w_bf16, const int64_t* N,
                                          const int64_t* K, uint8_t* const* q, float* const* s,
                                          uint8_t* const* qT, cudaStream_t stream);

/* F1 and F2 with the 1×128 quantiser fused into the epilogue ([digest] 方法步骤详情,
 * step 5: the quantisation is fused into the neighbouring kernels to cut its
 * overhead).  The output tile is rounded to bf16 as by jetfp8_gemm_fprop /
 * jetfp8_gemm_dgrad and quantised in 1×128 groups along its columns exactly as
 * by jetfp8_quant_act_1x128 applied to that bf16 output (the same codes and
 * scales, bit for bit), so the next linear's input comes straight from the GEMM:
 *   y_bf16 bf16 [M, N] or NULL (codes only)
 *   yq     E4M3 [M, N],  ys fp32 [N/128][roundup(M,4)]
 * Arguments otherwise as jetfp8_gemm_fprop (F1) and jetfp8_gemm_dgrad (F2,
 * output [M, K]).  The output width (N for F1, K for F2) must be a multiple of
 * 256: JETFP8_ERR_UNSUPPORTED_SHAPE otherwise.  M arbitrary. */
jetfp8_status jetfp8_gemm_fprop_quant(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                      const float* sw, int64_t M, int64_t N, int64_t K,
                                      void* y_bf16, uint8_t* yq, float* ys, cudaStream_t stream);
jetfp8_status jetfp8_gemm_dgrad_quant(const uint8_t* dyq, const float* sdy, const uint8_t* wqT,
                                      const float* sw, int64_t M, int64_t N, int64_t K,
                                      void* dx_bf16, uint8_t* dxq, float* dxs, cudaStream_t stream);

/* Test hook for the failure path (no counterpart on the pages).  As
 * jetfp8_gemm_fprop with a bf16 output, except that the kernel's TMA producer
 * never loads 128-deep block `drop_kb` (0 <= drop_kb < K/128, else
 * JETFP8_ERR_INVALID_ARG): the tensor core's bounded wait for that block's data
 * runs out (about 2 s), the kernel records JETFP8_ERR_TIMEOUT in the device error
 * word, lets the copies and MMAs in flight land, frees its TMEM and returns, and
 * the CUDA context stays usable.  y is left undefined.  The call itself returns
 * JETFP8_OK once launched; jetfp8_get_last_device_error reports the timeout. */
jetfp8_status jetfp8_test_gemm_fprop_drop_block(const uint8_t* xq, const float* sx,
                                               const uint8_t* wq, const float* sw, int64_t M,
                                               int64_t N, int64_t K, void* y, int drop_kb,
                                               cudaStream_t stream);

/* Test and diagnosis knob (no counterpart on the pages).  Chooses the kernel
 * of later GEMM launches of this process: 0 (the default) and 1 run every
 * GEMM on single-CTA tiles, 2 runs every GEMM that allows it (at least 256
 * rows of output, output width a multiple of 256, no fused output quantiser)
 * on CTA-pair tiles (tcgen05 cta_group::2, 256 x 256 per pair), which are
 * slower on GB300 and therefore not chosen by default.  Every output
 * element's arithmetic is the same on either kernel, so the results are
 * identical bit for bit; the knob lets tests check that.  Not synchronised with launches
 * in flight on other host threads.  Returns JETFP8_ERR_INVALID_ARG for any
 * other mode. */
jetfp8_status jetfp8_test_set_gemm_path(int mode);

/* ---------------------------------------------------------------------------
 * FP4 variant of the precision flow (next row N4).  The digest names carrying
 * the unified precision flow to FP4 on Blackwell as future work ([digest]
 * 未来方向, item (1)) and defines no FP4 format; this variant keeps the flow's
 * property that a token's forward result does not depend on its batch
 * ([summary] Figure 5), on the NVFP4-style format the tensor cores scale in
 * hardware (tcgen05.mma kind::mxf4nvf4, block scales applied by the MMA):
 *   codes  E2M1 (sign, 2 exponent bits, 1 mantissa bit; magnitudes 0, 0.5, 1,
 *          1.5, 2, 3, 4, 6), two per byte, element 2i in the low nibble:
 *          uint8 [R, K/2], row-major;
 *   block scales  one E4M3 code per 16 consecutive elements of a row, in the
 *          blocked layout: byte ((r/128·K/64 + b/4)·32 + r mod 32)·16 +
 *          ((r/32) mod 4)·4 + b mod 4 for row r, block b (512-byte atoms of
 *          128 rows × 64 elements); jetfp8_nvfp4_scale_bytes(R, K) bytes,
 *          rows past R inside the last atom carry zero scales;
 *   row scales  FP32 [R], one per row (token of X, output channel of W).
 * Rule, every step one correctly rounded FP32 operation:
 *   g = amax_row/2688 (1 if the row is zero), h = 6·g,
 *   s_b = E4M3(amax_b/h) (round to nearest even, saturating at 448),
 *   d_b = s_b·g,  q = E2M1(x/d_b) (nearest even, saturating at ±6; a zero
 *   with the sign of x when d_b = 0).
 * ------------------------------------------------------------------------- */

/* Bytes of the block-scale array for R rows of K elements (K a multiple of
 * 64): ceil(R/128)·(K/64)·512; 0 for invalid sizes. */
size_t jetfp8_nvfp4_scale_bytes(int64_t R, int64_t K);

/* Quantise the bf16 rows x [R, K] (K a multiple of 64; 32-byte aligned) to the
 * FP4 variant: codes q [R, K/2], block scales sf (blocked layout above) and row
 * scales g [R] (all 16-byte aligned, caller-owned; the call writes every byte
 * of q, sf and g, padding-row scales included).  A row's result depends only
 * on that row.  Errors: JETFP8_ERR_INVALID_ARG (null pointer, R <= 0),
 * JETFP8_ERR_UNSUPPORTED_SHAPE (K not a multiple of 64, or too large),
 * JETFP8_ERR_MISALIGNED, JETFP8_ERR_CUDA / JETFP8_ERR_UNSUPPORTED (no sm_103 device). */
jetfp8_status jetfp8_quant_nvfp4(const void* x_bf16, int64_t R, int64_t K, uint8_t* q, uint8_t* sf,
                                 float* g, cudaStream_t stream);

/* FP4 forward GEMM  Y[m,n] = bf16(RN(RN(D[m,n]·gx[m])·gw[n])),
 *   D[m,n] = Σ_k dec(xq[m,k])·dec(xsf[m,k/16])·dec(wq[n,k])·dec(wsf[n,k/16]),
 * accumulated in FP32 by the tensor core (block scales applied in the MMA).
 * xq [M, K/2], xsf, gx [M] from jetfp8_quant_nvfp4 of X; wq [N, K/2], wsf, gw [N]
 * from jetfp8_quant_nvfp4 of W; y bf16 [M, N] (caller-owned, 16-byte aligned).
 * N and K multiples of 256.  Errors as jetfp8_quant_nvfp4; a device-side
 * timeout is reported by jetfp8_get_last_device_error. */
jetfp8_status jetfp8_gemm_fprop_nvfp4(const uint8_t* xq, const uint8_t* xsf, const float* gx,
                                      const uint8_t* wq, const uint8_t* wsf, const float* gw, int64_t M,
                                      int64_t N, int64_t K, void* y_bf16, cudaStream_t stream);

/* Set the environment variable JETFP8_LOG (to anything but "" or "0") and every
 * entry point prints its name and sizes to stderr when called. */

/* RMSNorm backward, for the decoder layer around the quantised linears (the
 * pages fuse the forward only; this is the exact derivative of R1's
 * y = (x·r)·γ, r = 1/sqrt(mean(x²) + eps), using the r that R1 saved):
 *   ∇x_i = r·(dy_i·γ_i) − x_i·r³·(Σ_j dy_j·γ_j·x_j)/H       (FP32, rounded to bf16)
 *   ∇γ_j = Σ_rows dy_j·x_j·r                                 (deterministic on a given
 *          GPU: rows up to 4096 wide — FP32 sums over the rows each warp of a
 *          persistent CTA owns, the CTA's 8 warps added in warp order in FP32, the
 *          CTAs' sums added in a fixed order in FP64; wider rows — FP32 sums over
 *          128-row chunks, chunks added in a fixed order in FP64)
 *   x bf16 [M, H], gamma bf16 [H], rstd fp32 [M] (R1's output), dy bf16 [M, H]
 *   dx bf16 [M, H], dgamma fp32 [H]
 *   workspace: caller-owned device memory of at least
 *              jetfp8_rmsnorm_bwd_workspace_bytes(M, H) bytes (16-byte aligned),
 *              overwritten by the call; JETFP8_ERR_INVALID_ARG if smaller.  The
 *              size is min(ceil(M/8), 152)·H·4 bytes for H <= 4096 and
 *              ceil(M/128)·H·4 bytes for wider rows.
 * H multiple of 128, M >= 1. */
size_t jetfp8_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H);
jetfp8_status jetfp8_rmsnorm_bwd(const void* x_bf16, const void* gamma_bf16, const float* rstd,
                                 const void* dy_bf16, int64_t M, int64_t H, void* dx_bf16,
                                 float* dgamma, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* jetfp8_rmsnorm_bwd without a workspace argument: the library's own scratch
 * is a fixed device array of 8 MiB per device (created with the library, no
 * allocation at the call), so this entry point allocates nothing.  The pages
 * have no counterpart; it exists for callers that cannot hand the library
 * memory.  Results equal jetfp8_rmsnorm_bwd's bit for bit.
 *   Arguments as jetfp8_rmsnorm_bwd without workspace / workspace_bytes.
 *   JETFP8_ERR_UNSUPPORTED_SHAPE when jetfp8_rmsnorm_bwd_workspace_bytes(M, H)
 *   exceeds 8 MiB, which only rows wider than 4096 can reach (ceil(M/128)·H·4
 *   bytes; e.g. M <= 16384 rows at H = 16384, M <= 32768 at H = 8192).
 *   All calls share the one scratch array: calls that overlap in time (on
 *   other streams or from other host threads) race and must be serialised by
 *   the caller; calls on one stream are ordered and safe. */
jetfp8_status jetfp8_rmsnorm_bwd_noalloc(const void* x_bf16, const void* gamma_bf16, const float* rstd,
                                         const void* dy_bf16, int64_t M, int64_t H, void* dx_bf16,
                                         float* dgamma, cudaStream_t stream);

/* X1 — SwiGLU fused with the 1×128 quantiser, for the decoder MLP between the
 * gate/up and down projections (not described by the pages):
 *   h = bf16(silu(g)·u), silu(g) = g/(1+exp(-g)), in FP32 with the fast
 *   exponential and division (errors of a few FP32 ulps, below the bf16
 *   rounding of h); then Q1 on h, exactly as jetfp8_quant_act_1x128 on h.
 *   gu     bf16 [M, 2I]  (gate in columns [0,I), up in [I,2I))
 *   q      E4M3 [M, I],  s fp32 [I/128][roundup(M,4)]
 *   h_bf16 bf16 [M, I] or NULL
 * I multiple of 128, M arbitrary. */
jetfp8_status jetfp8_swiglu_quant(const void* gu_bf16, int64_t M, int64_t I, uint8_t* q,
                                  float* s, void* h_bf16, cudaStream_t stream);

/* X2 — SwiGLU backward: with σ = 1/(1+exp(-g)),
 *   ∇g = ∇h·u·σ·(1 + g·(1-σ)),  ∇u = ∇h·g·σ, in FP32, rounded once to bf16.
 *   gu  bf16 [M, 2I],  dh bf16 [M, I]  ->  dgu bf16 [M, 2I] = [∇g | ∇u]
 * I multiple of 128, M arbitrary. */
jetfp8_status jetfp8_swiglu_bwd(const void* gu_bf16, const void* dh_bf16, int64_t M,
                                int64_t I, void* dgu_bf16, cudaStream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* JETFP8_H_ */
