// Internal launch functions behind the jetfp8 C ABI.  Arguments reaching these
// have been validated by the ABI layer (shapes, alignment, null pointers).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace jetfp8 {

inline int64_t round_up4(int64_t v) { return (v + 3) / 4 * 4; }

cudaError_t launch_quant_rowgroups(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t st);
cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                uint8_t* qT, cudaStream_t st);
// Q2 for `count` weights (1..JETFP8_MAX_GROUP) in one launch; qT may be NULL
// (no transposes) or hold NULL entries.
cudaError_t launch_quant_weight_grouped(int count, const void* const* w, const int64_t* N, const int64_t* K,
                                        uint8_t* const* q, float* const* s, uint8_t* const* qT,
                                        cudaStream_t st);
cudaError_t launch_requant_row2col(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                   uint8_t* qT, float* sT, cudaStream_t st);
cudaError_t launch_quant_grad_dual(const void* dy, int64_t M, int64_t N, uint8_t* q_row,
                                   float* s_row, uint8_t* qT_col, float* sT_col, cudaStream_t st);
cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t M,
                                 int64_t H, uint8_t* q, float* s, float* rstd, void* y,
                                 cudaStream_t st);
size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H);
cudaError_t launch_rmsnorm_bwd(const void* x, const void* gamma, const float* rstd, const void* dy,
                               int64_t M, int64_t H, void* dx, float* dgamma, float* ws,
                               cudaStream_t st);
cudaError_t launch_swiglu_quant(const void* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                void* h, cudaStream_t st);
cudaError_t launch_swiglu_bwd(const void* gu, const void* dh, int64_t M, int64_t I, void* dgu,
                              cudaStream_t st);

// Block-scaled GEMM  out[i,j] = Σ_kb sA[kb][i]·sB(kb,j)·Σ_{k in kb} A[i,k]·B[j,k]
// with A [R, Kc] and B [C, Kc] both K-major E4M3.
enum class BScale : int {
  kBlock = 0,   // sB(kb, j) = sB[(j/128)*sb_j + kb*sb_k]   (128×128 weight blocks)
  kColumn = 1,  // sB(kb, j) = sB[kb*sb_k + j]              (one scale per column and block)
};

struct GemmArgs {
  const uint8_t* A;
  const uint8_t* B;
  const float* sA;
  int64_t ld_sA;     // row stride of sA ([Kc/128][ld_sA])
  const float* sB;
  int64_t sb_j, sb_k;
  BScale b_mode;
  void* out;
  bool out_fp32;
  int64_t R, C, Kc;  // rows of A / out, rows of B = columns of out, contraction length
  // optional: 1×128 quantisation of the bf16 output fused into the epilogue
  // (uniform scales only, C a multiple of 256); codes [R, C], scales [C/128][ld_out_s]
  uint8_t* out_q = nullptr;
  float* out_s = nullptr;
  int64_t ld_out_s = 0;
  // test hook: the 128-deep block the TMA producer leaves unloaded (-1: none)
  int drop_kb = -1;
};

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st);
// Kernel choice for later GEMM launches: 0 automatic, 1 single-CTA tiles
// wherever possible, 2 CTA-pair tiles wherever possible.
void set_gemm_path(int mode);
// `count` (1..4) column-scale (WGrad) problems in one persistent launch; each
// problem's output equals that of its own launch_gemm, bit for bit.
cudaError_t launch_gemm_grouped(const GemmArgs* a, int count, cudaStream_t st);

// FP4 variant (NVFP4-style E2M1 codes, E4M3 scales per 16 elements in the
// blocked layout, FP32 row scales; nvfp4.cu).
size_t nvfp4_scale_bytes(int64_t R, int64_t K);
cudaError_t launch_quant_nvfp4(const void* x, int64_t R, int64_t K, uint8_t* q, uint8_t* sf, float* g,
                               cudaStream_t st);
cudaError_t launch_gemm_nvfp4(const uint8_t* xq, const uint8_t* xsf, const float* gx, const uint8_t* wq,
                              const uint8_t* wsf, const float* gw, int64_t M, int64_t N, int64_t K, void* y,
                              cudaStream_t st);

}  // namespace jetfp8
