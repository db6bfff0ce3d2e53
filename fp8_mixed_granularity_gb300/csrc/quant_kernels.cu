// Memory-bound quantisation kernels of the mixed-granularity E4M3 linear layer.
//
// Jet-RL digest ("Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习"):
//   前置知识 › FP8 量化 (E4M3 格式)       — S = max|x|/448, x̂ = E4M3(x/S)
//   前置知识 › Per-group / Per-block 量化粒度 — 1×128 groups for activations and
//                                          gradients, 128×128 blocks for weights
//   方法步骤详情, steps 1-5              — where each quantiser sits in the layer
//
// All of them stream HBM once.  Loads and stores are 8 or 16 bytes per lane and
// coalesced within a warp; grids are a multiple of the SM count and walk the
// work with a grid stride.
#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"

namespace jetfp8 {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Half-warp (16-lane) max-reduction; every lane of the half gets the result.
__device__ __forceinline__ float halfwarp_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return v;
}

// Quantise the 8 values of one lane (a 16-byte slice of a 128-wide group whose
// other 15 slices sit in the neighbouring lanes of the same half-warp).
// Returns the 8 codes as two words; `S` receives the group scale.
__device__ __forceinline__ uint2 quant_slice8(const float f[8], bool valid, float& S) {
  float amax = 0.0f;
  if (valid) {
#pragma unroll
    for (int j = 0; j < 8; j += 4) amax = absmax4(amax, f[j], f[j + 1], f[j + 2], f[j + 3]);
  }
  amax = halfwarp_max(amax);
  GroupScale g = make_scale(amax);
  S = g.s;
  uint2 r;
  r.x = quant4(f[0], f[1], f[2], f[3], g);
  r.y = quant4(f[4], f[5], f[6], f[7], g);
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  float2 a = bf2_to_f2(v.x), b = bf2_to_f2(v.y), c = bf2_to_f2(v.z), d = bf2_to_f2(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// ---------------------------------------------------------------------------
// Q1: 1×128 row groups.  The tensor is a contiguous run of groups (group g =
// bytes [256g, 256g+256) of the bf16 input), so a half-warp takes one group and
// a warp takes two neighbouring ones: each lane loads 16 B, fully coalesced.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(kThreads)
k_quant_rowgroups(const uint16_t* __restrict__ x, uint32_t n_groups, uint32_t groups_per_row,
                  uint32_t ld_s, uint8_t* __restrict__ q, float* __restrict__ s) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t hl = lane & 15u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  for (uint32_t base = warp * 2u * U; base < n_groups; base += nwarps * 2u * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t g = base + 2u * u + (lane >> 4);
      v[u] = g < n_groups ? ldg_stream(x + (size_t)g * 128 + hl * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t g = base + 2u * u + (lane >> 4);
      float f[8];
      unpack8(v[u], f);
      float S;
      uint2 codes = quant_slice8(f, g < n_groups, S);
      if (g < n_groups) {
        *reinterpret_cast<uint2*>(q + (size_t)g * 128 + hl * 8) = codes;
        if (hl == 0) s[(size_t)(g % groups_per_row) * ld_s + g / groups_per_row] = S;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 128×128 tile helpers.  Thread t of 256 owns an 8×8 sub-block of the tile:
// rows 8·(t/16) .. +8, columns 8·(t%16) .. +8.  For a fixed row, the 16 lanes
// of a half-warp cover the tile's 128 columns (coalesced 256 B bf16 / 128 B
// fp8 rows); the 16 threads that share a column set span all 8 warps.
// ---------------------------------------------------------------------------
struct TileCoord {
  uint32_t r0;  // first row of this thread's 8×8 sub-block within the tile
  uint32_t c0;  // first column
};
__device__ __forceinline__ TileCoord tile_coord() {
  return {8u * (threadIdx.x >> 4), 8u * (threadIdx.x & 15u)};
}

// Column max over the 128 rows of the tile: colmax_in[8] are this thread's
// maxima over its 8 rows; the result for its 8 columns is returned in place.
// `red` is shared scratch [16 row groups][128 columns].
__device__ __forceinline__ void tile_colmax(float cm[8], float (*red)[128]) {
  const uint32_t rowgrp = threadIdx.x >> 4;       // 0..15
  const uint32_t c0 = 8u * (threadIdx.x & 15u);
#pragma unroll
  for (int j = 0; j < 8; ++j) red[rowgrp][c0 + j] = cm[j];
  __syncthreads();
  if (threadIdx.x < 128) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, red[i][threadIdx.x]);
    red[0][threadIdx.x] = m;   // row 0 was read by this same thread above
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 8; ++j) cm[j] = red[0][c0 + j];
}

// Quantise an 8×8 sub-block column-wise (one scale per column, scales[j]) and
// store it transposed: output row (col0 + j), columns row0 .. row0+7.
__device__ __forceinline__ void store_cols_transposed(const float v[8][8], const GroupScale gs[8],
                                                      uint8_t* __restrict__ outT, size_t ld_out,
                                                      size_t out_row0, size_t out_col0) {
  // codes of row i, columns 0..7 -> lo/hi words, then transpose bytes
  uint32_t lo[8], hi[8], olo[8], ohi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo[i] = cvt_e4m3x2(quotient(v[i][0], gs[0]), quotient(v[i][1], gs[1])) |
            (cvt_e4m3x2(quotient(v[i][2], gs[2]), quotient(v[i][3], gs[3])) << 16);
    hi[i] = cvt_e4m3x2(quotient(v[i][4], gs[4]), quotient(v[i][5], gs[5])) |
            (cvt_e4m3x2(quotient(v[i][6], gs[6]), quotient(v[i][7], gs[7])) << 16);
  }
  transpose8x8(lo, hi, olo, ohi);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint2*>(outT + (out_row0 + j) * ld_out + out_col0) = make_uint2(olo[j], ohi[j]);
}

// ---------------------------------------------------------------------------
// Q2: 128×128 weight blocks, optional transposed payload.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_quant_weight(const uint16_t* __restrict__ w, uint32_t N, uint32_t K, uint8_t* __restrict__ q,
               float* __restrict__ s, uint8_t* __restrict__ qT) {
  __shared__ float wmax[kThreads / 32];
  const uint32_t kblocks = K / 128, nblocks = N / 128;
  const TileCoord tc = tile_coord();
  for (uint32_t blk = blockIdx.x; blk < kblocks * nblocks; blk += gridDim.x) {
    const uint32_t nb = blk / kblocks, kb = blk % kblocks;
    const size_t row0 = (size_t)nb * 128 + tc.r0, col0 = (size_t)kb * 128 + tc.c0;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ldg_stream(w + (row0 + i) * K + col0);
    float f[8][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      unpack8(v[i], f[i]);
      amax = absmax4(amax, f[i][0], f[i][1], f[i][2], f[i][3]);
      amax = absmax4(amax, f[i][4], f[i][5], f[i][6], f[i][7]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = wmax[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
    __syncthreads();   // wmax is reused by the next block
    const GroupScale g = make_scale(amax);
    if (threadIdx.x == 0) s[(size_t)nb * kblocks + kb] = g.s;
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo[i] = quant4(f[i][0], f[i][1], f[i][2], f[i][3], g);
      hi[i] = quant4(f[i][4], f[i][5], f[i][6], f[i][7], g);
      *reinterpret_cast<uint2*>(q + (row0 + i) * K + col0) = make_uint2(lo[i], hi[i]);
    }
    if (qT != nullptr) {
      uint32_t olo[8], ohi[8];
      transpose8x8(lo, hi, olo, ohi);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint2*>(qT + (col0 + j) * N + row0) = make_uint2(olo[j], ohi[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Q3: dequantise 1×128 row groups, requantise 128×1 column groups, transpose.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_requant_row2col(const uint8_t* __restrict__ q, const float* __restrict__ s, uint32_t M,
                  uint32_t K, uint8_t* __restrict__ qT, float* __restrict__ sT) {
  __shared__ float red[16][128];
  const uint32_t kblocks = K / 128, mblocks = M / 128;
  const TileCoord tc = tile_coord();
  for (uint32_t blk = blockIdx.x; blk < kblocks * mblocks; blk += gridDim.x) {
    const uint32_t mb = blk / kblocks, kb = blk % kblocks;
    const size_t row0 = (size_t)mb * 128 + tc.r0, col0 = (size_t)kb * 128 + tc.c0;
    uint2 c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = *reinterpret_cast<const uint2*>(q + (row0 + i) * K + col0);
    const float4 s_lo = *reinterpret_cast<const float4*>(s + (size_t)kb * M + row0);
    const float4 s_hi = *reinterpret_cast<const float4*>(s + (size_t)kb * M + row0 + 4);
    const float srow[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
    float v[8][8];
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cm[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        uint32_t w = (j < 4 ? c[i].x : c[i].y) >> (8 * (j & 3));
        float2 d = dec_e4m3x2(w & 0xFFFFu);
        v[i][j] = __fmul_rn(d.x, srow[i]);
        v[i][j + 1] = __fmul_rn(d.y, srow[i]);
        cm[j] = fmaxf(cm[j], fabsf(v[i][j]));
        cm[j + 1] = fmaxf(cm[j + 1], fabsf(v[i][j + 1]));
      }
    }
    tile_colmax(cm, red);
    GroupScale gs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) gs[j] = make_scale(cm[j]);
    if (tc.r0 == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) sT[(size_t)mb * K + col0 + j] = gs[j].s;
    }
    store_cols_transposed(v, gs, qT, M, col0, row0);
    __syncthreads();   // `red` is reused by the next tile
  }
}

// ---------------------------------------------------------------------------
// Q4: one read of the bf16 gradient, row groups along N and 128-token column
// groups (transposed).  M must be a multiple of 128.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_quant_grad_dual(const uint16_t* __restrict__ dy, uint32_t M, uint32_t N, uint32_t ld_srow,
                  uint8_t* __restrict__ q_row, float* __restrict__ s_row,
                  uint8_t* __restrict__ qT_col, float* __restrict__ sT_col) {
  __shared__ float red[16][128];
  const uint32_t nblocks = N / 128, mblocks = M / 128;
  const TileCoord tc = tile_coord();
  for (uint32_t blk = blockIdx.x; blk < nblocks * mblocks; blk += gridDim.x) {
    const uint32_t mb = blk / nblocks, nb = blk % nblocks;
    const size_t row0 = (size_t)mb * 128 + tc.r0, col0 = (size_t)nb * 128 + tc.c0;
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = ldg_stream(dy + (row0 + i) * N + col0);
    float v[8][8];
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cm[j] = 0.0f;
    float srow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      unpack8(raw[i], v[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) cm[j] = fmaxf(cm[j], fabsf(v[i][j]));
      // (i) the row group of row i: 128 columns across the half-warp
      uint2 codes = quant_slice8(v[i], true, srow[i]);
      *reinterpret_cast<uint2*>(q_row + (row0 + i) * N + col0) = codes;
    }
    if (tc.c0 == 0) {
      *reinterpret_cast<float4*>(s_row + (size_t)nb * ld_srow + row0) =
          make_float4(srow[0], srow[1], srow[2], srow[3]);
      *reinterpret_cast<float4*>(s_row + (size_t)nb * ld_srow + row0 + 4) =
          make_float4(srow[4], srow[5], srow[6], srow[7]);
    }
    // (ii) the column groups of the tile
    tile_colmax(cm, red);
    GroupScale gs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) gs[j] = make_scale(cm[j]);
    if (tc.r0 == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) sT_col[(size_t)mb * N + col0 + j] = gs[j].s;
    }
    store_cols_transposed(v, gs, qT_col, M, col0, row0);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// R1: RMSNorm fused with the 1×128 quantiser.  One warp per row; a half-warp
// per 128-wide group.  Pass 1 accumulates Σx² (FP32 per lane, then FP64 across
// lanes); pass 2 re-reads the row (an L1/L2 hit) and writes y, q and S.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_rmsnorm_quant(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps,
                uint32_t M, uint32_t H, uint32_t ld_s, uint8_t* __restrict__ q,
                float* __restrict__ s, float* __restrict__ rstd, uint16_t* __restrict__ y) {
  const uint32_t lane = threadIdx.x & 31u, hl = lane & 15u, half = lane >> 4;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t groups = H / 128;
  for (uint32_t row = warp; row < M; row += nwarps) {
    const uint16_t* xr = x + (size_t)row * H;
    float ss = 0.0f;
    for (uint32_t g = half; g < groups; g += 2) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(xr + g * 128 + hl * 8), f);
      float cs = 0.0f;   // 8-term chunk sums keep the FP32 rounding error small
#pragma unroll
      for (int j = 0; j < 8; ++j) cs = __fmaf_rn(f[j], f[j], cs);
      ss = __fadd_rn(ss, cs);
    }
    double d = (double)ss;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    const float r = (float)(1.0 / sqrt(d / (double)H + (double)eps));
    if (lane == 0) rstd[row] = r;
    // all lanes run the same number of iterations so the shuffles stay converged
    for (uint32_t g0 = 0; g0 < groups; g0 += 2) {
      const uint32_t g = g0 + half;
      const bool valid = g < groups;
      float f[8], gm[8];
      if (valid) {
        unpack8(*reinterpret_cast<const uint4*>(xr + g * 128 + hl * 8), f);
        unpack8(*reinterpret_cast<const uint4*>(gamma + g * 128 + hl * 8), gm);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = gm[j] = 0.0f;
      }
      uint32_t yb[4];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float a = __fmul_rn(__fmul_rn(f[j], r), gm[j]);
        float b = __fmul_rn(__fmul_rn(f[j + 1], r), gm[j + 1]);
        yb[j / 2] = f2_to_bf2(a, b);
        float2 back = bf2_to_f2(yb[j / 2]);
        f[j] = back.x; f[j + 1] = back.y;
      }
      float S;
      uint2 codes = quant_slice8(f, valid, S);
      if (valid) {
        *reinterpret_cast<uint2*>(q + (size_t)row * H + g * 128 + hl * 8) = codes;
        if (y != nullptr)
          *reinterpret_cast<uint4*>(y + (size_t)row * H + g * 128 + hl * 8) =
              make_uint4(yb[0], yb[1], yb[2], yb[3]);
        if (hl == 0) s[(size_t)g * ld_s + row] = S;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// X1: SwiGLU fused with the 1×128 quantiser.  Group g of the output h [M, I]
// reads gate and up slices of the same row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_swiglu_quant(const uint16_t* __restrict__ gu, uint32_t M, uint32_t I, uint32_t ld_s,
               uint8_t* __restrict__ q, float* __restrict__ s, uint16_t* __restrict__ h) {
  const uint32_t lane = threadIdx.x & 31u, hl = lane & 15u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t gpr = I / 128;
  const uint32_t n_groups = M * gpr;
  for (uint32_t base = warp * 2u; base < n_groups; base += nwarps * 2u) {
    const uint32_t g = base + (lane >> 4);
    const bool valid = g < n_groups;
    const uint32_t row = valid ? g / gpr : 0, col = valid ? (g % gpr) * 128 + hl * 8 : 0;
    float fg[8], fu[8], f[8];
    if (valid) {
      unpack8(ldg_stream(gu + (size_t)row * 2 * I + col), fg);
      unpack8(ldg_stream(gu + (size_t)row * 2 * I + I + col), fu);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) fg[j] = fu[j] = 0.0f;
    }
    uint32_t hb[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float a = __fmul_rn(fg[j] / (1.0f + expf(-fg[j])), fu[j]);
      float b = __fmul_rn(fg[j + 1] / (1.0f + expf(-fg[j + 1])), fu[j + 1]);
      hb[j / 2] = f2_to_bf2(a, b);
      float2 back = bf2_to_f2(hb[j / 2]);
      f[j] = back.x; f[j + 1] = back.y;
    }
    float S;
    uint2 codes = quant_slice8(f, valid, S);
    if (valid) {
      *reinterpret_cast<uint2*>(q + (size_t)row * I + col) = codes;
      if (h != nullptr)
        *reinterpret_cast<uint4*>(h + (size_t)row * I + col) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
      if (hl == 0) s[(size_t)(g % gpr) * ld_s + row] = S;
    }
  }
}

// ---------------------------------------------------------------------------
// X2: SwiGLU backward, elementwise, 8 outputs of each half per lane.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_swiglu_bwd(const uint16_t* __restrict__ gu, const uint16_t* __restrict__ dh, uint32_t M,
             uint32_t I, uint16_t* __restrict__ dgu) {
  const size_t n_chunks = (size_t)M * I / 8;
  for (size_t c = (size_t)blockIdx.x * kThreads + threadIdx.x; c < n_chunks;
       c += (size_t)gridDim.x * kThreads) {
    const size_t row = c / (I / 8), col = (c % (I / 8)) * 8;
    float fg[8], fu[8], fd[8];
    unpack8(ldg_stream(gu + row * 2 * I + col), fg);
    unpack8(ldg_stream(gu + row * 2 * I + I + col), fu);
    unpack8(ldg_stream(dh + row * I + col), fd);
    uint32_t og[4], ou[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float sg0 = 1.0f / (1.0f + expf(-fg[j])), sg1 = 1.0f / (1.0f + expf(-fg[j + 1]));
      float dg0 = fd[j] * fu[j] * sg0 * (1.0f + fg[j] * (1.0f - sg0));
      float dg1 = fd[j + 1] * fu[j + 1] * sg1 * (1.0f + fg[j + 1] * (1.0f - sg1));
      float du0 = fd[j] * fg[j] * sg0, du1 = fd[j + 1] * fg[j + 1] * sg1;
      og[j / 2] = f2_to_bf2(dg0, dg1);
      ou[j / 2] = f2_to_bf2(du0, du1);
    }
    *reinterpret_cast<uint4*>(dgu + row * 2 * I + col) = make_uint4(og[0], og[1], og[2], og[3]);
    *reinterpret_cast<uint4*>(dgu + row * 2 * I + I + col) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
  }
}

inline unsigned grid_for(size_t work_items, unsigned per_block, unsigned blocks_per_sm) {
  size_t need = (work_items + per_block - 1) / per_block;
  size_t cap = (size_t)num_sms() * blocks_per_sm;
  if (need < 1) need = 1;
  return (unsigned)(need < cap ? need : cap);
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers (arguments already validated by the C ABI layer)
// ---------------------------------------------------------------------------
cudaError_t launch_quant_rowgroups(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t st) {
  const uint32_t n_groups = (uint32_t)(M * (K / 128));
  const uint32_t gpr = (uint32_t)(K / 128);
  const uint32_t ld_s = (uint32_t)round_up4(M);
  constexpr int U = 4;
  const unsigned grid = grid_for((size_t)n_groups, (kThreads / 32) * 2 * U, 8);
  k_quant_rowgroups<U><<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(x), n_groups, gpr,
                                                  ld_s, q, s);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                uint8_t* qT, cudaStream_t st) {
  const size_t blocks = (size_t)(N / 128) * (K / 128);
  const unsigned grid = grid_for(blocks, 1, 8);
  k_quant_weight<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(w), (uint32_t)N,
                                            (uint32_t)K, q, s, qT);
  return cudaGetLastError();
}

cudaError_t launch_requant_row2col(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                   uint8_t* qT, float* sT, cudaStream_t st) {
  const size_t blocks = (size_t)(M / 128) * (K / 128);
  const unsigned grid = grid_for(blocks, 1, 8);
  k_requant_row2col<<<grid, kThreads, 0, st>>>(q, s, (uint32_t)M, (uint32_t)K, qT, sT);
  return cudaGetLastError();
}

cudaError_t launch_quant_grad_dual(const void* dy, int64_t M, int64_t N, uint8_t* q_row,
                                   float* s_row, uint8_t* qT_col, float* sT_col, cudaStream_t st) {
  if (qT_col == nullptr) return launch_quant_rowgroups(dy, M, N, q_row, s_row, st);
  const size_t blocks = (size_t)(M / 128) * (N / 128);
  const unsigned grid = grid_for(blocks, 1, 8);
  k_quant_grad_dual<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(dy), (uint32_t)M,
                                               (uint32_t)N, (uint32_t)round_up4(M), q_row, s_row,
                                               qT_col, sT_col);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t M,
                                 int64_t H, uint8_t* q, float* s, float* rstd, void* y,
                                 cudaStream_t st) {
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_rmsnorm_quant<<<grid, kThreads, 0, st>>>(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(gamma), eps, (uint32_t)M,
      (uint32_t)H, (uint32_t)round_up4(M), q, s, rstd, static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quant(const void* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                void* h, cudaStream_t st) {
  const size_t groups = (size_t)M * (I / 128);
  const unsigned grid = grid_for(groups, (kThreads / 32) * 2, 8);
  k_swiglu_quant<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(gu), (uint32_t)M,
                                            (uint32_t)I, (uint32_t)round_up4(M), q, s,
                                            static_cast<uint16_t*>(h));
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const void* gu, const void* dh, int64_t M, int64_t I, void* dgu,
                              cudaStream_t st) {
  const size_t chunks = (size_t)M * I / 8;
  const unsigned grid = grid_for(chunks, kThreads, 8);
  k_swiglu_bwd<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(gu),
                                          static_cast<const uint16_t*>(dh), (uint32_t)M,
                                          (uint32_t)I, static_cast<uint16_t*>(dgu));
  return cudaGetLastError();
}

}  // namespace jetfp8
