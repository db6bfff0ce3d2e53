// Memory-bound quantisation kernels of the mixed-granularity E4M3 linear layer.
//
// Jet-RL digest ("Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习"):
//   前置知识 › FP8 量化 (E4M3 格式)            — S = max|x|/448, x̂ = E4M3(x/S)
//   前置知识 › Per-group / Per-block 量化粒度  — 1×128 groups for activations and
//                                           gradients, 128×128 blocks for weights
//   方法步骤详情, steps 1-5                   — where each quantiser sits in the layer
//
// Layout of the work:
//  * Row-group kernels (Q1, R1, X1) give each warp whole rows; eight lanes share
//    one 128-wide group and each lane moves 32 bytes with one 256-bit access,
//    so a warp instruction covers 1 KB of contiguous bf16.
//  * Tile kernels (Q2, Q3, Q4) work on 128×128 tiles with 256 threads; thread t
//    owns the 8×8 sub-block at rows 8·(t/16), columns 8·(t%16).  Transposed
//    outputs are staged in a 16 KB shared tile with an XOR swizzle (conflict-
//    free 8-byte writes) and leave as full 128-byte rows, 16 bytes per thread.
//  * Pairs of values that share a scale are quantised together with packed
//    FP32 multiplies (quant_pair): pairs run along rows for row groups and
//    down columns for column groups, which makes the column codes come out
//    already in transposed order.
#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"

namespace jetfp8 {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void ld32_stream(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void ld32_cached(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint32_t (&r)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// 256-bit read-only load under an L2 eviction policy (createpolicy).
__device__ __forceinline__ void ld32_policy(const void* p, uint32_t (&r)[8], uint64_t pol) {
  asm volatile("ld.global.nc.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p), "l"(pol));
}
// 16-byte read that stays in L1 for a second pass over the same tile.
__device__ __forceinline__ uint4 ldg_cached16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Max over the 8 lanes that share a group (lanes 8j .. 8j+7).
__device__ __forceinline__ float group8_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}
// Max over the 16 lanes of a half-warp.
__device__ __forceinline__ float group16_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 8));
  return group8_max(v);
}

// One lane's 16 values (8 packed pairs) of a 1×128 group held by 8 lanes,
// all bf16 values: group amax, scale, and the 16 codes (4 words, first value
// in the low byte).
__device__ __forceinline__ uint4 quant16(const float2 (&f)[8], bool valid, float& S) {
  float amax = 0.0f;
  if (valid) {
#pragma unroll
    for (int w = 0; w < 8; ++w) amax = fmaxf(amax, fmaxf(fabsf(f[w].x), fabsf(f[w].y)));
  }
  const GroupScale g = make_scale_bf16(group8_max(amax));
  S = g.s;
  uint32_t c[4];
  quant_pairs<8>(f, g, c);
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// ---------------------------------------------------------------------------
// Q1: 1×128 row groups, one warp per row.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(kThreads)
k_quant_rows(const uint16_t* __restrict__ x, uint32_t M, uint32_t K, uint32_t ld_s,
             uint8_t* __restrict__ q, float* __restrict__ s) {
  const uint32_t lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t groups = K >> 7;
  for (uint32_t row = warp; row < M; row += nwarps) {
    const uint16_t* xr = x + (size_t)row * K;
    uint8_t* qr = q + (size_t)row * K;
    for (uint32_t g0 = 0; g0 < groups; g0 += 4 * U) {
      uint32_t raw[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        if (grp < groups) {
          ld32_stream(xr + grp * 128 + l8 * 16, raw[u]);
        } else {
#pragma unroll
          for (int w = 0; w < 8; ++w) raw[u][w] = 0;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        const bool valid = grp < groups;
        float2 f[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) f[w] = bf2_to_f2(raw[u][w]);
        float S;
        const uint4 c = quant16(f, valid, S);
        if (valid) {
          *reinterpret_cast<uint4*>(qr + grp * 128 + l8 * 16) = c;
          if (l8 == 0) s[(size_t)grp * ld_s + row] = S;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Shared 128×128-byte tile for transposed stores.  Row k holds 16 units of 8
// bytes; unit u is stored at position u ^ ((k/8) mod 16).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ttile_put8(uint8_t* T, uint32_t k, uint32_t unit, uint32_t lo,
                                           uint32_t hi) {
  const uint32_t phys = unit ^ ((k >> 3) & 15u);
  *reinterpret_cast<uint2*>(T + k * 128 + phys * 8) = make_uint2(lo, hi);
}

// out[(row0 + k) * ld + col0 + 0..127] = tile row k, for k = 0..127.
__device__ __forceinline__ void ttile_store(const uint8_t* T, uint8_t* __restrict__ out, size_t ld,
                                            size_t row0, size_t col0) {
#pragma unroll
  for (uint32_t i = threadIdx.x; i < 128 * 8; i += kThreads) {
    const uint32_t k = i >> 3, v = i & 7u;
    const uint32_t sw = (k >> 3) & 15u;
    uint4 val = *reinterpret_cast<const uint4*>(T + k * 128 + ((v ^ (sw >> 1)) << 4));
    if (sw & 1u) {
      const uint32_t a = val.x, b = val.y;
      val.x = val.z; val.y = val.w; val.z = a; val.w = b;
    }
    *reinterpret_cast<uint4*>(out + (row0 + k) * ld + col0 + v * 16) = val;
  }
}

// Column scales of a 128×128 tile: each thread passes its 8 columns' maxima
// over its 8 rows; 128 threads reduce a column each, build its GroupScale and
// store S to sT_out[0..127]; afterwards every thread can read the scale of any
// column from shared memory.  BF16_AMAX: the maxima are of bf16 values, so the
// scale takes the division-free exact path.
struct ColScales {
  float red[16][128];
  // column c's (S, ra, rb, exact) at g[c + c/8]: one 16-byte read per column,
  // and the 16 columns a warp reads together fall on distinct banks
  float4 g[128 + 16];
};

template <bool BF16_AMAX>
__device__ __forceinline__ void col_scales(const float (&cm)[8], ColScales& cs, float* sT_out) {
  const uint32_t rowgrp = threadIdx.x >> 4, c0 = 8u * (threadIdx.x & 15u);
  *reinterpret_cast<float4*>(&cs.red[rowgrp][c0]) = make_float4(cm[0], cm[1], cm[2], cm[3]);
  *reinterpret_cast<float4*>(&cs.red[rowgrp][c0 + 4]) = make_float4(cm[4], cm[5], cm[6], cm[7]);
  __syncthreads();
  if (threadIdx.x < 128) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, cs.red[i][threadIdx.x]);
    const GroupScale g = BF16_AMAX ? make_scale_bf16(m) : make_scale(m);
    cs.g[threadIdx.x + (threadIdx.x >> 3)] = make_float4(g.s, g.ra, g.rb, g.exact ? 1.0f : 0.0f);
    sT_out[threadIdx.x] = g.s;
  }
  __syncthreads();
}

__device__ __forceinline__ GroupScale load_col_scale(const ColScales& cs, uint32_t c) {
  const float4 v = cs.g[c + (c >> 3)];
  GroupScale g;
  g.s = v.x;
  g.ra = v.y;
  g.rb = v.z;
  g.exact = v.w != 0.0f;
  return g;
}

// Quantise column j of an 8×8 sub-block (rows 0..7) with that column's scale:
// returns the 8 codes in row order as (lo = rows 0-3, hi = rows 4-7).
template <typename Get>
__device__ __forceinline__ uint2 quant_col8(Get get, int j, const GroupScale& g) {
  const uint32_t p0 = quant_pair(make_float2(get(0, j), get(1, j)), g);
  const uint32_t p1 = quant_pair(make_float2(get(2, j), get(3, j)), g);
  const uint32_t p2 = quant_pair(make_float2(get(4, j), get(5, j)), g);
  const uint32_t p3 = quant_pair(make_float2(get(6, j), get(7, j)), g);
  return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

struct TileSmem {
  ColScales cs;
  uint8_t T[128 * 128];
  float wmax[kThreads / 32];
};

// ---------------------------------------------------------------------------
// Q2: 128×128 weight blocks, optional transposed payload (same codes).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 4)
k_quant_weight(const uint16_t* __restrict__ w, uint32_t N, uint32_t K, uint8_t* __restrict__ q,
               float* __restrict__ s, uint8_t* __restrict__ qT) {
  __shared__ __align__(16) TileSmem sm;
  const uint32_t kblocks = K / 128, nblocks = N / 128;
  const uint32_t r0 = 8u * (threadIdx.x >> 4), c0 = 8u * (threadIdx.x & 15u);
  for (uint32_t blk = blockIdx.x; blk < kblocks * nblocks; blk += gridDim.x) {
    const uint32_t nb = blk / kblocks, kb = blk % kblocks;
    const size_t row0 = (size_t)nb * 128 + r0, col0 = (size_t)kb * 128 + c0;
    // read through L1; the codes pass reads the sub-block again (an L1 hit)
    // rather than holding it across the block-amax barrier
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = ldg_cached16(w + (row0 + i) * K + col0);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t ws[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 f = bf2_to_f2(ws[p]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    if ((threadIdx.x & 31) == 0) sm.wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = sm.wmax[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, sm.wmax[i]);
    const GroupScale g = make_scale_bf16(amax);
    if (threadIdx.x == 0) s[(size_t)nb * kblocks + kb] = g.s;
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = ldg_cached16(w + (row0 + i) * K + col0);
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo[i] = quant_pair(bf2_to_f2(raw[i].x), g) | (quant_pair(bf2_to_f2(raw[i].y), g) << 16);
      hi[i] = quant_pair(bf2_to_f2(raw[i].z), g) | (quant_pair(bf2_to_f2(raw[i].w), g) << 16);
      *reinterpret_cast<uint2*>(q + (row0 + i) * K + col0) = make_uint2(lo[i], hi[i]);
    }
    if (qT != nullptr) {
      uint32_t olo[8], ohi[8];
      transpose8x8(lo, hi, olo, ohi);
#pragma unroll
      for (int j = 0; j < 8; ++j) ttile_put8(sm.T, c0 + j, r0 >> 3, olo[j], ohi[j]);
      __syncthreads();
      ttile_store(sm.T, qT, N, (size_t)kb * 128, (size_t)nb * 128);
    }
    __syncthreads();   // wmax and T are reused by the next block
  }
}

// ---------------------------------------------------------------------------
// Q3: dequantise 1×128 row groups, requantise 128×1 column groups, transpose.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 3)
k_requant_row2col(const uint8_t* __restrict__ q, const float* __restrict__ s, uint32_t M,
                  uint32_t K, uint8_t* __restrict__ qT, float* __restrict__ sT) {
  __shared__ __align__(16) TileSmem sm;
  const uint32_t kblocks = K / 128, mblocks = M / 128;
  const uint32_t r0 = 8u * (threadIdx.x >> 4), c0 = 8u * (threadIdx.x & 15u);
  for (uint32_t blk = blockIdx.x; blk < kblocks * mblocks; blk += gridDim.x) {
    const uint32_t mb = blk / kblocks, kb = blk % kblocks;
    const size_t row0 = (size_t)mb * 128 + r0, col0 = (size_t)kb * 128 + c0;
    uint2 c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = *reinterpret_cast<const uint2*>(q + (row0 + i) * K + col0);
    const float4 s_lo = *reinterpret_cast<const float4*>(s + (size_t)kb * M + row0);
    const float4 s_hi = *reinterpret_cast<const float4*>(s + (size_t)kb * M + row0 + 4);
    const float srow[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
    // x̃ = fp32(dec(q)·S) for a column pair (j, j+1) of the 8 rows; computed
    // once for the column maxima and again for the codes, so that only the
    // 64 code bytes stay in registers across the column-scale barriers
    auto dequant = [&](int i, int j) {
      const uint32_t word = (j < 4 ? c[i].x : c[i].y) >> (8 * (j & 3));
      const float2 d = dec_e4m3x2(word & 0xFFFFu);
      return make_float2(__fmul_rn(d.x, srow[i]), __fmul_rn(d.y, srow[i]));
    };
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cm[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float2 v = dequant(i, j);
        cm[j] = fmaxf(cm[j], fabsf(v.x));
        cm[j + 1] = fmaxf(cm[j + 1], fabsf(v.y));
      }
    }
    col_scales<false>(cm, sm.cs, sT + (size_t)mb * K + (size_t)kb * 128);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float v0[8], v1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 v = dequant(i, j);
        v0[i] = v.x;
        v1[i] = v.y;
      }
      const uint2 codes0 = quant_col8([&](int i, int) { return v0[i]; }, j, load_col_scale(sm.cs, c0 + j));
      ttile_put8(sm.T, c0 + j, r0 >> 3, codes0.x, codes0.y);
      const uint2 codes1 =
          quant_col8([&](int i, int) { return v1[i]; }, j + 1, load_col_scale(sm.cs, c0 + j + 1));
      ttile_put8(sm.T, c0 + j + 1, r0 >> 3, codes1.x, codes1.y);
    }
    __syncthreads();
    ttile_store(sm.T, qT, M, (size_t)kb * 128, (size_t)mb * 128);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Q4: one read of the bf16 gradient: 1×128 row groups along N (stored as is)
// and 128×1 column groups along M (stored transposed).  M multiple of 128.
// The first pass reads the tile through L1 and the column pass reads the
// thread's 8×8 sub-block again (an L1 hit) instead of holding it in registers
// across the column-scale barriers, which leaves room for four CTAs per SM.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 4)
k_quant_grad_dual(const uint16_t* __restrict__ dy, uint32_t M, uint32_t N, uint32_t ld_srow,
                  uint8_t* __restrict__ q_row, float* __restrict__ s_row,
                  uint8_t* __restrict__ qT_col, float* __restrict__ sT_col) {
  __shared__ __align__(16) TileSmem sm;
  const uint32_t nblocks = N / 128, mblocks = M / 128;
  const uint32_t r0 = 8u * (threadIdx.x >> 4), c0 = 8u * (threadIdx.x & 15u);
  for (uint32_t blk = blockIdx.x; blk < nblocks * mblocks; blk += gridDim.x) {
    const uint32_t mb = blk / nblocks, nb = blk % nblocks;
    const size_t row0 = (size_t)mb * 128 + r0, col0 = (size_t)nb * 128 + c0;
    uint32_t raw[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 t = ldg_cached16(dy + (row0 + i) * N + col0);
      raw[i][0] = t.x; raw[i][1] = t.y; raw[i][2] = t.z; raw[i][3] = t.w;
    }
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cm[j] = 0.0f;
    float srow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 f[4];
      float amax = 0.0f;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        f[p] = bf2_to_f2(raw[i][p]);
        cm[2 * p] = fmaxf(cm[2 * p], fabsf(f[p].x));
        cm[2 * p + 1] = fmaxf(cm[2 * p + 1], fabsf(f[p].y));
        amax = fmaxf(amax, fmaxf(fabsf(f[p].x), fabsf(f[p].y)));
      }
      const GroupScale g = make_scale_bf16(group16_max(amax));
      srow[i] = g.s;
      uint32_t codes[2];
      quant_pairs<4>(f, g, codes);
      *reinterpret_cast<uint2*>(q_row + (row0 + i) * N + col0) = make_uint2(codes[0], codes[1]);
    }
    if (c0 == 0) {
      *reinterpret_cast<float4*>(s_row + (size_t)nb * ld_srow + row0) =
          make_float4(srow[0], srow[1], srow[2], srow[3]);
      *reinterpret_cast<float4*>(s_row + (size_t)nb * ld_srow + row0 + 4) =
          make_float4(srow[4], srow[5], srow[6], srow[7]);
    }
    col_scales<true>(cm, sm.cs, sT_col + (size_t)mb * N + (size_t)nb * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 t = ldg_cached16(dy + (row0 + i) * N + col0);
      raw[i][0] = t.x; raw[i][1] = t.y; raw[i][2] = t.z; raw[i][3] = t.w;
    }
    auto get = [&](int i, int j) {
      const uint32_t wv = raw[i][j >> 1];
      return __uint_as_float((j & 1) ? (wv & 0xFFFF0000u) : (wv << 16));
    };
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint2 codes = quant_col8(get, j, load_col_scale(sm.cs, c0 + j));
      ttile_put8(sm.T, c0 + j, r0 >> 3, codes.x, codes.y);
    }
    __syncthreads();
    ttile_store(sm.T, qT_col, M, (size_t)nb * 128, (size_t)mb * 128);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// R1: RMSNorm fused with the 1×128 quantiser.  One warp per row, 8 lanes per
// group.  Pass 1 accumulates Σx² (16-term FP32 chunk sums per lane, lanes
// combined in FP64); pass 2 re-reads the row (an L1/L2 hit) and writes y, q, S.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_rmsnorm_quant(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps,
                uint32_t M, uint32_t H, uint32_t ld_s, uint8_t* __restrict__ q,
                float* __restrict__ s, float* __restrict__ rstd, uint16_t* __restrict__ y) {
  constexpr int U = 4;
  const uint32_t lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t groups = H / 128;
  for (uint32_t row = warp; row < M; row += nwarps) {
    const uint16_t* xr = x + (size_t)row * H;
    float ss = 0.0f;
    for (uint32_t g0 = 0; g0 < groups; g0 += 4 * U) {
      uint32_t raw[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        if (grp < groups) {
          ld32_cached(xr + grp * 128 + l8 * 16, raw[u]);
        } else {
#pragma unroll
          for (int w = 0; w < 8; ++w) raw[u][w] = 0;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float cs = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float2 f = bf2_to_f2(raw[u][w]);
          cs = __fmaf_rn(f.x, f.x, cs);
          cs = __fmaf_rn(f.y, f.y, cs);
        }
        ss = __fadd_rn(ss, cs);
      }
    }
    double d = (double)ss;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(kFull, d, o);
    // every lane holds the same d; FP64 division and square root are slow on
    // this GPU, so one lane forms r and passes it on
    float r = 0.0f;
    if (lane == 0) {
      r = (float)(1.0 / sqrt(d / (double)H + (double)eps));
      rstd[row] = r;
    }
    r = __shfl_sync(kFull, r, 0);
    for (uint32_t g0 = 0; g0 < groups; g0 += 4) {
      const uint32_t grp = g0 + g4;
      const bool valid = grp < groups;
      uint32_t rx[8], rg[8];
      if (valid) {
        ld32_cached(xr + grp * 128 + l8 * 16, rx);
        ld32_cached(gamma + grp * 128 + l8 * 16, rg);
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) rx[w] = rg[w] = 0;
      }
      float2 f[8];
      uint32_t yb[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 t = mul2(mul2(bf2_to_f2(rx[w]), make_float2(r, r)), bf2_to_f2(rg[w]));
        yb[w] = f2_to_bf2(t.x, t.y);
        f[w] = bf2_to_f2(yb[w]);
      }
      float S;
      const uint4 c = quant16(f, valid, S);
      if (valid) {
        *reinterpret_cast<uint4*>(q + (size_t)row * H + grp * 128 + l8 * 16) = c;
        if (y != nullptr) st32(y + (size_t)row * H + grp * 128 + l8 * 16, yb);
        if (l8 == 0) s[(size_t)grp * ld_s + row] = S;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// RMSNorm backward (decoder-layer support).  With the forward's saved r:
//   ∇x_i = r·(dy_i·γ_i) − x_i·(r³·Σ_j dy_j·γ_j·x_j / H)
//   ∇γ_j = Σ_rows dy_j·x_j·r
// ∇x: one warp per row, 8 lanes per 128-wide group as in R1; the row sum is
// accumulated like R1's Σx² (16-term FP32 chunk sums per lane, lanes in FP64).
// ∇γ: deterministic two-stage column sums — FP32 partial sums over 128-row
// chunks into the caller's workspace [chunks][H], then each column's partials
// added in a fixed order in FP64.
// ---------------------------------------------------------------------------
constexpr int kNormBwdRows = 128;   // rows per ∇γ partial sum

__global__ void __launch_bounds__(kThreads)
k_rmsnorm_bwd_dx(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma,
                 const float* __restrict__ rstd, const uint16_t* __restrict__ dy, uint32_t M,
                 uint32_t H, uint16_t* __restrict__ dx) {
  constexpr int U = 4;
  const uint32_t lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t groups = H / 128;
  // x and ∇y are read twice per row: the first pass asks L2 to keep the lines
  // for the second, which asks it to drop them (x and ∇y of the rows in flight
  // otherwise overflow the caches and the second pass goes back to DRAM)
  uint64_t pol_keep, pol_drop;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_drop));
  for (uint32_t row = warp; row < M; row += nwarps) {
    const uint16_t* xr = x + (size_t)row * H;
    const uint16_t* dr = dy + (size_t)row * H;
    float dot = 0.0f;
    for (uint32_t g0 = 0; g0 < groups; g0 += 4 * U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        if (grp >= groups) continue;
        uint32_t rx[8], rd[8], rg[8];
        ld32_policy(xr + grp * 128 + l8 * 16, rx, pol_keep);
        ld32_policy(dr + grp * 128 + l8 * 16, rd, pol_keep);
        ld32_cached(gamma + grp * 128 + l8 * 16, rg);
        float cs = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float2 fx = bf2_to_f2(rx[w]), fd = bf2_to_f2(rd[w]), fg = bf2_to_f2(rg[w]);
          cs = __fmaf_rn(__fmul_rn(fd.x, fg.x), fx.x, cs);
          cs = __fmaf_rn(__fmul_rn(fd.y, fg.y), fx.y, cs);
        }
        dot = __fadd_rn(dot, cs);
      }
    }
    double d = (double)dot;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(kFull, d, o);
    const float r = rstd[row];
    // every lane holds the same d: one lane forms c (FP64 is slow on this GPU)
    float c = 0.0f;
    if (lane == 0) c = (float)((double)r * (double)r * (double)r * d / (double)H);
    c = __shfl_sync(kFull, c, 0);
    for (uint32_t g0 = 0; g0 < groups; g0 += 4) {
      const uint32_t grp = g0 + g4;
      if (grp >= groups) continue;
      uint32_t rx[8], rd[8], rg[8], out[8];
      ld32_policy(xr + grp * 128 + l8 * 16, rx, pol_drop);
      ld32_policy(dr + grp * 128 + l8 * 16, rd, pol_drop);
      ld32_cached(gamma + grp * 128 + l8 * 16, rg);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 fx = bf2_to_f2(rx[w]), fd = bf2_to_f2(rd[w]), fg = bf2_to_f2(rg[w]);
        const float a = __fsub_rn(__fmul_rn(r, __fmul_rn(fd.x, fg.x)), __fmul_rn(fx.x, c));
        const float b = __fsub_rn(__fmul_rn(r, __fmul_rn(fd.y, fg.y)), __fmul_rn(fx.y, c));
        out[w] = f2_to_bf2(a, b);
      }
      st32(dx + (size_t)row * H + grp * 128 + l8 * 16, out);
    }
  }
}

// Partial ∇γ over rows [128p, 128p + 128) for 512 columns per CTA (2 per thread).
__global__ void __launch_bounds__(kThreads)
k_rmsnorm_bwd_dgamma_partial(const uint16_t* __restrict__ x, const float* __restrict__ rstd,
                             const uint16_t* __restrict__ dy, uint32_t M, uint32_t H,
                             float* __restrict__ ws) {
  const uint32_t col = blockIdx.x * 512u + 2u * threadIdx.x;
  const uint32_t p = blockIdx.y;
  const uint32_t r0 = p * kNormBwdRows, r1 = min(M, r0 + kNormBwdRows);
  if (col >= H) return;
  float ax = 0.0f, ay = 0.0f;
  // eight rows' loads in flight per thread (the sums still run in row order)
#pragma unroll 8
  for (uint32_t m = r0; m < r1; ++m) {
    const float2 fx = bf2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(x + (size_t)m * H + col)));
    const float2 fd = bf2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(dy + (size_t)m * H + col)));
    const float r = __ldg(rstd + m);
    ax = __fadd_rn(ax, __fmul_rn(__fmul_rn(fd.x, fx.x), r));
    ay = __fadd_rn(ay, __fmul_rn(__fmul_rn(fd.y, fx.y), r));
  }
  *reinterpret_cast<float2*>(ws + (size_t)p * H + col) = make_float2(ax, ay);
}

// 32 columns per CTA, eight threads per column (one per warp): thread j adds
// the partials of chunks j, j + 8, j + 16, ... in FP64, then the eight sums are
// added in j order.  The order is fixed, so the result is deterministic; the
// dependent FP64 chain per thread is chunks/8 long (FP64 is slow on this GPU).
constexpr uint32_t kReduceWays = kThreads / 32;
__global__ void __launch_bounds__(kThreads)
k_rmsnorm_bwd_dgamma_reduce(const float* __restrict__ ws, uint32_t chunks, uint32_t H,
                            float* __restrict__ dgamma) {
  __shared__ double part[kReduceWays][32];
  const uint32_t cl = threadIdx.x & 31u, j = threadIdx.x >> 5;
  const uint32_t col = blockIdx.x * 32 + cl;
  double s = 0.0;
  if (col < H)
    for (uint32_t p = j; p < chunks; p += kReduceWays) s += (double)__ldg(ws + (size_t)p * H + col);
  part[j][cl] = s;
  __syncthreads();
  if (j == 0 && col < H) {
    double t = 0.0;
#pragma unroll
    for (uint32_t i = 0; i < kReduceWays; ++i) t += part[i][cl];
    dgamma[col] = (float)t;
  }
}

// ---------------------------------------------------------------------------
// X1: SwiGLU fused with the 1×128 quantiser; one warp per row of h [M, I].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_swiglu_quant(const uint16_t* __restrict__ gu, uint32_t M, uint32_t I, uint32_t ld_s,
               uint8_t* __restrict__ q, float* __restrict__ s, uint16_t* __restrict__ h) {
  const uint32_t lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kThreads) >> 5;
  const uint32_t groups = I / 128;
  for (uint32_t row = warp; row < M; row += nwarps) {
    const uint16_t* gr = gu + (size_t)row * 2 * I;
    for (uint32_t g0 = 0; g0 < groups; g0 += 4) {
      const uint32_t grp = g0 + g4;
      const bool valid = grp < groups;
      uint32_t rg[8], ru[8];
      if (valid) {
        ld32_stream(gr + grp * 128 + l8 * 16, rg);
        ld32_stream(gr + I + grp * 128 + l8 * 16, ru);
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) rg[w] = ru[w] = 0;
      }
      float2 f[8];
      uint32_t hb[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 gg = bf2_to_f2(rg[w]), uu = bf2_to_f2(ru[w]);
        // SiLU with the fast exponential and division (a few FP32 ulps, far below
        // the bf16 rounding of h that follows; the exact IEEE forms made this
        // kernel issue-bound)
        const float a = __fmul_rn(__fdividef(gg.x, 1.0f + __expf(-gg.x)), uu.x);
        const float b = __fmul_rn(__fdividef(gg.y, 1.0f + __expf(-gg.y)), uu.y);
        hb[w] = f2_to_bf2(a, b);
        f[w] = bf2_to_f2(hb[w]);
      }
      float S;
      const uint4 c = quant16(f, valid, S);
      if (valid) {
        *reinterpret_cast<uint4*>(q + (size_t)row * I + grp * 128 + l8 * 16) = c;
        if (h != nullptr) st32(h + (size_t)row * I + grp * 128 + l8 * 16, hb);
        if (l8 == 0) s[(size_t)grp * ld_s + row] = S;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// X2: SwiGLU backward, elementwise; each thread handles 16 gate and 16 up
// outputs (32-byte accesses).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_swiglu_bwd(const uint16_t* __restrict__ gu, const uint16_t* __restrict__ dh, uint32_t M,
             uint32_t I, uint16_t* __restrict__ dgu) {
  const size_t n_chunks = (size_t)M * I / 16;
  for (size_t c = (size_t)blockIdx.x * kThreads + threadIdx.x; c < n_chunks;
       c += (size_t)gridDim.x * kThreads) {
    const size_t row = c / (I / 16), col = (c % (I / 16)) * 16;
    uint32_t rg[8], ru[8], rd[8], og[8], ou[8];
    ld32_stream(gu + row * 2 * I + col, rg);
    ld32_stream(gu + row * 2 * I + I + col, ru);
    ld32_stream(dh + row * I + col, rd);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float2 g = bf2_to_f2(rg[w]), u = bf2_to_f2(ru[w]), d = bf2_to_f2(rd[w]);
      const float s0 = 1.0f / (1.0f + expf(-g.x)), s1 = 1.0f / (1.0f + expf(-g.y));
      og[w] = f2_to_bf2(d.x * u.x * s0 * (1.0f + g.x * (1.0f - s0)),
                        d.y * u.y * s1 * (1.0f + g.y * (1.0f - s1)));
      ou[w] = f2_to_bf2(d.x * g.x * s0, d.y * g.y * s1);
    }
    st32(dgu + row * 2 * I + col, og);
    st32(dgu + row * 2 * I + I + col, ou);
  }
}

inline unsigned grid_for(size_t work_items, unsigned per_block, unsigned blocks_per_sm) {
  size_t need = (work_items + per_block - 1) / per_block;
  const size_t cap = (size_t)num_sms() * blocks_per_sm;
  if (need < 1) need = 1;
  return (unsigned)(need < cap ? need : cap);
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers (arguments already validated by the C ABI layer)
// ---------------------------------------------------------------------------
cudaError_t launch_quant_rowgroups(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t st) {
  constexpr int U = 2;
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_quant_rows<U><<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(x), (uint32_t)M,
                                             (uint32_t)K, (uint32_t)round_up4(M), q, s);
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
  const unsigned grid = grid_for(blocks, 1, 6);
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

size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H) {
  return (size_t)((M + kNormBwdRows - 1) / kNormBwdRows) * (size_t)H * sizeof(float);
}

cudaError_t launch_rmsnorm_bwd(const void* x, const void* gamma, const float* rstd, const void* dy,
                               int64_t M, int64_t H, void* dx, float* dgamma, float* ws,
                               cudaStream_t st) {
  const auto* xb = static_cast<const uint16_t*>(x);
  const auto* db = static_cast<const uint16_t*>(dy);
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_rmsnorm_bwd_dx<<<grid, kThreads, 0, st>>>(xb, static_cast<const uint16_t*>(gamma), rstd, db,
                                              (uint32_t)M, (uint32_t)H, static_cast<uint16_t*>(dx));
  const uint32_t chunks = (uint32_t)((M + kNormBwdRows - 1) / kNormBwdRows);
  const dim3 pgrid((unsigned)((H + 511) / 512), chunks);
  k_rmsnorm_bwd_dgamma_partial<<<pgrid, kThreads, 0, st>>>(xb, rstd, db, (uint32_t)M, (uint32_t)H, ws);
  k_rmsnorm_bwd_dgamma_reduce<<<(unsigned)((H + 31) / 32), kThreads, 0, st>>>(
      ws, chunks, (uint32_t)H, dgamma);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quant(const void* gu, int64_t M, int64_t I, uint8_t* q, float* s,
                                void* h, cudaStream_t st) {
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_swiglu_quant<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(gu), (uint32_t)M,
                                            (uint32_t)I, (uint32_t)round_up4(M), q, s,
                                            static_cast<uint16_t*>(h));
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const void* gu, const void* dh, int64_t M, int64_t I, void* dgu,
                              cudaStream_t st) {
  const size_t chunks = (size_t)M * I / 16;
  const unsigned grid = grid_for(chunks, kThreads, 8);
  k_swiglu_bwd<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t*>(gu),
                                          static_cast<const uint16_t*>(dh), (uint32_t)M,
                                          (uint32_t)I, static_cast<uint16_t*>(dgu));
  return cudaGetLastError();
}

}  // namespace jetfp8
