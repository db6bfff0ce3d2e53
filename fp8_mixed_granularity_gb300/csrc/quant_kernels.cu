// Memory-bound quantisation kernels of the mixed-granularity E4M3 linear layer.
//
// Jet-RL digest ("Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习"):
//   前置知识 › FP8 量化 (E4M3 格式)            — S = max|x|/448, x̂ = E4M3(x/S)
//   前置知识 › Per-group / Per-block 量化粒度  — 1×128 groups for activations and
//                                           gradients, 128×128 blocks for weights
//   方法步骤详情, steps 1-5                   — where each quantiser sits in the layer
//
// Layout of the work (details at the TMA-fed kernels below):
//  * Row streams (Q1, R1): each warp streams its own row segments (R1: whole
//    rows) into a private two-slot shared-memory ring with bulk copies; eight
//    lanes share a 1×128 group.  Wider R1 rows and the SwiGLU quantiser (X1)
//    read global memory directly, one warp per row.
//  * Tile pipelines (Q2, Q3, Q4): persistent CTAs of warpgroups, each with a
//    private double-buffered ring of 128×128 tiles loaded by the tensor-memory
//    accelerator; a row pass and a column pass read the tile from shared
//    memory with their own thread mappings, so every group maximum is a
//    half-warp shuffle and every output a coalesced 8-byte store.
//  * Element codes: the correctly rounded quotient x/S formed without a
//    division (codes4_bf16 / codes4_neg_f32 in jetfp8_common.cuh), then the
//    saturating E4M3 cast.
#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"
#include "jetfp8_tma.cuh"

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
// Max over the 8 lanes that share a group (lanes 8j .. 8j+7).
__device__ __forceinline__ float group8_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}
// ===========================================================================
// TMA-fed quantisers.  Two shapes of work:
//  * row streams (Q1, R1): each warp owns a private ring of shared-memory
//    slots and streams its own row segments into them with bulk copies one
//    unit ahead of the one it quantises; codes and scales go straight to
//    global memory.  R1 holds the whole row in its slot, so the row is read
//    from HBM once for both of its passes.
//  * tile pipelines (Q2, Q3, Q4): persistent CTAs of several warpgroups; each
//    warpgroup owns a private double-buffered ring of 128×128 tiles
//    (128-byte swizzled tensor-map boxes), filled by its first thread one tile
//    ahead of the one it quantises.  A tile is read from shared memory once
//    per grouping: in the row pass thread t holds rows 8·(t/16)+i, columns
//    8·(t%16)+0..7, so the 16 threads of a row group are one half-warp; in the
//    column pass thread t holds columns 8·(t/16)+0..7 of rows 8·(t%16)+i, so
//    the 16 threads of a 128-row column group are one half-warp.  Both group
//    maxima are half-warp shuffles, and both outputs leave as 8-byte stores
//    that a half-warp makes into one 128-byte line (column codes come out in
//    transposed order).  In the column pass thread t reads its rows in the
//    rotated order i -> 8·(t%16) + ((i + t%16) mod 8), which spreads a
//    half-warp's reads over all banks under the 128-byte swizzle; its codes
//    are rotated back into row order before the store.
// Codes come from the exact division-free quotient of jetfp8_common.cuh
// (codes4_bf16 and relatives: two Markstein corrections of RN(x·RN(1/S)) on the
// negated values), four at a time in packed FP32 pairs; groups whose maximum is
// below 2^-80 run the same sequence on operands scaled by 2^96.  Of the 8 group
// scales a half-warp needs, each lane computes one and the others arrive by
// shuffle.  Every wait is bounded (jetfp8_tma.cuh);
// on expiry the kernel records the error word, stops issuing copies, waits
// for the copies it issued and returns.
// ===========================================================================
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

// Per half of two packed bf16 pairs: a value whose magnitude is max(|a|, |b|)
// (its sign bit is not meaningful; mask with 0x7FFF7FFF).
__device__ __forceinline__ uint32_t amax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// f16 (one half of a decoded pair) -> FP32, exact.
__device__ __forceinline__ float h2f(uint16_t b) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(b));
  return f;
}

// Max over the 16 lanes of a half-warp of 8 per-lane column values a[0..7],
// returned in the lane l of column l mod 8.  Each exchange step hands the
// partner the half of the columns it keeps (lane bit 0 picks the column's bit 0,
// bit 1 its bit 1, bit 2 its bit 2), so 8 shuffles replace 32.
__device__ __forceinline__ float half_warp_colmax8(const float (&a)[8]) {
  const uint32_t lane = threadIdx.x & 31u;
  const bool b0 = lane & 1u, b1 = lane & 2u, b2 = lane & 4u;
  float r1[4], r2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b0 ? a[2 * i + 1] : a[2 * i], send = b0 ? a[2 * i] : a[2 * i + 1];
    r1[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, 1));
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = b1 ? r1[2 * j + 1] : r1[2 * j], send = b1 ? r1[2 * j] : r1[2 * j + 1];
    r2[j] = fmaxf(keep, __shfl_xor_sync(kFull, send, 2));
  }
  const float keep = b2 ? r2[1] : r2[0], send = b2 ? r2[0] : r2[1];
  const float r3 = fmaxf(keep, __shfl_xor_sync(kFull, send, 4));
  return fmaxf(r3, __shfl_xor_sync(kFull, r3, 8));
}

// Quotient constants of 8 groups whose maxima are already reduced so that lane
// l holds group (l mod 8)'s: lane l computes that group's S and -RN(1/S), and the
// half-warp shares them by shuffle; bit i of the returned mask marks group i as
// slow (0 < amax < kQuotientMinAmax).
__device__ __forceinline__ uint32_t half_warp_qscales_of(float a, float (&s)[8], float (&ny)[8]) {
  const uint32_t base = threadIdx.x & 16u;
  const float s_mine = make_scale(a).s;
  const float ny_mine = -__frcp_rn(s_mine);
  const bool slow = a != 0.0f && a < kQuotientMinAmax;
  const uint32_t mask = (__ballot_sync(kFull, slow) >> base) & 0xFFu;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s[i] = __shfl_sync(kFull, s_mine, base + i);
    ny[i] = __shfl_sync(kFull, ny_mine, base + i);
  }
  return mask;
}

// max(|a|, |b|, |c|) in one three-input maximum.
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

__device__ __forceinline__ QScale qscale_of(float s, float ny) {
  QScale g;
  g.s = s;
  g.slow = false;
  g.s2 = pack_f2(s, s);
  g.ny2 = pack_f2(ny, ny);
  return g;
}

__device__ __forceinline__ void record_timeout(volatile int* abort_word, unsigned* err) {
  if (abort_word != nullptr) *abort_word = 1;
  atomicOr(err, kErrTimeout);
}

// 8 codes held as (lo, hi) with byte i from rotated slot i, i.e. tile row
// (i + k) mod 8 -> bytes in row order (byte r <- byte (r - k) mod 8): two byte
// permutes whose selectors depend only on k (0..7), formed once per thread.
__device__ __forceinline__ uint2 unrotate_selectors(uint32_t k) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (uint32_t r = 0; r < 4; ++r) {
    lo |= ((r - k) & 7u) << (4u * r);
    hi |= ((r + 4u - k) & 7u) << (4u * r);
  }
  return make_uint2(lo, hi);
}
__device__ __forceinline__ uint2 unrotate8(uint32_t lo, uint32_t hi, uint2 sel) {
  return make_uint2(__byte_perm(lo, hi, sel.x), __byte_perm(lo, hi, sel.y));
}

// Offset of 16-byte chunk c (0..7) of row r in a box of 128-byte rows stored
// with the 128-byte swizzle (box base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// ---------------------------------------------------------------------------
// Row streams.  Lanes 8j..8j+7 share 128-element groups g with g ≡ j (mod 4);
// lane l holds elements 8·(l mod 8) + 0..7 and 64 + 8·(l mod 8) + 0..7 of its
// group (two 16-byte reads that are conflict-free across the warp).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_group16(uint32_t gb, uint32_t l8, uint32_t (&w)[8]) {
  const uint4 a = lds128(gb + l8 * 16u), b = lds128(gb + 128u + l8 * 16u);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// One lane's 16 bf16 values of a group (8 packed words; of -x when NEG, of x
// otherwise): the group's maximum over its 8 lanes, its scale, and the 16 codes
// of x as (first half, second half).
template <bool NEG>
__device__ __forceinline__ void group16_codes_of(const uint32_t (&w)[8], bool valid, float& S, uint2& c0,
                                                 uint2& c1) {
  uint32_t m = amax2(amax2(amax2(w[0], w[1]), amax2(w[2], w[3])), amax2(amax2(w[4], w[5]), amax2(w[6], w[7])));
  m &= 0x7FFF7FFFu;
  float amax = valid ? fmaxf(bf_lo(m), bf_hi(m)) : 0.0f;
  amax = group8_max(amax);
  S = make_scale(amax).s;
  uint32_t c[4];
  if (amax != 0.0f && amax < kQuotientMinAmax) {
    constexpr float k96 = NEG ? 0x1p96f : -0x1p96f;   // the scaled negated values
    const QScale g = qscale_from_s(S * 0x1p96f, false);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = bf2_to_f2(w[2 * k]), b = bf2_to_f2(w[2 * k + 1]);
      c[k] = codes4_neg_f32(pack_f2(a.x * k96, a.y * k96), pack_f2(b.x * k96, b.y * k96), g);
    }
  } else {
    const QScale g = qscale_from_s(S, false);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      c[k] = NEG ? codes4_negbf16(w[2 * k], w[2 * k + 1], g) : codes4_bf16(w[2 * k], w[2 * k + 1], g);
  }
  c0 = make_uint2(c[0], c[1]);
  c1 = make_uint2(c[2], c[3]);
}

__device__ __forceinline__ void group16_codes_neg(const uint32_t (&nw)[8], bool valid, float& S, uint2& c0,
                                                  uint2& c1) {
  group16_codes_of<true>(nw, valid, S, c0, c1);
}
__device__ __forceinline__ void group16_codes(const uint32_t (&w)[8], bool valid, float& S, uint2& c0, uint2& c1) {
  group16_codes_of<false>(w, valid, S, c0, c1);
}

// c plus the squares of one lane's 16 bf16 values (8 packed words), added in
// element order, each step one FMA on the bf16 operands (the square is exact in FP32).
__device__ __forceinline__ float add_squares16(const uint32_t (&w)[8], float c) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
        "fma.rn.f32.bf16 %0, l, l, %0;\n\t"
        "fma.rn.f32.bf16 %0, h, h, %0;\n\t}"
        : "+f"(c) : "r"(w[e]));
  return c;
}

// For a pair of bf16 x (wx) and γ (wg): -bf16(RN(RN(x·γ)·r)) as a bf16 pair,
// given nr2 = (-r, -r).  x·γ is one FMA on the bf16 operands with a -0 addend,
// exact while |x·γ| is a normal FP32 number; the product with -r is one FP32
// rounding, then the bf16 rounding (both symmetric, so the result is -y).
__device__ __forceinline__ uint32_t neg_norm_pair(uint32_t wx, uint32_t wg, uint64_t nr2) {
  uint32_t o;
  asm("{\n\t.reg .b16 xl, xh, gl, gh;\n\t.reg .b32 pl, ph;\n\t.reg .b64 p;\n\t"
      "mov.b32 {xl, xh}, %1;\n\t"
      "mov.b32 {gl, gh}, %2;\n\t"
      "fma.rn.f32.bf16 pl, xl, gl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 ph, xh, gh, 0f80000000;\n\t"
      "mov.b64 p, {pl, ph};\n\t"
      "mul.rn.f32x2 p, p, %3;\n\t"
      "mov.b64 {pl, ph}, p;\n\t"
      "cvt.rn.bf16x2.f32 %0, ph, pl;\n\t}"
      : "=r"(o) : "r"(wx), "r"(wg), "l"(nr2));
  return o;
}

constexpr uint32_t kSeg = 2048;   // Q1 unit: 4 KB of bf16

template <int W, int D>
__global__ void __launch_bounds__(32 * W, 1)
k_quant_rows_tma(const uint16_t* __restrict__ x, uint32_t M, uint32_t K, uint32_t ld_s,
                 uint8_t* __restrict__ q, float* __restrict__ s, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[W][D];
  constexpr uint32_t SLOT = kSeg * 2;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t nseg = (K + kSeg - 1) / kSeg;
  const uint64_t units = (uint64_t)M * nseg;
  const uint64_t gw = (uint64_t)blockIdx.x * W + warp, GW = (uint64_t)gridDim.x * W;
  const uint32_t slot0 = smem_addr(dsm) + warp * D * SLOT;
  const uint32_t bar0 = smem_addr(&full[warp][0]);
  if (lane == 0) {
    for (int d = 0; d < D; ++d) mbar_init_s(bar0 + 8 * d, 1);
    mbar_fence_init();
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();
  auto issue = [&](uint64_t j) {
    const uint64_t u = gw + j * GW;
    if (u >= units) return;
    const uint32_t row = (uint32_t)(u / nseg), col0 = (uint32_t)(u % nseg) * kSeg;
    const uint32_t bytes = min(K - col0, kSeg) * 2u, d = (uint32_t)(j % D);
    mbar_expect_tx(bar0 + 8 * d, bytes);
    bulk_g2s(slot0 + d * SLOT, x + (size_t)row * K + col0, bytes, bar0 + 8 * d, pol);
  };
  if (lane == 0)
    for (int d = 0; d < D; ++d) issue(d);
  uint64_t j = 0;
  bool ok = true;
  for (; gw + j * GW < units; ++j) {
    const uint64_t u = gw + j * GW;
    const uint32_t row = (uint32_t)(u / nseg), col0 = (uint32_t)(u % nseg) * kSeg;
    const uint32_t ng = min(K - col0, kSeg) >> 7, d = (uint32_t)(j % D);
    if (!mbar_wait_bounded(bar0 + 8 * d, (uint32_t)(j / D) & 1u)) {
      ok = false;
      break;
    }
    const uint32_t sb = slot0 + d * SLOT;
    uint8_t* qr = q + (size_t)row * K + col0;
    for (uint32_t g0 = 0; g0 < ng; g0 += 8) {
      uint32_t w[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t grp = g0 + 4 * h + g4;
        if (grp < ng) {
          load_group16(sb + grp * 256u, l8, w[h]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) w[h][k] = 0;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t grp = g0 + 4 * h + g4;
        const bool valid = grp < ng;
        float S;
        uint2 c0, c1;
        group16_codes(w[h], valid, S, c0, c1);
        if (valid) {
          *reinterpret_cast<uint2*>(qr + grp * 128u + l8 * 8u) = c0;
          *reinterpret_cast<uint2*>(qr + grp * 128u + 64u + l8 * 8u) = c1;
          if (l8 == 0) s[(size_t)((col0 >> 7) + grp) * ld_s + row] = S;
        }
      }
    }
    __syncwarp();
    if (lane == 0) issue(j + D);
  }
  if (!ok && lane == 0) record_timeout(nullptr, err);
  // copies still in flight into this warp's slots land before the CTA exits
  if (lane == 0)
    for (uint64_t jj = j; jj < j + D && gw + jj * GW < units; ++jj)
      mbar_wait_bounded(bar0 + 8 * (uint32_t)(jj % D), (uint32_t)(jj / D) & 1u);
}

// R1 on a row stream: one unit = one whole row (H ≤ SLOT_ELEMS), γ staged in
// shared memory once per CTA.  Σx² in FP32: per lane a 16-term FMA chain per
// group, the lane's groups (at most SLOT_ELEMS/512 = 16) added as a binary
// tree, the 32 lanes by a butterfly; r = RN(1/sqrt(RN(Σx²·RN(1/H)) + eps))
// (IEEE reciprocal square root).  With at most 16 + 4 + 5 roundings on a sum
// of positive terms, the relative error of Σx² is at most 25·2^-24 (first
// order), and that of r at most 14.25·2^-24.  y = bf16(RN(RN(x·γ)·r)): x·γ is
// exact (a product of two bf16 values) while it stays a normal FP32 number, which
// holds for every row whose Σx² is itself accurate (|x| within about 1e-19..1e19)
// when 1e-19 < |γ| < 1e19; the quantiser then works on -y, which the same
// roundings give directly from -r.
// With one slot per warp (D = 1) the row arrives in P parts, each with its own
// barrier: once the quantising pass has left a part, the next row's copy of that
// part is requested, so the next row streams in while this one is finished.
template <int W, int D, uint32_t SLOT_ELEMS, int P>
__global__ void __launch_bounds__(32 * W, 1)
k_rmsnorm_quant_tma(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps,
                    float inv_h, uint32_t M, uint32_t H, uint32_t ld_s, uint8_t* __restrict__ q,
                    float* __restrict__ s, float* __restrict__ rstd, uint16_t* __restrict__ y,
                    unsigned* err) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[W][D * P];
  __shared__ __align__(8) uint64_t gbar;
  constexpr uint32_t SLOT = SLOT_ELEMS * 2;
  constexpr int NC = (int)(SLOT_ELEMS / 512);               // 4-group chunks of a slot
  constexpr uint32_t GP = SLOT_ELEMS / 128 / P;             // groups per part
  constexpr int KP = (int)GP / 4;                           // chunks per part
  static_assert(P == 1 || D == 1, "parts need one slot per warp");
  static_assert(KP >= 1 && NC % KP == 0, "a part is whole 4-group chunks");
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t gsm = smem_addr(dsm);                       // γ
  const uint32_t slot0 = gsm + SLOT + warp * D * SLOT;
  const uint32_t bar0 = smem_addr(&full[warp][0]), gb = smem_addr(&gbar);
  const uint64_t gw = (uint64_t)blockIdx.x * W + warp, GW = (uint64_t)gridDim.x * W;
  const uint32_t ng = H >> 7;
  if (threadIdx.x == 0) {
    mbar_init_s(gb, 1);
    mbar_fence_init();
    mbar_expect_tx(gb, H * 2u);
    bulk_g2s_plain(gsm, gamma, H * 2u, gb);
  }
  if (lane == 0) {
    for (int d = 0; d < D * P; ++d) mbar_init_s(bar0 + 8 * d, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const uint64_t pol = policy_evict_first();
  // part p of unit j: groups [p·GP, min(ng, (p+1)·GP)) into slot j mod D
  auto issue = [&](uint64_t j, uint32_t p) {
    const uint64_t row = gw + j * GW;
    const uint32_t lo = p * GP, hi = min(ng, lo + GP);
    if (row >= M || lo >= hi) return;
    const uint32_t d = (uint32_t)(j % D), bar = bar0 + 8 * (d * P + p);
    mbar_expect_tx(bar, (hi - lo) * 256u);
    bulk_g2s(slot0 + d * SLOT + lo * 256u, x + (size_t)row * H + lo * 128u, (hi - lo) * 256u, bar, pol);
  };
  if (lane == 0)
    for (int d = 0; d < D; ++d)
      for (int p = 0; p < P; ++p) issue(d, p);
  bool ok = mbar_wait_bounded(gb, 0);
  uint64_t j = 0;
  for (; ok && gw + j * GW < M; ++j) {
    const uint32_t row = (uint32_t)(gw + j * GW), d = (uint32_t)(j % D);
    const uint32_t ph = (uint32_t)(j / D) & 1u;
    const uint32_t sb = slot0 + d * SLOT;
    // chunk sums of the lane's groups g4, g4 + 4, ... (zero past the row); each
    // part is waited for before its first chunk
    bool got = true;
    float cs[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      if (k % KP == 0 && (uint32_t)(k / KP) * GP < ng)
        got = got && mbar_wait_bounded(bar0 + 8 * (d * P + k / KP), ph);
      const uint32_t grp = g4 + 4u * k;
      float c = 0.0f;
      if (grp < ng) {
        uint32_t w[8];
        load_group16(sb + grp * 256u, l8, w);
        c = add_squares16(w, c);
      }
      cs[k] = c;
    }
    if (!got) {
      ok = false;
      break;
    }
#pragma unroll
    for (int width = NC / 2; width >= 1; width /= 2)
#pragma unroll
      for (int k = 0; k < width; ++k) cs[k] = __fadd_rn(cs[k], cs[k + width]);
    float ss = cs[0];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, o));
    const float r = __frsqrt_rn(__fadd_rn(__fmul_rn(ss, inv_h), eps));
    if (lane == 0) rstd[row] = r;
    const uint64_t nr2 = pack_f2(-r, -r);
    for (uint32_t g0 = 0; g0 < ng; g0 += 4) {
      const uint32_t grp = g0 + g4;
      const bool valid = grp < ng;
      uint32_t wx[8], wg[8];
      if (valid) {
        load_group16(sb + grp * 256u, l8, wx);
        load_group16(gsm + grp * 256u, l8, wg);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) wx[k] = wg[k] = 0;
      }
      uint32_t nyb[8];   // -y
#pragma unroll
      for (int k = 0; k < 8; ++k) nyb[k] = neg_norm_pair(wx[k], wg[k], nr2);
      float S;
      uint2 c0, c1;
      group16_codes_neg(nyb, valid, S, c0, c1);
      if (valid) {
        uint8_t* qg = q + (size_t)row * H + grp * 128u;
        *reinterpret_cast<uint2*>(qg + l8 * 8u) = c0;
        *reinterpret_cast<uint2*>(qg + 64u + l8 * 8u) = c1;
        if (y != nullptr) {
          constexpr uint32_t kNeg = 0x80008000u;
          uint16_t* yr = y + (size_t)row * H + grp * 128u;
          *reinterpret_cast<uint4*>(yr + l8 * 8u) =
              make_uint4(nyb[0] ^ kNeg, nyb[1] ^ kNeg, nyb[2] ^ kNeg, nyb[3] ^ kNeg);
          *reinterpret_cast<uint4*>(yr + 64u + l8 * 8u) =
              make_uint4(nyb[4] ^ kNeg, nyb[5] ^ kNeg, nyb[6] ^ kNeg, nyb[7] ^ kNeg);
        }
        if (l8 == 0) s[(size_t)grp * ld_s + row] = S;
      }
      // the warp has left part g0 / GP: the slot's next row may take it
      if ((g0 + 4u) % GP == 0 || g0 + 4u >= ng) {
        __syncwarp();
        if (lane == 0) issue(j + D, g0 / GP);
      }
    }
  }
  if (!ok && lane == 0) record_timeout(nullptr, err);
  if (lane == 0) {
    for (uint64_t jj = j; jj < j + D && gw + jj * GW < M; ++jj)
      for (uint32_t p = 0; p < (uint32_t)P && p * GP < ng; ++p)
        mbar_wait_bounded(bar0 + 8 * ((uint32_t)(jj % D) * P + p), (uint32_t)(jj / D) & 1u);
    if (warp == 0 && !ok) mbar_wait_bounded(gb, 0);
  }
}

// ---------------------------------------------------------------------------
// Tile pipelines (Q2, Q3, Q4)
// ---------------------------------------------------------------------------
constexpr int kMaxWG = 4, kRing = 2;

struct TileRing {
  uint64_t full[kMaxWG][kRing];
  uint64_t empty[kMaxWG][kRing];
  // Q2: per-warp block maxima of a warpgroup's tiles, double-buffered by tile
  // parity, each buffer with a barrier the 8 warps arrive on (a bounded wait
  // instead of a warpgroup barrier, so a warp that gives up cannot strand the others)
  uint64_t redbar[kMaxWG][2];
  float red[kMaxWG][2][8];
};

// Warpgroup w of CTA b takes the tiles j·(gridDim·NWG) + b·NWG + w; its tile j
// sits in its stage j mod 2.  The warpgroup's first thread fills a stage
// (`issue(tile, stage address, full barrier)`, STAGE_TX bytes) once all 8 warps
// have released it, one tile ahead of the tile being quantised.  `consume(tile,
// stage address, warpgroup, thread in warpgroup, j, ring, release)` quantises a
// tile and calls release() after its warp's last read of the stage.
template <int NWG, uint32_t STAGE_BYTES, uint32_t STAGE_TX, class Issue, class Consume>
__device__ __forceinline__ void run_tile_pipeline(uint32_t ntiles, unsigned* err, Issue issue,
                                                  Consume consume) {
  static_assert(NWG <= kMaxWG && STAGE_BYTES % 1024 == 0, "stages 1024-byte aligned (128-byte swizzle)");
  extern __shared__ __align__(1024) uint8_t dsm[];
  __shared__ TileRing ring;
  const uint32_t base = (smem_addr(dsm) + 1023u) & ~1023u;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t wg = warp >> 3, tid = threadIdx.x & 255u;
  const uint32_t first = blockIdx.x * NWG + wg, step = gridDim.x * NWG;
  const uint32_t nj = first < ntiles ? (ntiles - first + step - 1) / step : 0u;
  const uint32_t st0 = base + wg * kRing * STAGE_BYTES;
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init_s(smem_addr(&ring.full[wg][i]), 1);
      mbar_init_s(smem_addr(&ring.empty[wg][i]), 8);
    }
    mbar_init_s(smem_addr(&ring.redbar[wg][0]), 8);
    mbar_init_s(smem_addr(&ring.redbar[wg][1]), 8);
    mbar_fence_init();
  }
  __syncthreads();
  auto fill = [&](uint32_t j) {
    const uint32_t st = j % kRing, fb = smem_addr(&ring.full[wg][st]);
    mbar_expect_tx(fb, STAGE_TX);
    issue(first + j * step, st0 + st * STAGE_BYTES, fb);
  };
  uint32_t issued = 0;   // tiles whose copies this warpgroup's first thread started
  if (tid == 0)
    for (; issued < kRing && issued < nj; ++issued) fill(issued);
  bool ok = true;
  uint32_t j = 0;
  for (; j < nj; ++j) {
    const uint32_t st = j % kRing;
    if (tid == 0 && j >= 1 && issued < nj) {
      // refill the stage of tile j-1 with tile j+1 once all warps released it
      const uint32_t sp = (j - 1) % kRing;
      if (!mbar_wait_bounded(smem_addr(&ring.empty[wg][sp]), ((j - 1) / kRing) & 1u)) {
        record_timeout(nullptr, err);
        ok = false;
      } else {
        fill(issued++);
      }
    }
    if (!ok || !mbar_wait_bounded(smem_addr(&ring.full[wg][st]), (j / kRing) & 1u)) {
      if (lane == 0) record_timeout(nullptr, err);
      break;
    }
    const uint32_t eb = smem_addr(&ring.empty[wg][st]);
    consume(first + j * step, st0 + st * STAGE_BYTES, wg, tid, j, &ring, [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive_s(eb);
    });
  }
  // the copies this warpgroup started land before the CTA's shared memory goes away
  if (tid == 0)
    for (uint32_t jj = j; jj < issued; ++jj)
      mbar_wait_bounded(smem_addr(&ring.full[wg][jj % kRing]), (jj / kRing) & 1u);
}

// Row pass of a bf16 tile (two 64-column boxes, 16 KB apart): thread (rg, cg)
// = (tid/16, tid%16) loads rows 8rg + i, columns 8cg + 0..7.
__device__ __forceinline__ void load_rows_bf16(uint32_t sbase, uint32_t tid, uint32_t (&w)[8][4]) {
  const uint32_t rg = tid >> 4, cg = tid & 15u;
  const uint32_t b = sbase + (cg >> 3) * 16384u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = lds128(b + sw128(8u * rg + i, cg & 7u));
    w[i][0] = v.x; w[i][1] = v.y; w[i][2] = v.z; w[i][3] = v.w;
  }
}
// Column pass of a bf16 tile: thread (rg, cg) = (tid%16, tid/16) loads
// columns 8cg + 0..7 of rows 8rg + ((i + rg) mod 8) into slot i.
__device__ __forceinline__ void load_cols_bf16(uint32_t sbase, uint32_t tid, uint32_t (&w)[8][4]) {
  const uint32_t rg = tid & 15u, cg = tid >> 4;
  const uint32_t b = sbase + (cg >> 3) * 16384u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = lds128(b + sw128(8u * rg + ((i + rg) & 7u), cg & 7u));
    w[i][0] = v.x; w[i][1] = v.y; w[i][2] = v.z; w[i][3] = v.w;
  }
}

// Maxima over a half-warp of 8 per-lane values held as 4 packed bf16 pairs
// r[k] = (value 2k, value 2k + 1) (magnitudes; sign bits not meaningful),
// reduced transposed: each exchange hands the partner the half of the values it
// keeps, so 5 shuffles replace 16.  Lane l (bits b0, b1, b2 of l) ends with the
// maximum of value 4·b1 + 2·b0 + b2; value i sits in lane half_warp_lane_of(i).
__device__ __forceinline__ float half_warp_max8_packed(const uint32_t (&r)[4]) {
  const uint32_t lane = threadIdx.x & 31u;
  const bool b0 = lane & 1u, b1 = lane & 2u, b2 = lane & 4u;
  uint32_t r1[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t keep = b0 ? r[2 * j + 1] : r[2 * j], send = b0 ? r[2 * j] : r[2 * j + 1];
    r1[j] = amax2(keep, __shfl_xor_sync(kFull, send, 1));
  }
  const uint32_t keep = b1 ? r1[1] : r1[0], send = b1 ? r1[0] : r1[1];
  const uint32_t r2 = amax2(keep, __shfl_xor_sync(kFull, send, 2)) & 0x7FFF7FFFu;
  const float lo = bf_lo(r2), hi = bf_hi(r2);
  const float r3 = fmaxf(b2 ? hi : lo, __shfl_xor_sync(kFull, b2 ? lo : hi, 4));
  return fmaxf(r3, __shfl_xor_sync(kFull, r3, 8));
}
__host__ __device__ constexpr uint32_t half_warp_lane_of(int i) {
  return (uint32_t)(((i >> 1) & 1) | ((i >> 2) << 1) | ((i & 1) << 2));
}

// Group constants of 8 groups whose maxima half_warp_max8_packed left one per
// lane: lane l computes its group's S and -RN(1/S), the half-warp shares them by
// shuffle; bit i of the returned mask marks group i as slow.
__device__ __forceinline__ uint32_t half_warp_qscales_packed(float a, float (&s)[8], float (&ny)[8]) {
  const uint32_t base = threadIdx.x & 16u;
  const float s_mine = make_scale(a).s;
  const float ny_mine = -__frcp_rn(s_mine);
  const uint32_t bits = (__ballot_sync(kFull, a != 0.0f && a < kQuotientMinAmax) >> base) & 0xFFu;
  uint32_t mask = 0;
  if (bits) {
#pragma unroll
    for (int i = 0; i < 8; ++i) mask |= ((bits >> half_warp_lane_of(i)) & 1u) << i;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s[i] = __shfl_sync(kFull, s_mine, base + half_warp_lane_of(i));
    ny[i] = __shfl_sync(kFull, ny_mine, base + half_warp_lane_of(i));
  }
  return mask;
}

// Row pass: the constants of the 8 rows' groups (each row's 128-column group
// spans the half-warp).
__device__ __forceinline__ uint32_t row_group_qscales(const uint32_t (&w)[8][4], float (&s)[8], float (&ny)[8]) {
  uint32_t r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t m0 = amax2(amax2(w[2 * k][0], w[2 * k][1]), amax2(w[2 * k][2], w[2 * k][3]));
    const uint32_t m1 = amax2(amax2(w[2 * k + 1][0], w[2 * k + 1][1]), amax2(w[2 * k + 1][2], w[2 * k + 1][3]));
    // rows 2k (low half) and 2k+1 (high half): low halves against high halves
    r[k] = amax2(__byte_perm(m0, m1, 0x5410), __byte_perm(m0, m1, 0x7632));
  }
  return half_warp_qscales_packed(half_warp_max8_packed(r), s, ny);
}

// Column pass: the constants of the thread's 8 columns' groups (the maxima over
// the 128 rows of the tile; a column group spans the half-warp).
__device__ __forceinline__ uint32_t col_group_qscales(const uint32_t (&w)[8][4], float (&s)[8], float (&ny)[8]) {
  uint32_t r[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t m = w[0][c];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = amax2(m, w[i][c]);
    r[c] = m;
  }
  return half_warp_qscales_packed(half_warp_max8_packed(r), s, ny);
}

// Codes of the 8 rows of a row-pass block under per-row constants (s[i],
// ny[i]); row i's 8 codes (columns in order) go to put(i, codes).  Rows whose
// group is slow (bit i of `slow`) are stored again from scaled operands.
template <class Put>
__device__ __forceinline__ void row_codes_bf16(const uint32_t (&w)[8][4], const float (&s)[8],
                                               const float (&ny)[8], uint32_t slow, Put put) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const QScale g = qscale_of(s[i], ny[i]);
    put(i, make_uint2(codes4_bf16(w[i][0], w[i][1], g), codes4_bf16(w[i][2], w[i][3], g)));
  }
  if (slow) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (slow & (1u << i))
        put(i, make_uint2(codes4_tiny(bf2_to_f2(w[i][0]), bf2_to_f2(w[i][1]), s[i]),
                          codes4_tiny(bf2_to_f2(w[i][2]), bf2_to_f2(w[i][3]), s[i])));
  }
}

// Codes of the 8 columns of a column-pass block under per-column constants:
// column j's 8 codes in slot order (rotated rows) go to put(j, lo, hi).
template <class Put>
__device__ __forceinline__ void col_codes_bf16(const uint32_t (&w)[8][4], const float (&s)[8],
                                               const float (&ny)[8], uint32_t slow, Put put) {
  // column j, slots (i, i+1): the pair's bf16 values from two row words
  auto pair = [&](int j, int i) { return __byte_perm(w[i][j >> 1], w[i + 1][j >> 1], (j & 1) ? 0x7632 : 0x5410); };
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const QScale g = qscale_of(s[j], ny[j]);
    put(j, codes4_bf16(pair(j, 0), pair(j, 2), g), codes4_bf16(pair(j, 4), pair(j, 6), g));
  }
  if (slow) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (slow & (1u << j))
        put(j, codes4_tiny(bf2_to_f2(pair(j, 0)), bf2_to_f2(pair(j, 2)), s[j]),
            codes4_tiny(bf2_to_f2(pair(j, 4)), bf2_to_f2(pair(j, 6)), s[j]));
  }
}

struct Q4Args {
  uint32_t M, N, ld_srow;
  uint8_t* q_row;
  float* s_row;
  uint8_t* qT_col;
  float* sT_col;
  unsigned* err;
};

constexpr int kBf16WG = 2;     // warpgroups per CTA for 32 KB bf16 tiles (two-tile rings: 128 KB); 3 spill at 85 registers and run slower

// Q4: one read of the bf16 gradient → 1×128 row groups along N (stored as is)
// and 128×1 column groups along M (stored transposed).
__global__ void __launch_bounds__(256 * kBf16WG, 1)
k_quant_grad_dual_tma(const __grid_constant__ CUtensorMap map, const Q4Args a) {
  const uint32_t nb_n = a.N / 128, ntiles = (a.M / 128) * nb_n;
  const uint64_t pol = policy_evict_first();
  auto issue = [&](uint32_t tile, uint32_t dst, uint32_t fb) {
    const int m0 = (int)(tile / nb_n) * 128, n0 = (int)(tile % nb_n) * 128;
    tma_g2s_2d(dst, &map, fb, n0, m0, pol);
    tma_g2s_2d(dst + 16384u, &map, fb, n0 + 64, m0, pol);
  };
  auto consume = [&](uint32_t tile, uint32_t sb, uint32_t, uint32_t tid, uint32_t, TileRing*, auto release) {
    const uint32_t mb = tile / nb_n, nb = tile % nb_n;
    const size_t m0 = (size_t)mb * 128, n0 = (size_t)nb * 128;
    {  // row groups
      uint32_t w[8][4];
      load_rows_bf16(sb, tid, w);
      float sc[8], ny[8];
      const uint32_t slow = row_group_qscales(w, sc, ny);
      const uint32_t rg = tid >> 4, cg = tid & 15u;
      uint8_t* qp = a.q_row + (m0 + 8 * rg) * a.N + n0 + 8 * cg;
      row_codes_bf16(w, sc, ny, slow, [&](int i, uint2 c) { *reinterpret_cast<uint2*>(qp + (size_t)i * a.N) = c; });
      if (cg == 0) {
        float* sp = a.s_row + (size_t)nb * a.ld_srow + m0 + 8 * rg;
        *reinterpret_cast<float4*>(sp) = make_float4(sc[0], sc[1], sc[2], sc[3]);
        *reinterpret_cast<float4*>(sp + 4) = make_float4(sc[4], sc[5], sc[6], sc[7]);
      }
    }
    {  // column groups, stored transposed
      uint32_t w[8][4];
      load_cols_bf16(sb, tid, w);
      release();
      float sc[8], ny[8];
      const uint32_t slow = col_group_qscales(w, sc, ny);
      const uint32_t rg = tid & 15u, cg = tid >> 4;
      uint8_t* qp = a.qT_col + (n0 + 8 * cg) * a.M + m0 + 8 * rg;
      col_codes_bf16(w, sc, ny, slow, [&](int j, uint32_t lo, uint32_t hi) {
        *reinterpret_cast<uint2*>(qp + (size_t)j * a.M) = unrotate8(lo, hi, unrotate_selectors(rg & 7u));
      });
      if (rg == 0) {
        float* sp = a.sT_col + (size_t)mb * a.N + n0 + 8 * cg;
        *reinterpret_cast<float4*>(sp) = make_float4(sc[0], sc[1], sc[2], sc[3]);
        *reinterpret_cast<float4*>(sp + 4) = make_float4(sc[4], sc[5], sc[6], sc[7]);
      }
    }
  };
  run_tile_pipeline<kBf16WG, 32768u, 32768u>(ntiles, a.err, issue, consume);
}

struct Q2Args {
  uint32_t N, K;
  uint8_t* q;
  float* s;
  uint8_t* qT;
};

// Up to JETFP8_MAX_GROUP weights quantised by one launch: problem p owns the
// global tiles [tile_end[p-1], tile_end[p]) (tile_end[-1] = 0), each problem's
// tiles in its own row-major block order.
struct Q2Params {
  CUtensorMap map[JETFP8_MAX_GROUP];
  Q2Args a[JETFP8_MAX_GROUP];
  uint32_t tile_end[JETFP8_MAX_GROUP];
  uint32_t count;
  unsigned* err;
};

// Q2: 128×128 weight blocks; the optional transposed payload Ŵᵀ holds the
// same codes (each column of the block quantised again with the block's scale).
__global__ void __launch_bounds__(256 * kBf16WG, 1)
k_quant_weight_tma(const __grid_constant__ Q2Params P) {
  const uint64_t pol = policy_evict_first();
  // global tile -> (problem, tile within it)
  auto locate = [&](uint32_t tile, uint32_t& local) {
    uint32_t p = 0, start = 0;
#pragma unroll
    for (uint32_t i = 0; i + 1 < JETFP8_MAX_GROUP; ++i)
      if (i + 1 < P.count && tile >= P.tile_end[i]) {
        p = i + 1;
        start = P.tile_end[i];
      }
    local = tile - start;
    return p;
  };
  auto issue = [&](uint32_t tile, uint32_t dst, uint32_t fb) {
    uint32_t lt;
    const uint32_t p = locate(tile, lt), kblocks = P.a[p].K / 128;
    const int n0 = (int)(lt / kblocks) * 128, k0 = (int)(lt % kblocks) * 128;
    tma_g2s_2d(dst, &P.map[p], fb, k0, n0, pol);
    tma_g2s_2d(dst + 16384u, &P.map[p], fb, k0 + 64, n0, pol);
  };
  auto consume = [&](uint32_t tile, uint32_t sb, uint32_t wg, uint32_t tid, uint32_t j, TileRing* ring,
                     auto release) {
    uint32_t lt;
    const Q2Args& a = P.a[locate(tile, lt)];
    const uint32_t kblocks = a.K / 128;
    const uint32_t nb = lt / kblocks, kb = lt % kblocks;
    const size_t n0 = (size_t)nb * 128, k0 = (size_t)kb * 128;
    uint32_t w[8][4];
    load_rows_bf16(sb, tid, w);
    if (a.qT == nullptr) release();
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = amax2(m, amax2(amax2(w[i][0], w[i][1]), amax2(w[i][2], w[i][3])));
    m &= 0x7FFF7FFFu;
    float amax = fmaxf(bf_lo(m), bf_hi(m));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    // the warpgroup's j-th tile uses buffer j mod 2 for the (j/2)-th time
    const uint32_t buf = j & 1u;
    float* red = ring->red[wg][buf];
    const uint32_t rb = smem_addr(&ring->redbar[wg][buf]);
    if ((tid & 31u) == 0) {
      red[tid >> 5] = amax;
      mbar_arrive_s(rb);   // release: the write above is seen by the waiters
    }
    if (!mbar_wait_bounded(rb, (j >> 1) & 1u)) {
      if ((tid & 31u) == 0) record_timeout(nullptr, P.err);
      if (a.qT != nullptr) release();
      return;
    }
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    float sc[8], ny[8];
    sc[0] = make_scale(amax).s;
    ny[0] = -__frcp_rn(sc[0]);
    const uint32_t slow = (amax != 0.0f && amax < kQuotientMinAmax) ? 0xFFu : 0u;
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      sc[i] = sc[0];
      ny[i] = ny[0];
    }
    if (tid == 0) a.s[(size_t)nb * kblocks + kb] = sc[0];
    const uint32_t rg = tid >> 4, cg = tid & 15u;
    uint8_t* qp = a.q + (n0 + 8 * rg) * a.K + k0 + 8 * cg;
    row_codes_bf16(w, sc, ny, slow, [&](int i, uint2 c) { *reinterpret_cast<uint2*>(qp + (size_t)i * a.K) = c; });
    if (a.qT != nullptr) {
      load_cols_bf16(sb, tid, w);
      release();
      const uint32_t rgc = tid & 15u, cgc = tid >> 4;
      uint8_t* tp = a.qT + (k0 + 8 * cgc) * a.N + n0 + 8 * rgc;
      col_codes_bf16(w, sc, ny, slow, [&](int c, uint32_t lo, uint32_t hi) {
        *reinterpret_cast<uint2*>(tp + (size_t)c * a.N) = unrotate8(lo, hi, unrotate_selectors(rgc & 7u));
      });
    }
  };
  run_tile_pipeline<kBf16WG, 32768u, 32768u>(P.tile_end[P.count - 1], P.err, issue, consume);
}

struct Q3Args {
  uint32_t M, K;
  const float* s;
  uint8_t* qT;
  float* sT;
  unsigned* err;
};

constexpr int kQ3WG = 2;       // warpgroups per CTA for 17 KB code tiles (two-tile rings: 68 KB)

// Q3: dequantise 1×128 row groups (x̃ = fp32(dec(q)·S)), requantise in 128×1
// column groups, store transposed.  A stage holds the 128×128 code tile
// (one 128-byte swizzled box) and the tile rows' 128 scales.
__global__ void __launch_bounds__(256 * kQ3WG, 1)
k_requant_row2col_tma(const __grid_constant__ CUtensorMap map, const Q3Args a) {
  constexpr uint32_t STAGE = 17408;   // 16 KB codes + 512 B scales, padded to 1 KB
  const uint32_t kblocks = a.K / 128, ntiles = (a.M / 128) * kblocks;
  const uint64_t pol = policy_evict_first();
  auto issue = [&](uint32_t tile, uint32_t dst, uint32_t fb) {
    const uint32_t mb = tile / kblocks, kb = tile % kblocks;
    tma_g2s_2d(dst, &map, fb, (int)(kb * 128), (int)(mb * 128), pol);
    bulk_g2s(dst + 16384u, a.s + (size_t)kb * a.M + (size_t)mb * 128, 512u, fb, pol);
  };
  auto consume = [&](uint32_t tile, uint32_t sb, uint32_t, uint32_t tid, uint32_t, TileRing*, auto release) {
    const uint32_t mb = tile / kblocks, kb = tile % kblocks;
    const size_t m0 = (size_t)mb * 128, k0 = (size_t)kb * 128;
    const uint32_t rg = tid & 15u, cg = tid >> 4;
    // slot i: row 8rg + ((i + rg) mod 8), columns 8cg + 0..7 (8 codes) and the row's scale
    uint2 u[8];
    float sr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t r = 8u * rg + ((i + rg) & 7u);
      u[i] = lds64(sb + sw128(r, cg >> 1) + ((cg & 1u) << 3));
      sr[i] = lds32f(sb + 16384u + r * 4u);
    }
    release();
    // nx[j][p] = -x̃ of column j in slots (2p, 2p+1): the two codes side by
    // side (byte permute), decoded exactly (E4M3 -> f16 -> FP32) and multiplied
    // by the negated row scales (one FP32 multiply each: the exact negative of x̃)
    uint64_t nx[8][4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint64_t ns = pack_f2(-sr[2 * p], -sr[2 * p + 1]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w0 = j < 4 ? u[2 * p].x : u[2 * p].y, w1 = j < 4 ? u[2 * p + 1].x : u[2 * p + 1].y;
        const uint32_t sel = (uint32_t)(j & 3) | ((4u + (uint32_t)(j & 3)) << 4);   // byte j%4 of w0, then of w1
        const uint16_t two = (uint16_t)__byte_perm(w0, w1, sel);
        uint32_t hh;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(two));
        const uint64_t v = pack_f2(h2f((uint16_t)(hh & 0xFFFFu)), h2f((uint16_t)(hh >> 16)));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(nx[j][p]) : "l"(v), "l"(ns));
      }
    }
    float amax[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 v0 = bits_f2(nx[j][0]), v1 = bits_f2(nx[j][1]), v2 = bits_f2(nx[j][2]), v3 = bits_f2(nx[j][3]);
      const float m = max3_abs(max3_abs(v0.x, v0.y, v1.x), max3_abs(v1.y, v2.x, v2.y), max3_abs(v3.x, v3.y, 0.0f));
      amax[j] = m;
    }
    float sc[8], ny[8];
    const uint32_t slow = half_warp_qscales_of(half_warp_colmax8(amax), sc, ny);
    uint8_t* qp = a.qT + (k0 + 8 * cg) * a.M + m0 + 8 * rg;
    auto put = [&](int jj, uint32_t lo, uint32_t hi) {
      *reinterpret_cast<uint2*>(qp + (size_t)jj * a.M) = unrotate8(lo, hi, unrotate_selectors(rg & 7u));
    };
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const QScale g = qscale_of(sc[jj], ny[jj]);
      put(jj, codes4_neg_f32(nx[jj][0], nx[jj][1], g), codes4_neg_f32(nx[jj][2], nx[jj][3], g));
    }
    if (slow) {
      auto xpair = [&](int jj, int p) {
        const float2 v = bits_f2(nx[jj][p]);
        return make_float2(-v.x, -v.y);
      };
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (slow & (1u << jj))
          put(jj, codes4_tiny(xpair(jj, 0), xpair(jj, 1), sc[jj]), codes4_tiny(xpair(jj, 2), xpair(jj, 3), sc[jj]));
    }
    if (rg == 0) {
      float* sp = a.sT + (size_t)mb * a.K + k0 + 8 * cg;
      *reinterpret_cast<float4*>(sp) = make_float4(sc[0], sc[1], sc[2], sc[3]);
      *reinterpret_cast<float4*>(sp + 4) = make_float4(sc[4], sc[5], sc[6], sc[7]);
    }
  };
  run_tile_pipeline<kQ3WG, STAGE, 16384u + 512u>(ntiles, a.err, issue, consume);
}

// ---------------------------------------------------------------------------
// R1: RMSNorm fused with the 1×128 quantiser.  One warp per row, 8 lanes per
// group.  Pass 1 accumulates Σx² (16-term FP32 chunk sums per lane, the
// chunks and then the lanes combined in FP64); pass 2 re-reads the row (an
// L1/L2 hit) and writes y, q, S.  Serves rows wider than 8192.
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
    double ss = 0.0;
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
        ss += (double)cs;
      }
    }
    double d = ss;
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
      uint32_t yb[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 t = mul2(mul2(bf2_to_f2(rx[w]), make_float2(r, r)), bf2_to_f2(rg[w]));
        yb[w] = f2_to_bf2(t.x, t.y);
      }
      float S;
      uint2 c0, c1;
      group16_codes(yb, valid, S, c0, c1);
      if (valid) {
        *reinterpret_cast<uint4*>(q + (size_t)row * H + grp * 128 + l8 * 16) = make_uint4(c0.x, c0.y, c1.x, c1.y);
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
// Rows up to 4096 wide run the fused kernel below (∇x and the ∇γ partial sums
// in one pass over x and ∇y).  Wider rows: ∇γ by deterministic two-stage column
// sums — FP32 partial sums over 128-row chunks into the caller's workspace
// [chunks][H], then each column's partials added in a fixed order in FP64.
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

// Partial ∇γ over rows [128p, 128p + 128) for 512 columns per CTA (2 per
// thread); the CTAs of one grid column take the chunks p = blockIdx.y,
// blockIdx.y + gridDim.y, ... (the grid's y extent is capped at 65535).
__global__ void __launch_bounds__(kThreads)
k_rmsnorm_bwd_dgamma_partial(const uint16_t* __restrict__ x, const float* __restrict__ rstd,
                             const uint16_t* __restrict__ dy, uint32_t M, uint32_t H,
                             uint32_t chunks, float* __restrict__ ws) {
  const uint32_t col = blockIdx.x * 512u + 2u * threadIdx.x;
  if (col >= H) return;
  for (uint32_t p = blockIdx.y; p < chunks; p += gridDim.y) {
    const uint32_t r0 = p * kNormBwdRows, r1 = min(M, r0 + kNormBwdRows);
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
}

// The fused backward for rows up to 4096 wide: W warps per CTA, one CTA per SM
// (the accumulators fill shared memory), warp w of CTA b owning the rows
// b·W + w + k·W·gridDim.  Each row's ∇x is formed exactly as by
// k_rmsnorm_bwd_dx (x and ∇y are read twice; few enough rows are in flight for
// the second read to come from L2), and its ∇γ terms RN(RN(dy·x)·r) are added,
// in row order, to the warp's own FP32 accumulator row in shared memory.  At the
// end the CTA adds its W rows in warp order (FP32) into its workspace row; the
// CTA rows are then added in a fixed order in FP64 (k_rmsnorm_bwd_dgamma_reduce).
// An accumulator row keeps lane l8's 16 columns 128g + 16·l8 + 4i + (0..3) at
// 128g + 32i + 4·l8 + (0..3), so the eight lanes of a group touch 128
// consecutive bytes per access.
constexpr uint32_t kNormBwdMaxCtas = 152;   // workspace rows: at most one per CTA

template <int W>
__global__ void __launch_bounds__(32 * W, 1)
k_rmsnorm_bwd_fused(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma,
                    const float* __restrict__ rstd, const uint16_t* __restrict__ dy, uint32_t M,
                    uint32_t H, double inv_h, uint16_t* __restrict__ dx, float* __restrict__ ws) {
  extern __shared__ __align__(16) float acc_s[];   // [W][H]
  constexpr int U = 4;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u, g4 = lane >> 3, l8 = lane & 7u;
  const uint32_t GW = gridDim.x * W;
  const uint32_t groups = H / 128;
  float* acc = acc_s + (size_t)warp * H;
  for (uint32_t i = 4 * lane; i < H; i += 128) *reinterpret_cast<float4*>(acc + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncwarp();
  uint64_t pol_keep, pol_drop;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_drop));
  // each warp asks L2 for its next row of x and ∇y while it works on the
  // current one, so DRAM keeps streaming through the row's FP64 step and second
  // pass (measured at 16384 × 4096: 108 µs one row ahead, 130 two rows ahead,
  // 133 without; the three-kernel path 137)
  auto prefetch_row = [&](uint32_t row) {
    if (lane == 0 && row < M) {
      bulk_prefetch_l2(x + (size_t)row * H, H * 2u);
      bulk_prefetch_l2(dy + (size_t)row * H, H * 2u);
    }
  };
  prefetch_row(blockIdx.x * W + warp);
  for (uint32_t row = blockIdx.x * W + warp; row < M; row += GW) {
    const uint16_t* xr = x + (size_t)row * H;
    const uint16_t* dr = dy + (size_t)row * H;
    prefetch_row(row + GW);
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
    float c = 0.0f;
    // (1/H in FP64: a relative error of 2^-53, far below c's FP32 rounding)
    if (lane == 0) c = (float)((double)r * (double)r * (double)r * d * inv_h);
    c = __shfl_sync(kFull, c, 0);
    constexpr int U2 = 4;   // groups per lane whose loads are in flight together
    for (uint32_t g0 = 0; g0 < groups; g0 += 4 * U2) {
      uint32_t rx[U2][8], rd[U2][8], rg[U2][8];
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        if (grp >= groups) continue;
        ld32_policy(xr + grp * 128 + l8 * 16, rx[u], pol_drop);
        ld32_policy(dr + grp * 128 + l8 * 16, rd[u], pol_drop);
        ld32_cached(gamma + grp * 128 + l8 * 16, rg[u]);
      }
#pragma unroll
      for (int u = 0; u < U2; ++u) {
        const uint32_t grp = g0 + 4 * u + g4;
        if (grp >= groups) continue;
        uint32_t out[8];
        float t[16];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float2 fx = bf2_to_f2(rx[u][w]), fd = bf2_to_f2(rd[u][w]), fg = bf2_to_f2(rg[u][w]);
          const float a = __fsub_rn(__fmul_rn(r, __fmul_rn(fd.x, fg.x)), __fmul_rn(fx.x, c));
          const float b = __fsub_rn(__fmul_rn(r, __fmul_rn(fd.y, fg.y)), __fmul_rn(fx.y, c));
          out[w] = f2_to_bf2(a, b);
          t[2 * w] = __fmul_rn(__fmul_rn(fd.x, fx.x), r);
          t[2 * w + 1] = __fmul_rn(__fmul_rn(fd.y, fx.y), r);
        }
        st32(dx + (size_t)row * H + grp * 128 + l8 * 16, out);
        float* ap = acc + grp * 128 + 4 * l8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float4 v = *reinterpret_cast<float4*>(ap + 32 * i);
          v.x = __fadd_rn(v.x, t[4 * i]);
          v.y = __fadd_rn(v.y, t[4 * i + 1]);
          v.z = __fadd_rn(v.z, t[4 * i + 2]);
          v.w = __fadd_rn(v.w, t[4 * i + 3]);
          *reinterpret_cast<float4*>(ap + 32 * i) = v;
        }
      }
    }
  }
  __syncthreads();
  // stored index s = 128g + 32i + 4l + e holds column 128g + 16l + 4i + e
  float* wrow = ws + (size_t)blockIdx.x * H;
  for (uint32_t s4 = 4 * threadIdx.x; s4 < H; s4 += 4 * 32 * W) {
    float4 v = *reinterpret_cast<const float4*>(acc_s + s4);
#pragma unroll
    for (int w = 1; w < W; ++w) {
      const float4 u = *reinterpret_cast<const float4*>(acc_s + (size_t)w * H + s4);
      v.x = __fadd_rn(v.x, u.x);
      v.y = __fadd_rn(v.y, u.y);
      v.z = __fadd_rn(v.z, u.z);
      v.w = __fadd_rn(v.w, u.w);
    }
    const uint32_t g = s4 >> 7, i = (s4 >> 5) & 3u, l = (s4 >> 2) & 7u;
    *reinterpret_cast<float4*>(wrow + 128 * g + 16 * l + 4 * i) = v;
  }
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
      }
      // the lane's 16 values of h (consecutive) quantised with its group's scale
      float S;
      uint2 c0, c1;
      group16_codes(hb, valid, S, c0, c1);
      if (valid) {
        *reinterpret_cast<uint4*>(q + (size_t)row * I + grp * 128 + l8 * 16) = make_uint4(c0.x, c0.y, c1.x, c1.y);
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
// Dynamic shared memory above 48 KB needs an opt-in per kernel and device.
template <class Kern>
cudaError_t opt_in_smem(Kern kern, int bytes, int (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = 1;
  }
  return cudaSuccess;
}

constexpr int kRowW = 24, kRowD = 2;            // Q1: warps per CTA, slots per warp

cudaError_t launch_quant_rowgroups(const void* x, int64_t M, int64_t K, uint8_t* q, float* s,
                                   cudaStream_t st) {
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  auto kern = k_quant_rows_tma<kRowW, kRowD>;
  constexpr int smem = kRowW * kRowD * (int)kSeg * 2;
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  const size_t units = (size_t)M * ((K + kSeg - 1) / kSeg);
  const unsigned grid = grid_for(units, kRowW, 1);
  kern<<<grid, 32 * kRowW, smem, st>>>(static_cast<const uint16_t*>(x), (uint32_t)M, (uint32_t)K,
                                       (uint32_t)round_up4(M), q, s, err);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight_grouped(int count, const void* const* w, const int64_t* N, const int64_t* K,
                                        uint8_t* const* q, float* const* s, uint8_t* const* qT,
                                        cudaStream_t st) {
  unsigned* err = device_error_word();
  if (err == nullptr || count < 1 || count > JETFP8_MAX_GROUP) return cudaErrorInvalidValue;
  Q2Params P{};
  P.count = (uint32_t)count;
  P.err = err;
  size_t tiles = 0;
  for (int i = 0; i < count; ++i) {
    if (!encode_map_2d(&P.map[i], w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)K[i], (uint64_t)N[i],
                       (uint64_t)K[i] * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
      return cudaErrorInvalidValue;
    P.a[i] = Q2Args{(uint32_t)N[i], (uint32_t)K[i], q[i], s[i], qT == nullptr ? nullptr : qT[i]};
    tiles += (size_t)(N[i] / 128) * (K[i] / 128);
    if (tiles > 0xFFFFFFFFu) return cudaErrorInvalidValue;
    P.tile_end[i] = (uint32_t)tiles;
  }
  auto kern = k_quant_weight_tma;
  constexpr int smem = kBf16WG * kRing * 32768 + 1024;
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  kern<<<grid_for(tiles, kBf16WG, 1), 256 * kBf16WG, smem, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, uint8_t* q, float* s,
                                uint8_t* qT, cudaStream_t st) {
  return launch_quant_weight_grouped(1, &w, &N, &K, &q, &s, &qT, st);
}

cudaError_t launch_requant_row2col(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                   uint8_t* qT, float* sT, cudaStream_t st) {
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!encode_map_2d(&map, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)K, (uint64_t)M, (uint64_t)K, 128,
                     128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  auto kern = k_requant_row2col_tma;
  constexpr int smem = kQ3WG * kRing * 17408 + 1024;
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  const size_t tiles = (size_t)(M / 128) * (K / 128);
  kern<<<grid_for(tiles, kQ3WG, 1), 256 * kQ3WG, smem, st>>>(
      map, Q3Args{(uint32_t)M, (uint32_t)K, s, qT, sT, err});
  return cudaGetLastError();
}

cudaError_t launch_quant_grad_dual(const void* dy, int64_t M, int64_t N, uint8_t* q_row,
                                   float* s_row, uint8_t* qT_col, float* sT_col, cudaStream_t st) {
  if (qT_col == nullptr) return launch_quant_rowgroups(dy, M, N, q_row, s_row, st);
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!encode_map_2d(&map, dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2,
                     64, 128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  auto kern = k_quant_grad_dual_tma;
  constexpr int smem = kBf16WG * kRing * 32768 + 1024;
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  const size_t tiles = (size_t)(M / 128) * (N / 128);
  kern<<<grid_for(tiles, kBf16WG, 1), 256 * kBf16WG, smem, st>>>(
      map, Q4Args{(uint32_t)M, (uint32_t)N, (uint32_t)round_up4(M), q_row, s_row, qT_col, sT_col, err});
  return cudaGetLastError();
}

template <int W, int D, uint32_t SLOT, int P>
cudaError_t launch_rmsnorm_tma(const void* x, const void* gamma, float eps, int64_t M, int64_t H,
                               uint8_t* q, float* s, float* rstd, void* y, unsigned* err, cudaStream_t st) {
  auto kern = k_rmsnorm_quant_tma<W, D, SLOT, P>;
  constexpr int smem = (1 + W * D) * (int)SLOT * 2;
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, smem, done);
  if (e != cudaSuccess) return e;
  kern<<<grid_for((size_t)M, W, 1), 32 * W, smem, st>>>(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(gamma), eps, 1.0f / (float)H, (uint32_t)M,
      (uint32_t)H, (uint32_t)round_up4(M), q, s, rstd, static_cast<uint16_t*>(y), err);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t M,
                                 int64_t H, uint8_t* q, float* s, float* rstd, void* y,
                                 cudaStream_t st) {
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  // rows up to 8192 wide stream whole through shared memory; wider rows take
  // the register kernel (which reads each row twice).  Rows up to 4096 wide:
  // one slot per warp and as many warps as shared memory holds (27, one CTA
  // per SM): the kernel is issue-bound and more warps hide more of each row's
  // latency; 8192 rows then take exactly two rounds.  Graph-timed at 8192 and
  // 32768 rows × 4096: 18, 20, 24, 27 warps give 4304 / 4803, 4254 / 5193,
  // 3821 / 5487, 4717 / 5548 GB/s.  Fewer than 4096 rows spread over more SMs
  // with 8 warps per CTA.  Each row arrives in one piece: graph-timed at 8192 /
  // 32768 rows, one, two, four and eight parts per row (the next row's part
  // requested as soon as the quantising pass has left it) give 4741 / 5305,
  // 4752 / 5395, 4249 / 5212 and 3852 / 4710 GB/s, but inside the layer step
  // two parts measured 3299 - 3424 GB/s against 3410 - 3440 for one.
  if (H <= 4096) {
    if (M >= 4096) return launch_rmsnorm_tma<27, 1, 4096, 1>(x, gamma, eps, M, H, q, s, rstd, y, err, st);
    return launch_rmsnorm_tma<8, 1, 4096, 1>(x, gamma, eps, M, H, q, s, rstd, y, err, st);
  }
  if (H <= 8192) return launch_rmsnorm_tma<6, 2, 8192, 1>(x, gamma, eps, M, H, q, s, rstd, y, err, st);
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_rmsnorm_quant<<<grid, kThreads, 0, st>>>(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(gamma), eps, (uint32_t)M,
      (uint32_t)H, (uint32_t)round_up4(M), q, s, rstd, static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

// Warps per CTA of the fused backward (0: rows too wide, the three-kernel path).
inline int norm_bwd_warps(int64_t H) { return H <= 4096 ? 8 : 0; }
// Workspace rows of the fused backward: one per CTA (at most kNormBwdMaxCtas).
inline int64_t norm_bwd_ctas(int64_t M, int64_t H) {
  const int64_t w = norm_bwd_warps(H), need = (M + w - 1) / w;
  return need < (int64_t)kNormBwdMaxCtas ? need : (int64_t)kNormBwdMaxCtas;
}

size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H) {
  if (norm_bwd_warps(H) > 0) return (size_t)norm_bwd_ctas(M, H) * (size_t)H * sizeof(float);
  return (size_t)((M + kNormBwdRows - 1) / kNormBwdRows) * (size_t)H * sizeof(float);
}

template <int W>
cudaError_t launch_rmsnorm_bwd_fused(const uint16_t* x, const uint16_t* gamma, const float* rstd,
                                     const uint16_t* dy, int64_t M, int64_t H, uint16_t* dx,
                                     float* dgamma, float* ws, cudaStream_t st) {
  auto kern = k_rmsnorm_bwd_fused<W>;
  const int smem = W * (int)H * (int)sizeof(float);
  // (opted in once per device at the widest rows the instance serves, 4096)
  static int done[64] = {0};
  cudaError_t e = opt_in_smem(kern, W * 4096 * (int)sizeof(float), done);
  if (e != cudaSuccess) return e;
  int64_t ctas = norm_bwd_ctas(M, H);
  if (ctas > num_sms()) ctas = num_sms();
  kern<<<(unsigned)ctas, 32 * W, smem, st>>>(x, gamma, rstd, dy, (uint32_t)M, (uint32_t)H, 1.0 / (double)H, dx,
                                             ws);
  k_rmsnorm_bwd_dgamma_reduce<<<(unsigned)((H + 31) / 32), kThreads, 0, st>>>(ws, (uint32_t)ctas,
                                                                            (uint32_t)H, dgamma);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const void* x, const void* gamma, const float* rstd, const void* dy,
                               int64_t M, int64_t H, void* dx, float* dgamma, float* ws,
                               cudaStream_t st) {
  const auto* xb = static_cast<const uint16_t*>(x);
  const auto* db = static_cast<const uint16_t*>(dy);
  const auto* gb = static_cast<const uint16_t*>(gamma);
  auto* dxb = static_cast<uint16_t*>(dx);
  if (norm_bwd_warps(H) == 8) return launch_rmsnorm_bwd_fused<8>(xb, gb, rstd, db, M, H, dxb, dgamma, ws, st);
  const unsigned grid = grid_for((size_t)M, kThreads / 32, 8);
  k_rmsnorm_bwd_dx<<<grid, kThreads, 0, st>>>(xb, static_cast<const uint16_t*>(gamma), rstd, db,
                                              (uint32_t)M, (uint32_t)H, static_cast<uint16_t*>(dx));
  const uint32_t chunks = (uint32_t)((M + kNormBwdRows - 1) / kNormBwdRows);
  const dim3 pgrid((unsigned)((H + 511) / 512), chunks < 65535u ? chunks : 65535u);
  k_rmsnorm_bwd_dgamma_partial<<<pgrid, kThreads, 0, st>>>(xb, rstd, db, (uint32_t)M, (uint32_t)H,
                                                           chunks, ws);
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
