// FP4 variant of the unified precision flow (NVFP4-style), forward GEMM.
//
// The Jet-RL digest ("Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习",
// 未来方向, item (1)) names carrying the unified precision flow to FP4 on
// Blackwell as future work and defines no FP4 format.  This variant keeps the
// flow's property that a token's forward result does not depend on its batch
// (rollout and training see the same numbers), on the FP4 format the tensor
// cores scale in hardware:
//   * E2M1 codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte, the
//     element with the even index in the low nibble;
//   * one E4M3 block scale per 16 consecutive elements along the contraction;
//   * one FP32 scale per row (a token of X, an output channel of W):
//       g = RN(amax_row / 2688), h = RN(6·g), s_b = E4M3(RN(amax_b / h)),
//       d_b = RN(s_b·g), q = E2M1(RN(x / d_b))  (a signed zero when d_b = 0),
//     every step one correctly rounded FP32 operation (the element quotients
//     by the division-free exact sequence in quot2_bf16).
//   Y[m,n] = bf16(RN(RN(D[m,n]·gx[m])·gw[n])),  D = Σ_k x̂q·ŵq (block-scaled).
//
// Block scales live in a blocked layout that the GEMM moves into tensor memory
// without reshuffling: for row r and 16-element block b,
//   byte ((r/128 · K/64 + b/4) · 32 + r mod 32) · 16 + ((r/32) mod 4) · 4 + b mod 4,
// i.e. 512-byte atoms of 128 rows × 64 elements (four blocks), line r mod 32 of
// an atom holding rows r, r+32, r+64, r+96.  The tensor core reads the scale
// of A row m from TMEM lane m, column m/32, and the scale of B row n from
// column n/32 at lane n mod 32 of every lane quarter, byte j for block j of
// the K = 64 MMA (measured on GB300 with a layout probe), so each warp of the
// scale-staging warpgroup writes one atom line per lane, unchanged, into its
// own lane quarter.
//
// GEMM (persistent, one CTA per SM, 512 threads), tile 128 × 256, K in stages
// of 256 elements (128 bytes per row):
//   warp 0      TMA producer: A 16 KB and B 32 KB (128-byte swizzle) and the
//               stage's block-scale atoms (2 + 4 KB, bulk copies), one barrier.
//   warp 1      allocates TMEM (the 256-column accumulator and a ring of
//               block-scale columns); one lane issues four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X per stage.
//   warps 4-7   copy each stage's block scales from shared memory into the
//               stage's TMEM scale columns (tcgen05.st), then signal the MMA.
//   warps 8-15  epilogue, two warps per lane quarter (128 columns each):
//               accumulator → row and column scales → bf16 → global.
// The tensor core applies the block scales, so nothing is promoted per block.
// Every wait is bounded (about 2 s); on expiry the kernel records an error
// word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstring>

#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"
#include "jetfp8_tma.cuh"

namespace jetfp8 {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Quantiser: one warp per row; lane l handles 16-element blocks l, l+32, ...
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_block16(const uint16_t* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                 "=r"(w[7])
               : "l"(p));
}

// Two E2M1 codes, lo in bits 0-3, hi in bits 4-7 (round to nearest even,
// saturating at ±6).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// E4M3 code of v >= 0 (round to nearest even, saturating at 448), and its value.
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// Correctly rounded quotients (x0/d, x1/d) without a division: two Markstein
// corrections of q0 = RN(x·y), y = RN(1/d) (P. Markstein, IBM J. Res. Dev.
// 34(1), 1990), on -x and -y so the sign of a zero survives; the same
// sequence as the E4M3 quantisers'.  Exact while every intermediate is normal,
// which holds for d >= 2^-90 whenever the quotient is 2^-11 or larger; smaller
// quotients stay below 2^-10 with the sign of x, and every such value has the
// E2M1 code of a zero.
// Here for the two bf16 values of w (first value in the low half), each negated
// FP32 value formed in one integer operation: (w << 16) + 2^31 (adding 2^31
// modulo 2^32 flips bit 31) and (w & 0xFFFF0000) ^ 2^31 (lop3, table 0x6A).
__device__ __forceinline__ float2 quot2_bf16(uint32_t w, uint64_t s2, uint64_t ny2) {
  uint64_t q;
  asm("{\n\t.reg .b32 a0, a1;\n\t.reg .b64 nx, r;\n\t"
      "mad.lo.u32 a0, %1, 65536, 0x80000000;\n\t"
      "lop3.b32 a1, %1, 0xFFFF0000, 0x80000000, 0x6A;\n\t"
      "mov.b64 nx, {a0, a1};\n\t"
      "mul.rn.f32x2 %0, nx, %3;\n\t"
      "fma.rn.f32x2 r, %0, %2, nx;\n\t"
      "fma.rn.f32x2 %0, r, %3, %0;\n\t"
      "fma.rn.f32x2 r, %0, %2, nx;\n\t"
      "fma.rn.f32x2 %0, r, %3, %0;\n\t}"
      : "=&l"(q) : "r"(w), "l"(s2), "l"(ny2));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(q));
  return r;
}

// Per half of two packed bf16 pairs: a value whose magnitude is max(|a|, |b|)
// (sign bit not meaningful).
__device__ __forceinline__ uint32_t bf_amax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// The largest magnitude among 8 packed bf16 pairs, as a float.
__device__ __forceinline__ float bf_amax16(const uint32_t (&w)[8]) {
  const uint32_t m = bf_amax2(bf_amax2(bf_amax2(w[0], w[1]), bf_amax2(w[2], w[3])),
                              bf_amax2(bf_amax2(w[4], w[5]), bf_amax2(w[6], w[7]))) & 0x7FFF7FFFu;
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

__device__ __forceinline__ size_t scale_offset(uint32_t r, uint32_t b, uint32_t kg) {
  return ((size_t)((r >> 7) * kg + (b >> 2)) * 32u + (r & 31u)) * 16u + ((r >> 5) & 3u) * 4u + (b & 3u);
}

__global__ void __launch_bounds__(256)
k_quant_nvfp4_rows(const uint16_t* __restrict__ x, uint32_t R, uint32_t K, uint8_t* __restrict__ q,
                   uint8_t* __restrict__ sf, float* __restrict__ g_out) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warps = blockDim.x >> 5;
  const uint32_t nb = K >> 4, kg = K >> 6;
  const uint32_t rows_padded = (R + 127u) & ~127u;
  for (uint32_t r = blockIdx.x * warps + (threadIdx.x >> 5); r < rows_padded; r += gridDim.x * warps) {
    if (r >= R) {
      // padding rows of the last 128-row atom: zero block scales
      for (uint32_t b = lane; b < nb; b += 32) sf[scale_offset(r, b, kg)] = 0;
      continue;
    }
    const uint16_t* xr = x + (size_t)r * K;
    float amax = 0.0f;
    for (uint32_t b = lane; b < nb; b += 32) {
      uint32_t w[8];
      ld_block16(xr + 16u * b, w);
      amax = fmaxf(amax, bf_amax16(w));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
    const float g = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    const float h = __fmul_rn(6.0f, g);
    if (lane == 0) g_out[r] = g;
    uint8_t* qr = q + (size_t)r * (K >> 1);
    for (uint32_t b = lane; b < nb; b += 32) {
      uint32_t w[8];
      ld_block16(xr + 16u * b, w);
      const float ab = bf_amax16(w);
      const uint32_t s = e4m3_code(__fdiv_rn(ab, h));
      const float d = __fmul_rn(dec_e4m3x2(s).x, g);
      uint32_t c[2] = {0u, 0u};
      if (d >= 0x1p-90f) {
        const float ny = -__frcp_rn(d);
        uint64_t s2, ny2;
        asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(d));
        asm("mov.b64 %0, {%1, %1};" : "=l"(ny2) : "f"(ny));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 qq = quot2_bf16(w[i], s2, ny2);
          c[i >> 2] |= e2m1x2(qq.x, qq.y) << (8 * (i & 3));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 fi = bf2_to_f2(w[i]);
          uint32_t byte;
          if (d > 0.0f) {
            byte = e2m1x2(__fdiv_rn(fi.x, d), __fdiv_rn(fi.y, d));
          } else {
            byte = ((__float_as_uint(fi.x) >> 31) << 3) | ((__float_as_uint(fi.y) >> 31) << 7);
          }
          c[i >> 2] |= byte << (8 * (i & 3));
        }
      }
      *reinterpret_cast<uint2*>(qr + 8u * b) = make_uint2(c[0], c[1]);
      sf[scale_offset(r, b, kg)] = (uint8_t)s;
    }
  }
}

// ---------------------------------------------------------------------------
// GEMM
// ---------------------------------------------------------------------------
constexpr int BM = 128, BN = 256;
constexpr int KSTAGE_BYTES = 128;                  // 256 FP4 elements per row per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * KSTAGE_BYTES;         // 16 KB
constexpr int B_BYTES = BN * KSTAGE_BYTES;         // 32 KB
constexpr int SFA_BYTES = 4 * 512;                 // four K = 64 MMAs × one 128-row atom
constexpr int SFB_BYTES = (BN / 128) * 4 * 512;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;   // 54 KB
constexpr int THREADS = 512;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = BN;                       // columns 0..255: the accumulator
constexpr int SF_COLS = 4 * 4 + 4 * 8;             // per stage: SFA 4 × 4, SFB 4 × 8 columns
// + per epilogue warp one row of its 128 column scales (gw), read back as broadcasts
constexpr int GWS_BYTES = 8 * 128 * 4;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 1024 + GWS_BYTES;
static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the 128-byte swizzle");
static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory");
// Instruction descriptor of the block-scaled kinds: A and B E2M1 (format 1,
// bits 7-9 and 10-12), K-major, N/8 in bits 17-22, scale format UE4M3 (bit 23
// = 0), M/16 in bits 24-28; scale-factor IDs (bits 4-5, 29-30) 0.
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sfready[STAGES];
  uint64_t tfull, tempty, done;
  uint32_t tmem_base;
  int abort_flag;
};

struct Fp4Args {
  int M, N, K;
  int tiles_m, tiles_n, m_fastest;
  uint32_t kg;                     // K / 64
  const uint8_t* xsf;
  const uint8_t* wsf;
  const float* gx;
  const float* gw;
  uint16_t* y;
  unsigned* err;
};

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// A bounded wait; on expiry (or when another role has given up) the CTA's
// abort flag is set and the error word records the timeout.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, Bars* bars, unsigned* err) {
  if (mbar_wait_bounded(bar, parity, &bars->abort_flag)) return true;
  *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
  atomicOr(err, kErrTimeout);
  return false;
}

// Tiled 2-D TMA load of one box at (x, y) into this CTA's shared memory.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tile_mn(const Fp4Args& a, int tile, int& mt, int& nt) {
  if (a.m_fastest) {
    mt = tile % a.tiles_m;
    nt = tile / a.tiles_m;
  } else {
    nt = tile % a.tiles_n;
    mt = tile / a.tiles_n;
  }
}

__global__ void __launch_bounds__(THREADS, 1)
k_gemm_nvfp4_fprop(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Fp4Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = a.tiles_m * a.tiles_n;
  const int nkc = a.K / 256;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init_s(smem_addr(&bars->full[s]), 1);
      mbar_init_s(smem_addr(&bars->empty[s]), 1);
      mbar_init_s(smem_addr(&bars->sfready[s]), 4);
    }
    mbar_init_s(smem_addr(&bars->tfull), 1);
    mbar_init_s(smem_addr(&bars->tempty), 8);
    mbar_init_s(smem_addr(&bars->done), 1);
    bars->abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&bars->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_map(&tmA);
      prefetch_map(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        int mt, nt;
        tile_mn(a, tile, mt, nt);
        for (int kc = 0; kc < nkc; ++kc, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_or_abort(smem_addr(&bars->empty[s]), ph ^ 1u, bars, a.err)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_addr(&bars->full[s]);
          const uint32_t st = smem_addr(smem + s * STAGE_BYTES);
          mbar_expect_tx(full, STAGE_BYTES);
          tma_load(st, &tmA, full, kc * KSTAGE_BYTES, mt * BM);
          tma_load(st + A_BYTES, &tmB, full, kc * KSTAGE_BYTES, nt * BN);
          bulk_g2s_plain(st + A_BYTES + B_BYTES, a.xsf + ((size_t)mt * a.kg + 4u * kc) * 512u, SFA_BYTES, full);
#pragma unroll
          for (int t = 0; t < BN / 128; ++t)
            bulk_g2s_plain(st + A_BYTES + B_BYTES + SFA_BYTES + t * 2048,
                           a.wsf + ((size_t)(nt * (BN / 128) + t) * a.kg + 4u * kc) * 512u, 2048, full);
        }
      }
      // every copy issued lands before the CTA's shared memory goes away
      const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_bounded(smem_addr(&bars->full[j % STAGES]), (j / STAGES) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, tj = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++tj) {
        if (!wait_or_abort(smem_addr(&bars->tempty), (tj & 1u) ^ 1u, bars, a.err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int kc = 0; kc < nkc; ++kc, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_or_abort(smem_addr(&bars->sfready[s]), ph, bars, a.err)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a_addr = smem_addr(smem + s * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
          const uint32_t sf0 = tmem + ACC_COLS + s * SF_COLS;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (kc > 0 || k > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(tmem),
                "l"(sdesc_sw128(a_addr + 32 * k)), "l"(sdesc_sw128(b_addr + 32 * k)), "r"(IDESC),
                "r"(sf0 + 4 * k), "r"(sf0 + 16 + 8 * k), "r"(acc));
          }
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           smem_addr(&bars->empty[s]))
                       : "memory");
        }
        if (!ok) break;
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_addr(&bars->tfull))
                     : "memory");
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_addr(&bars->done))
                   : "memory");
      if (!mbar_wait_bounded(smem_addr(&bars->done), 0)) atomicOr(a.err, kErrTimeout);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- block scales: shared memory -> TMEM ----------------
    const uint32_t lq = (uint32_t)(warp & 3);
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      for (int kc = 0; kc < nkc; ++kc, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        bool good = wait_or_abort(smem_addr(&bars->full[s]), ph, bars, a.err);
        if (!__all_sync(kFullMask, good)) {
          ok = false;
          break;
        }
        const uint8_t* sfa = smem + s * STAGE_BYTES + A_BYTES + B_BYTES;
        const uint8_t* sfb = sfa + SFA_BYTES;
        uint32_t va[16], vb[32];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 w = *reinterpret_cast<const uint4*>(sfa + k * 512 + lane * 16);
          va[4 * k] = w.x;
          va[4 * k + 1] = w.y;
          va[4 * k + 2] = w.z;
          va[4 * k + 3] = w.w;
#pragma unroll
          for (int t = 0; t < BN / 128; ++t) {
            const uint4 v = *reinterpret_cast<const uint4*>(sfb + t * 2048 + k * 512 + lane * 16);
            vb[8 * k + 4 * t] = v.x;
            vb[8 * k + 4 * t + 1] = v.y;
            vb[8 * k + 4 * t + 2] = v.z;
            vb[8 * k + 4 * t + 3] = v.w;
          }
        }
        const uint32_t col = tmem + ((lq * 32u) << 16) + ACC_COLS + s * SF_COLS;
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(col),
            "r"(va[0]), "r"(va[1]), "r"(va[2]), "r"(va[3]), "r"(va[4]), "r"(va[5]), "r"(va[6]), "r"(va[7]),
            "r"(va[8]), "r"(va[9]), "r"(va[10]), "r"(va[11]), "r"(va[12]), "r"(va[13]), "r"(va[14]), "r"(va[15])
            : "memory");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
            "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(col + 16),
            "r"(vb[0]), "r"(vb[1]), "r"(vb[2]), "r"(vb[3]), "r"(vb[4]), "r"(vb[5]), "r"(vb[6]), "r"(vb[7]),
            "r"(vb[8]), "r"(vb[9]), "r"(vb[10]), "r"(vb[11]), "r"(vb[12]), "r"(vb[13]), "r"(vb[14]), "r"(vb[15]),
            "r"(vb[16]), "r"(vb[17]), "r"(vb[18]), "r"(vb[19]), "r"(vb[20]), "r"(vb[21]), "r"(vb[22]), "r"(vb[23]),
            "r"(vb[24]), "r"(vb[25]), "r"(vb[26]), "r"(vb[27]), "r"(vb[28]), "r"(vb[29]), "r"(vb[30]), "r"(vb[31])
            : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_s(smem_addr(&bars->sfready[s]));
      }
    }
  } else if (warp >= 8) {
    // ---------------- epilogue ----------------
    // The row's scale and this warp's 128 column scales are fetched before the
    // accumulator is waited for (the column scales into the warp's own row of
    // shared memory, read back as broadcasts); the 128 columns are converted to
    // bf16 in registers and the accumulator is handed back to the tensor core
    // before the stores, so the next tile's MMAs run under them.
    const uint32_t lq = (uint32_t)(warp & 3);
    const int half = (warp - 8) >> 2;            // columns [128·half, 128·half + 128)
    float* gws = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 1024) + (warp - 8) * 128;
    uint32_t tj = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tj) {
      int mt, nt;
      tile_mn(a, tile, mt, nt);
      const int row = mt * BM + (int)lq * 32 + lane;
      const bool row_ok = row < a.M;
      const float gx = row_ok ? __ldg(a.gx + row) : 0.0f;
      const float4 g4 = __ldg(reinterpret_cast<const float4*>(a.gw + (size_t)nt * BN + 128 * half) + lane);
      __syncwarp();   // the previous tile's reads of the row are done
      *reinterpret_cast<float4*>(gws + 4 * lane) = g4;
      __syncwarp();
      const bool good = wait_or_abort(smem_addr(&bars->tfull), tj & 1u, bars, a.err);
      if (!__all_sync(kFullMask, good)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t o[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
            "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(tmem + ((lq * 32u) << 16) + (uint32_t)(128 * half + 32 * c)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 w2 = *reinterpret_cast<const float2*>(gws + 32 * c + 2 * j);
          const float v0 = __fmul_rn(__fmul_rn(__uint_as_float(r[2 * j]), gx), w2.x);
          const float v1 = __fmul_rn(__fmul_rn(__uint_as_float(r[2 * j + 1]), gx), w2.y);
          o[c][j] = f2_to_bf2(v0, v1);
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_s(smem_addr(&bars->tempty));
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(a.y + (size_t)row * a.N + (size_t)nt * BN + 128 * half);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[4 * c + j] = make_uint4(o[c][4 * j], o[c][4 * j + 1], o[c][4 * j + 2], o[c][4 * j + 3]);
      }
    }
  }

  // ---------------- teardown ----------------
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

}  // namespace

size_t nvfp4_scale_bytes(int64_t R, int64_t K) { return (size_t)((R + 127) / 128) * (size_t)(K / 64) * 512u; }

cudaError_t launch_quant_nvfp4(const void* x, int64_t R, int64_t K, uint8_t* q, uint8_t* sf, float* g,
                               cudaStream_t st) {
  const int64_t rows = (R + 127) / 128 * 128;
  const int64_t want = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 8;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  k_quant_nvfp4_rows<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), (uint32_t)R, (uint32_t)K, q, sf,
                                            g);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4(const uint8_t* xq, const uint8_t* xsf, const float* gx, const uint8_t* wq,
                              const uint8_t* wsf, const float* gw, int64_t M, int64_t N, int64_t K, void* y,
                              cudaStream_t st) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(k_gemm_nvfp4_fprop, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  // packed FP4 rows are K/2 bytes; boxes of 128 bytes (256 elements) × 128 or 256 rows
  if (!encode_map_2d(&ta, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)(K / 2), (uint64_t)M, (uint64_t)(K / 2),
                     KSTAGE_BYTES, BM, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !encode_map_2d(&tb, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)(K / 2), (uint64_t)N, (uint64_t)(K / 2),
                     KSTAGE_BYTES, BN, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  Fp4Args a;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.tiles_m = (int)((M + BM - 1) / BM);
  a.tiles_n = (int)(N / BN);
  a.m_fastest = M <= N ? 1 : 0;
  a.kg = (uint32_t)(K / 64);
  a.xsf = xsf;
  a.wsf = wsf;
  a.gx = gx;
  a.gw = gw;
  a.y = static_cast<uint16_t*>(y);
  a.err = err;
  const int tiles = a.tiles_m * a.tiles_n;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  k_gemm_nvfp4_fprop<<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace jetfp8
