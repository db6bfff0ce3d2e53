// Device helpers shared by the jetfp8 kernels (sm_103a).
//
// Quantisation rule (Jet-RL digest "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8
// 强化学习", 前置知识 › FP8 量化 (E4M3 格式)): S = max|x|/448 and x̂ = E4M3(x/S).
// Both quotients are correctly rounded FP32 divisions; the E4M3 cast rounds to
// nearest even and saturates (cvt.rn.satfinite).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/jetfp8.h"

namespace jetfp8 {

constexpr float kE4M3Max = 448.0f;
// Group maxima below this (and above 0) form their element quotients on operands scaled by 2^96.
constexpr float kQuotientMinAmax = 0x1p-80f;

// Error bits recorded in the device error word.
constexpr unsigned kErrTimeout = 1u;

// Host side: device address of this device's error word (set-up once per device).
unsigned* device_error_word();
int num_sms();
bool device_is_sm103();

// -------------------------------------------------------------------------
// E4M3 quantisation of the correctly rounded FP32 quotient
// -------------------------------------------------------------------------
// Packed FP32 pair arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ uint64_t f2_bits(float2 v) {
  return (uint64_t)__float_as_uint(v.x) | ((uint64_t)__float_as_uint(v.y) << 32);
}
__device__ __forceinline__ float2 bits_f2(uint64_t b) {
  return make_float2(__uint_as_float((uint32_t)b), __uint_as_float((uint32_t)(b >> 32)));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

// Bracketing factors 1 ± 2^-20 (exact in FP32).
constexpr float kBracketUp = 1.0f + 0x1p-20f;
constexpr float kBracketDn = 1.0f - 0x1p-20f;

struct GroupScale {
  float s;      // S = fp32(amax/448), or 1 when amax == 0
  float ra;     // ≈ (1/S)·(1 + 2^-20), within 2^-21 relative
  float rb;     // ≈ (1/S)·(1 - 2^-20), within 2^-21 relative
  bool exact;   // 1/S is 1e37 or more (or not finite): always divide
};

// Bracketing factors from S.  rcp.approx is within a few ulp of 1/S; the
// bracket argument in quant_pair only needs ra, rb within 2^-21 relative of
// (1/S)(1 ± 2^-20).  Reciprocals of 1e37 or more (S subnormal or zero) and
// non-finite ones send every value of the group to the division.
__device__ __forceinline__ void set_brackets(GroupScale& g) {
  float rs;
  asm("rcp.approx.f32 %0, %1;" : "=f"(rs) : "f"(g.s));
  g.exact = !(rs < 1.0e37f);
  g.ra = __fmul_rn(rs, kBracketUp);
  g.rb = __fmul_rn(rs, kBracketDn);
}

// S = fp32(amax/448), the correctly rounded quotient, for any finite amax >= 0,
// without a division: Markstein's quotient correction (P. Markstein, IBM J.
// Res. Dev. 34(1), 1990): with c = fp32(1/448) (within half an ulp of 1/448)
// and q0 = RN(amax·c) (within one ulp of the quotient), the residual
// r = amax - 448·q0 is exact (one FMA) and RN(q0 + r·c) (one FMA) is the
// correctly rounded quotient.  tests/test_scale_division_free.py checks the
// sequence in exact arithmetic for every positive finite bf16 value and for
// every FP32 significand of a binade; it holds for every amax whose
// intermediates are normal numbers (amax >= 2^-100), and smaller maxima take
// the IEEE division.  amax == 0 gives S = 1.
__device__ __forceinline__ GroupScale make_scale(float amax) {
  constexpr float kInv448 = 1.0f / 448.0f;   // fp32(1/448)
  GroupScale g;
  if (amax == 0.0f) {
    g.s = 1.0f;
  } else if (amax < 0x1p-100f) {
    g.s = __fdiv_rn(amax, kE4M3Max);
  } else {
    const float q0 = __fmul_rn(amax, kInv448);
    const float r = __fmaf_rn(-q0, kE4M3Max, amax);
    g.s = __fmaf_rn(r, kInv448, q0);
  }
  set_brackets(g);
  return g;
}

// Two E4M3 codes (v0 in the low byte) from two FP32 values.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float v0, float v1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v1), "f"(v0));
  return (uint32_t)r;
}

// E4M3(fp32(v/S)) for two values that share the scale S, without a division
// in the common case.  With ra, rb within 2^-21 relative of 1/S·(1 ± 2^-20),
// a = v·ra and b = v·rb (each rounded once more, 2^-24) sit at least
// 2^-20 - 2^-21 - 2^-23 > 2^-24 relative away from v/S on either side, while
// the correctly rounded quotient RN(v/S) is within 2^-24 of it: a and b
// bracket RN(v/S) strictly.  E4M3 rounding (nearest-even, saturating) is
// monotone, so if a and b round to the same code, RN(v/S) rounds to it too.
// Otherwise — a quotient within about 2^-20 of an E4M3 rounding boundary, or a
// scale whose reciprocal overflows — the IEEE division decides.  Zeros keep
// their sign on both paths.
__device__ __forceinline__ uint32_t quant_pair(float2 v, const GroupScale& g) {
  const float2 a = mul2(v, make_float2(g.ra, g.ra));
  const float2 b = mul2(v, make_float2(g.rb, g.rb));
  uint32_t ca = cvt_e4m3x2(a.x, a.y);
  const uint32_t cb = cvt_e4m3x2(b.x, b.y);
  if (ca != cb || g.exact) ca = cvt_e4m3x2(__fdiv_rn(v.x, g.s), __fdiv_rn(v.y, g.s));
  return ca;
}

// N pairs sharing one scale -> 2N codes packed little-endian into N/2 words
// (pair 2w in the low half of word w).  All brackets are formed first and one
// branch takes the rare division path for the whole set.
template <int N>
__device__ __forceinline__ void quant_pairs(const float2 (&v)[N], const GroupScale& g, uint32_t (&out)[N / 2]) {
  static_assert(N % 2 == 0, "pairs come in twos");
  uint32_t cb[N / 2];
  bool diff = g.exact;
#pragma unroll
  for (int w = 0; w < N / 2; ++w) {
    const float2 a0 = mul2(v[2 * w], make_float2(g.ra, g.ra));
    const float2 a1 = mul2(v[2 * w + 1], make_float2(g.ra, g.ra));
    const float2 b0 = mul2(v[2 * w], make_float2(g.rb, g.rb));
    const float2 b1 = mul2(v[2 * w + 1], make_float2(g.rb, g.rb));
    out[w] = cvt_e4m3x2(a0.x, a0.y) | (cvt_e4m3x2(a1.x, a1.y) << 16);
    cb[w] = cvt_e4m3x2(b0.x, b0.y) | (cvt_e4m3x2(b1.x, b1.y) << 16);
    diff |= out[w] != cb[w];
  }
  if (diff) {
#pragma unroll
    for (int w = 0; w < N / 2; ++w)
      out[w] = quant_pair(v[2 * w], g) | (quant_pair(v[2 * w + 1], g) << 16);
  }
}

// ---------------------------------------------------------------------------
// Element codes without a division and without a fallback branch.  Per group,
// besides S: y = RN(1/S) (IEEE reciprocal).  Per element x, the correctly
// rounded quotient RN(x/S) by two Markstein corrections of q0 = RN(x·y):
//   q1 = RN(q0 + (x - q0·S)·y),  q2 = RN(q1 + (x - q1·S)·y)  (residuals by FMA)
// after which q1 is within one ulp of x/S, so the second residual is exact and
// q2 = RN(x/S) (P. Markstein, IBM J. Res. Dev. 34(1), 1990).  The sequence runs
// on -x and -y so that the sign of a zero survives.  It holds while every
// intermediate is a normal number, i.e. for groups with amax >= 2^-80 (and
// amax = 0); groups with smaller maxima (`slow`) run it on x·2^96 and S·2^96.  The sequence was
// checked in exact arithmetic against RN(x/S) for every bf16 element of
// sampled groups and for FP32 elements next to every kind of E4M3 midpoint.
// ---------------------------------------------------------------------------
struct QScale {
  uint64_t s2;    // (S, S)
  uint64_t ny2;   // (-y, -y), y = RN(1/S)
  float s;
  bool slow;      // 0 < amax < 2^-80: quotients formed on scaled operands (codes4_tiny)
};

__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// The quotient constants of a group from its S (and whether it is slow).
__device__ __forceinline__ QScale qscale_from_s(float s, bool slow) {
  QScale g;
  g.s = s;
  g.slow = slow;
  const float ny = -__frcp_rn(s);
  g.s2 = pack_f2(s, s);
  g.ny2 = pack_f2(ny, ny);
  return g;
}

// Four E4M3 codes (byte k = value k) of the bf16 values whose negations are
// in nw0 (values 0, 1) and nw1 (values 2, 3), under group constants g (not slow).
__device__ __forceinline__ uint32_t codes4_negbf16(uint32_t nw0, uint32_t nw1, const QScale& g) {
  uint32_t c;
  asm("{\n\t.reg .b32 a0, a1, a2, a3;\n\t.reg .b64 x0, x1, q0, q1, r0, r1;\n\t.reg .b16 l, h;\n\t"
      "shl.b32 a0, %1, 16;\n\t"
      "and.b32 a1, %1, 0xFFFF0000;\n\t"
      "shl.b32 a2, %2, 16;\n\t"
      "and.b32 a3, %2, 0xFFFF0000;\n\t"
      "mov.b64 x0, {a0, a1};\n\t"
      "mov.b64 x1, {a2, a3};\n\t"
      "mul.rn.f32x2 q0, x0, %4;\n\t"
      "mul.rn.f32x2 q1, x1, %4;\n\t"
      "fma.rn.f32x2 r0, q0, %3, x0;\n\t"
      "fma.rn.f32x2 r1, q1, %3, x1;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "fma.rn.f32x2 r0, q0, %3, x0;\n\t"
      "fma.rn.f32x2 r1, q1, %3, x1;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "mov.b64 {a0, a1}, q0;\n\t"
      "mov.b64 {a2, a3}, q1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, a3, a2;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(c) : "r"(nw0), "r"(nw1), "l"(g.s2), "l"(g.ny2));
  return c;
}

// The same for the bf16 values themselves in w0 (values 0, 1) and w1 (values 2, 3):
// each negated FP32 value in one integer operation, (w << 16) + 2^31 for the low
// half (adding 2^31 modulo 2^32 flips bit 31) and (w & 0xFFFF0000) ^ 2^31 for the
// high half (lop3, table 0x6A = (a & b) ^ c).
__device__ __forceinline__ uint32_t codes4_bf16(uint32_t w0, uint32_t w1, const QScale& g) {
  uint32_t c;
  asm("{\n\t.reg .b32 a0, a1, a2, a3;\n\t.reg .b64 x0, x1, q0, q1, r0, r1;\n\t.reg .b16 l, h;\n\t"
      "mad.lo.u32 a0, %1, 65536, 0x80000000;\n\t"
      "lop3.b32 a1, %1, 0xFFFF0000, 0x80000000, 0x6A;\n\t"
      "mad.lo.u32 a2, %2, 65536, 0x80000000;\n\t"
      "lop3.b32 a3, %2, 0xFFFF0000, 0x80000000, 0x6A;\n\t"
      "mov.b64 x0, {a0, a1};\n\t"
      "mov.b64 x1, {a2, a3};\n\t"
      "mul.rn.f32x2 q0, x0, %4;\n\t"
      "mul.rn.f32x2 q1, x1, %4;\n\t"
      "fma.rn.f32x2 r0, q0, %3, x0;\n\t"
      "fma.rn.f32x2 r1, q1, %3, x1;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "fma.rn.f32x2 r0, q0, %3, x0;\n\t"
      "fma.rn.f32x2 r1, q1, %3, x1;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "mov.b64 {a0, a1}, q0;\n\t"
      "mov.b64 {a2, a3}, q1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, a3, a2;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(c) : "r"(w0), "r"(w1), "l"(g.s2), "l"(g.ny2));
  return c;
}

// The same for FP32 values given negated as two packed pairs (nx0 = (-v0, -v1),
// nx1 = (-v2, -v3)).
__device__ __forceinline__ uint32_t codes4_neg_f32(uint64_t nx0, uint64_t nx1, const QScale& g) {
  uint32_t c;
  asm("{\n\t.reg .b32 a0, a1, a2, a3;\n\t.reg .b64 q0, q1, r0, r1;\n\t.reg .b16 l, h;\n\t"
      "mul.rn.f32x2 q0, %1, %4;\n\t"
      "mul.rn.f32x2 q1, %2, %4;\n\t"
      "fma.rn.f32x2 r0, q0, %3, %1;\n\t"
      "fma.rn.f32x2 r1, q1, %3, %2;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "fma.rn.f32x2 r0, q0, %3, %1;\n\t"
      "fma.rn.f32x2 r1, q1, %3, %2;\n\t"
      "fma.rn.f32x2 q0, r0, %4, q0;\n\t"
      "fma.rn.f32x2 q1, r1, %4, q1;\n\t"
      "mov.b64 {a0, a1}, q0;\n\t"
      "mov.b64 {a2, a3}, q1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, a3, a2;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(c) : "l"(nx0), "l"(nx1), "l"(g.s2), "l"(g.ny2));
  return c;
}

// Four codes of a group with a tiny maximum (0 < amax < kQuotientMinAmax):
// the elements and S scaled by 2^96 (exact, the quotients unchanged) put every
// intermediate of the sequence above in the normal range.
__device__ __forceinline__ uint32_t codes4_tiny(float2 v0, float2 v1, float s) {
  constexpr float k = 0x1p96f;
  const QScale g = qscale_from_s(s * k, false);
  return codes4_neg_f32(pack_f2(v0.x * -k, v0.y * -k), pack_f2(v1.x * -k, v1.y * -k), g);
}

// Two E4M3 codes (low byte first) -> two exact floats.
__device__ __forceinline__ float2 dec_e4m3x2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_codes));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// bf16x2 word -> two floats (exact)
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // a -> low half
  return *reinterpret_cast<uint32_t*>(&h);
}

// 4×4 byte transpose: rows a,b,c,d (byte i = column i) -> columns.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  uint32_t t0 = __byte_perm(a, b, 0x5140);   // a0 b0 a1 b1
  uint32_t t1 = __byte_perm(a, b, 0x7362);   // a2 b2 a3 b3
  uint32_t t2 = __byte_perm(c, d, 0x5140);   // c0 d0 c1 d1
  uint32_t t3 = __byte_perm(c, d, 0x7362);   // c2 d2 c3 d3
  o0 = __byte_perm(t0, t2, 0x5410);          // a0 b0 c0 d0
  o1 = __byte_perm(t0, t2, 0x7632);          // a1 b1 c1 d1
  o2 = __byte_perm(t1, t3, 0x5410);
  o3 = __byte_perm(t1, t3, 0x7632);
}

// 8×8 byte transpose.  In: row r = (lo[r], hi[r]) (columns 0-3, 4-7).
// Out: column c = (olo[c], ohi[c]) (rows 0-3, 4-7).
__device__ __forceinline__ void transpose8x8(const uint32_t lo[8], const uint32_t hi[8],
                                             uint32_t olo[8], uint32_t ohi[8]) {
  transpose4x4(lo[0], lo[1], lo[2], lo[3], olo[0], olo[1], olo[2], olo[3]);
  transpose4x4(lo[4], lo[5], lo[6], lo[7], ohi[0], ohi[1], ohi[2], ohi[3]);
  transpose4x4(hi[0], hi[1], hi[2], hi[3], olo[4], olo[5], olo[6], olo[7]);
  transpose4x4(hi[4], hi[5], hi[6], hi[7], ohi[4], ohi[5], ohi[6], ohi[7]);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

}  // namespace jetfp8
