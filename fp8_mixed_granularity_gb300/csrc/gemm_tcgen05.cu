// Block-scaled E4M3 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   out[i,j] = Σ_kb sA[kb][i] · sB(kb,j) · Σ_{k in kb} A[i,k]·B[j,k]      (kb = 128-wide block)
//
// This one kernel serves FProp, DGrad and WGrad of the Jet-RL linear layer
// (digest "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习", 核心方法:
// FProp (1×128)×(128×128), DGrad reuses it with the transposed weight, WGrad
// (1×128)×(128×1); 方法步骤详情, steps 2 and 4).  The scales are FP32, not
// power-of-two microscales, so the tensor core cannot apply them: every
// 128-deep block is accumulated on its own in TMEM and promoted in registers,
//   acc[i,j] += partial_kb[i,j] · sA[kb][i] · sB(kb,j).
//
// CTA organisation (persistent, one CTA per SM, 384 threads), for a tile of
// 128 rows × BN columns (BN = 256 with two TMEM accumulators, or BN = 128 with
// four, so the tensor core can run further ahead of the promotion):
//   warp 0      TMA producer: A tile 128 rows × 128 bytes and B tile BN rows ×
//               128 bytes per stage, 128-byte swizzle, multi-stage ring.
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=BN, K=32, E4M3×E4M3→FP32) four times per block into
//               the next TMEM accumulator, then commits.
//   warp 2      uniform scales: stage forwarder (hands each block's operand
//               stage back once its accumulator is complete).
//   warp 3      column scales: scale loader (bulk-copies each block's row and
//               column scales into a ring of shared-memory slots).
//               Warps 0-3 form the control warpgroup, which gives registers
//               back (setmaxnreg.dec) to the promotion warps.
//   warps 4-11  two warpgroups; warpgroup w owns output columns
//               [w·BN/2, (w+1)·BN/2) of the tile, each warp the 32 TMEM lanes
//               (tile rows) it may access.  Per block they load the partial
//               from TMEM, hand the accumulator back as soon as the last piece
//               is in registers, and promote with packed FP32 arithmetic;
//               after the last block the tile is written out as bf16 or fp32.
//     uniform scales (FProp, DGrad: sB is one value per 128 output columns):
//               each thread owns one row and 32-column chunks of it;
//               promotion is one FMA per element with the product sA·sB,
//               with the TMEM loads of the next two chunks in flight; the
//               scales are prefetched two blocks ahead into registers.
//     column scales (WGrad: sB is one value per output column): the partial
//               is read as 16-lane × 256-bit fragments, so a thread holds 4
//               rows × 2 adjacent columns of every 8 and needs only a quarter
//               of the column scales, which it reads (with its 4 row scales)
//               from the block's slot of the scale ring.  Promotion is
//               (partial·sB)·sA, a multiply and an FMA per element, with the
//               TMEM loads of the next two fragments in flight.
// A launch may carry up to four problems of one configuration (the WGrads of a
// layer's linears, which share the token count): their tiles form one
// persistent sequence, each tile computed exactly as in a launch of its own.
// The same kernel body also runs on CTA pairs (tcgen05 cta_group::2, a
// cluster of two CTAs on two SMs per 256 × 256 tile): each CTA loads its 128
// rows of A and half of B, the leader issues M = 256 MMAs, and both CTAs
// promote their own 128 rows exactly as above, so the two kernels' results
// are identical bit for bit.  The pair kernel is for tests and diagnosis; the
// single-CTA kernel is faster on GB300 and is the default.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records an
// error word, lets copies and MMAs in flight land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstring>
#include <type_traits>

#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"
#include "jetfp8_tma.cuh"

namespace jetfp8 {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                             // warps 0-3: control warpgroup
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // 384
// Register split.  The kernel is launched with LAUNCH_REGS per thread
// (384 × 168 = 64512); the control warpgroup gives registers back and the two
// promotion warpgroups take them: 128·CTRL_REGS + 256·EPI_REGS must not exceed
// the launch total, or setmaxnreg.inc would wait forever.  The host refuses to
// launch unless the compiled kernel uses exactly LAUNCH_REGS.
constexpr int LAUNCH_REGS = 168;
// Every launch splits 24 / 240: grouped launches (whose control warps also
// track which problem a tile belongs to) spill a few bytes in the control warps
// that way, but the column-scale promotion runs 4.6 % faster than with 32 / 232.
constexpr int CTRL_REGS = 24;
constexpr int EPI_REGS = 240;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= THREADS * LAUNCH_REGS, "register split");
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int MAX_STAGES = 8, MAX_BUFS = 4;
// column-mode scale ring depth, in 128-deep blocks (see the scale loader)
constexpr int SRING = 8;
// bf16 output leaves through shared memory in 32-row × 32-column chunks, one
// 2 KB staging buffer per promotion warp, written to global memory by TMA.
// The buffer uses the 64-byte swizzle: the 16-byte granule g of row r sits at
// r·64 + 16·(g ^ ((r/2) mod 4)), so rows written by neighbouring lanes fall on
// different banks.
constexpr int OUT_CHUNK_BYTES = 32 * 32 * 2;

// Tile configuration.  PAIR: a CTA pair computes a 256 × BN tile (BN = 256);
// each CTA holds its 128 rows of A and half (BN/2 rows) of the B tile.
template <int BN_, bool PAIR = false>
struct Cfg {
  static constexpr int BN = BN_;
  static_assert(!PAIR || BN_ == 256, "CTA pairs use 256-wide tiles");
  // deeper rings for smaller stages (same shared-memory budget)
  static constexpr int STAGES = PAIR ? 6 : (BN_ == 256 ? 4 : (BN_ == 128 ? 6 : 8));
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_BUFS = TMEM_COLS / BN < MAX_BUFS ? TMEM_COLS / BN : MAX_BUFS;
  static constexpr int TMEM_ALLOC = ACC_BUFS * BN;   // a power of two >= 32
  static constexpr int EPI_COLS = BN / 2;        // columns per promotion warp
  static constexpr int CHUNKS = EPI_COLS / 32;   // 32-column TMEM loads per block
  // UMMA instruction descriptor: D = F32 (bits 4-5 = 1), A = B = E4M3 (format 0),
  // both K-major, N/8 at bits 17-22, M/16 at bits 24-28 (M = 256 for a pair).
  static constexpr uint32_t IDESC =
      (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((PAIR ? 2 * BM : BM) >> 4) << 24);
  // Column mode: the scales of each 128-deep block — the tile's BN column
  // scales, then this CTA's 128 row scales — arrive by bulk copy in a ring of
  // SRING slots.  Uniform mode uses the same area to stage the fused output
  // quantiser's codes (1 KB per promotion warp).
  static constexpr int SSLOT_F = BN + BM;
  static constexpr int AUX_BYTES =
      SRING * SSLOT_F * 4 > EPI_WARPS * 1024 ? SRING * SSLOT_F * 4 : EPI_WARPS * 1024;
  static constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES +
                                    1024 /*barriers*/ + AUX_BYTES + EPI_WARPS * OUT_CHUNK_BYTES;
  static_assert(STAGES <= MAX_STAGES && ACC_BUFS <= MAX_BUFS, "barrier arrays");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert((SSLOT_F * 4) % 16 == 0, "bulk-copy destinations 16-byte aligned");
  static_assert(AUX_BYTES % 128 == 0 && OUT_CHUNK_BYTES % 128 == 0,
                "output staging buffers (TMA store sources) 128-byte aligned");
};

struct Barriers {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[MAX_BUFS];
  uint64_t tempty[MAX_BUFS];
  uint64_t sfull[SRING];    // column mode: a block's scales have landed in their slot
  uint64_t sempty[SRING];   // column mode: every promotion warp has read the slot
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

struct DevArgs {
  const float* sA;
  long long ld_sA;
  const float* sB;
  long long sb_j, sb_k;
  void* out;       // may be null when out_q is set
  int R, C, nKB, tiles_m, tiles_n;
  int m_fastest;   // tile order: 1 = consecutive tiles walk down M (share a B tile)
  int out_fp32;
  // fused 1×128 quantisation of the bf16 output (uniform mode, 256-wide tiles):
  // codes [R, C] (stored through tmQ), scales [C/128][ld_out_s]
  uint8_t* out_q;
  float* out_s;
  long long ld_out_s;
  unsigned* err;
  int drop_kb;     // test hook: the producer never loads this block (-1: none)
};

// Kernel parameters: G problems of one tile configuration run as a single
// persistent tile sequence; problem g owns the tiles [tile_end[g-1], tile_end[g]).
// A plain GEMM is G = 1.  Grouping lets the last wave of one problem's tiles be
// filled with another's (the WGrads of a layer's linears share the token
// count, so their tiles cost the same).  tmQ serves the fused output
// quantiser, which only single-problem launches use.
constexpr int MAX_GROUP = 4;
template <int G>
struct KParams {
  CUtensorMap tmA[G], tmB[G], tmOut[G];
  CUtensorMap tmQ;
  DevArgs p[G];
  int tile_end[G];
  int nkb;   // 128-deep blocks per tile, the same for every problem of a launch
};

// Global tile index -> (problem, tile index within that problem).
template <int G>
__device__ __forceinline__ int problem_of(const KParams<G>& kp, int tile, int& local) {
  int g = 0, start = 0;
#pragma unroll
  for (int i = 0; i + 1 < G; ++i)
    if (tile >= kp.tile_end[i]) {
      g = i + 1;
      start = kp.tile_end[i];
    }
  local = tile - start;
  return g;
}

// Field f of problem g as a chain of selects over constant-index parameter
// reads: the control warps, on 24 registers, then make no indexed parameter
// loads and keep no table (a grouped launch spilled and ran 10 % slower per
// tile with indexed loads).
template <int G, typename T>
__device__ __forceinline__ T pick(const KParams<G>& kp, int g, T DevArgs::*f) {
  T v = kp.p[0].*f;
#pragma unroll
  for (int i = 1; i < G; ++i)
    if (g == i) v = kp.p[i].*f;
  return v;
}

// Tile index -> (m tile, n tile).  Consecutive tiles (which run at the same
// time on neighbouring SMs) share one operand tile; the other operand is
// streamed once per band, so the order keeps the re-streamed operand the
// smaller of the two.
__device__ __forceinline__ void tile_coords(const DevArgs& p, int tile, int& mt, int& nt) {
  if (p.m_fastest) {
    mt = tile % p.tiles_m;
    nt = tile / p.tiles_m;
  } else {
    nt = tile % p.tiles_n;
    mt = tile / p.tiles_n;
  }
}
// The same for problem g of a launch, through pick().
template <int G>
__device__ __forceinline__ void tile_coords_of(const KParams<G>& kp, int g, int tile, int& mt, int& nt) {
  if (pick(kp, g, &DevArgs::m_fastest)) {
    const int tm = pick(kp, g, &DevArgs::tiles_m);
    mt = tile % tm;
    nt = tile / tm;
  } else {
    const int tn = pick(kp, g, &DevArgs::tiles_n);
    nt = tile % tn;
    mt = tile / tn;
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Polls two barriers at once (both lookups in flight together).
__device__ __forceinline__ void mbar_try_wait2(uint32_t a, uint32_t pa, uint32_t b, uint32_t pb, bool& oka,
                                               bool& okb) {
  uint32_t ra, rb;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%2], %3;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%4], %5;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "selp.u32 %1, 1, 0, q;\n\t}"
      : "=r"(ra), "=r"(rb) : "r"(a), "r"(pa), "r"(b), "r"(pb) : "memory");
  oka = ra != 0;
  okb = rb != 0;
}

// Wait for the phase of parity `parity` to complete.  Gives up (false) after
// WAIT_NS, or early when another role has already aborted and `honour_abort`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          bool honour_abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if (globaltimer_ns() - t0 > WAIT_NS) return false;
  }
}

// The same wait on 32-bit shared-memory addresses (barrier and abort flag),
// for the TMA producer, which runs on few registers.
__device__ __forceinline__ bool mbar_wait_s(uint32_t bar, uint32_t parity, uint32_t abort_addr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    int flag;
    asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(flag) : "r"(abort_addr) : "memory");
    if (flag) return false;
    if (globaltimer_ns() - t0 > WAIT_NS) return false;
  }
}

__device__ __forceinline__ void record_abort(volatile int* abort_flag, unsigned* err) {
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Bulk tensor store of a shared-memory box to global memory (async proxy).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
      "r"(src), "r"(x), "r"(y)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until the previous bulk stores of this thread have finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major tile stored as 128-byte rows
// with the 128-byte swizzle (8-row atoms of 1024 B): start address >> 4,
// leading offset 16 B (unused for this layout), stride offset 1024 B, the
// descriptor version bit 46, swizzle mode 2 (128 B) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// Starts loading 32 TMEM columns into r[0..31]; the values are valid only
// after tmem_wait_ld(r).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Waits for this thread's TMEM loads.  The destination registers of the load
// are tied to the wait so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Orders later uses of r after the tcgen05.wait::ld just issued (which waits
// for all of this thread's TMEM loads): ties further destination registers.
__device__ __forceinline__ void tmem_tie32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// acc[j] += (p[2j], p[2j+1]) · s2 for 16 packed FP32 pairs (one scale pair).
// Volatile so that it stays between the TMEM load of the next chunk and the
// wait for it.
__device__ __forceinline__ void fma32_uniform(uint64_t (&acc)[16], const uint32_t (&p)[32], uint64_t s2) {
  asm volatile("{\n\t.reg .b64 q;\n\t"
      "mov.b64 q, {%16, %17};\n\t"
      "fma.rn.f32x2 %0, q, %48, %0;\n\t"
      "mov.b64 q, {%18, %19};\n\t"
      "fma.rn.f32x2 %1, q, %48, %1;\n\t"
      "mov.b64 q, {%20, %21};\n\t"
      "fma.rn.f32x2 %2, q, %48, %2;\n\t"
      "mov.b64 q, {%22, %23};\n\t"
      "fma.rn.f32x2 %3, q, %48, %3;\n\t"
      "mov.b64 q, {%24, %25};\n\t"
      "fma.rn.f32x2 %4, q, %48, %4;\n\t"
      "mov.b64 q, {%26, %27};\n\t"
      "fma.rn.f32x2 %5, q, %48, %5;\n\t"
      "mov.b64 q, {%28, %29};\n\t"
      "fma.rn.f32x2 %6, q, %48, %6;\n\t"
      "mov.b64 q, {%30, %31};\n\t"
      "fma.rn.f32x2 %7, q, %48, %7;\n\t"
      "mov.b64 q, {%32, %33};\n\t"
      "fma.rn.f32x2 %8, q, %48, %8;\n\t"
      "mov.b64 q, {%34, %35};\n\t"
      "fma.rn.f32x2 %9, q, %48, %9;\n\t"
      "mov.b64 q, {%36, %37};\n\t"
      "fma.rn.f32x2 %10, q, %48, %10;\n\t"
      "mov.b64 q, {%38, %39};\n\t"
      "fma.rn.f32x2 %11, q, %48, %11;\n\t"
      "mov.b64 q, {%40, %41};\n\t"
      "fma.rn.f32x2 %12, q, %48, %12;\n\t"
      "mov.b64 q, {%42, %43};\n\t"
      "fma.rn.f32x2 %13, q, %48, %13;\n\t"
      "mov.b64 q, {%44, %45};\n\t"
      "fma.rn.f32x2 %14, q, %48, %14;\n\t"
      "mov.b64 q, {%46, %47};\n\t"
      "fma.rn.f32x2 %15, q, %48, %15;\n\t"
      "}"
      : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7]),
        "+l"(acc[8]), "+l"(acc[9]), "+l"(acc[10]), "+l"(acc[11]), "+l"(acc[12]), "+l"(acc[13]), "+l"(acc[14]), "+l"(acc[15])
      : "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]),
        "r"(p[6]), "r"(p[7]), "r"(p[8]), "r"(p[9]), "r"(p[10]), "r"(p[11]),
        "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15]), "r"(p[16]), "r"(p[17]),
        "r"(p[18]), "r"(p[19]), "r"(p[20]), "r"(p[21]), "r"(p[22]), "r"(p[23]),
        "r"(p[24]), "r"(p[25]), "r"(p[26]), "r"(p[27]), "r"(p[28]), "r"(p[29]),
        "r"(p[30]), "r"(p[31]), "l"(s2));
}

// 16-lane × 256-bit TMEM fragments, four of them side by side (16 rows × 32
// columns): for j < 4, r[4j], r[4j+1] are row lane/4 and r[4j+2], r[4j+3]
// row lane/4 + 8 (of the 16 lanes addressed), both at columns
// 8j + 2·(lane mod 4) + {0, 1}.  Valid after tmem_wait_ld16(r).
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_tie16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Column-scale promotion of one fragment (layout of tmem_ld16x256_x4):
//   acc[2j]   += ({p[4j],   p[4j+1]} · sb[j]) · sa_lo      (row lane/4)
//   acc[2j+1] += ({p[4j+2], p[4j+3]} · sb[j]) · sa_hi      (row lane/4 + 8)
// sb[j] holds the scales of the fragment's two columns, sa_lo / sa_hi the
// row scale twice.  All eight products are formed before the eight FMAs, so
// no FMA waits on the multiply just before it.  Volatile so that it stays
// between the TMEM load of the next fragment and the wait for it.
__device__ __forceinline__ void promote_cols_frag(uint64_t* acc, const uint32_t (&p)[16],
                                                  const uint64_t (&sb)[4], uint64_t sa_lo, uint64_t sa_hi) {
  asm volatile(
      "{\n\t.reg .b64 q0, q1, q2, q3, q4, q5, q6, q7;\n\t"
      "mov.b64 q0, {%8, %9};\n\t"
      "mov.b64 q1, {%10, %11};\n\t"
      "mov.b64 q2, {%12, %13};\n\t"
      "mov.b64 q3, {%14, %15};\n\t"
      "mov.b64 q4, {%16, %17};\n\t"
      "mov.b64 q5, {%18, %19};\n\t"
      "mov.b64 q6, {%20, %21};\n\t"
      "mov.b64 q7, {%22, %23};\n\t"
      "mul.rn.f32x2 q0, q0, %24;\n\t"
      "mul.rn.f32x2 q1, q1, %24;\n\t"
      "mul.rn.f32x2 q2, q2, %25;\n\t"
      "mul.rn.f32x2 q3, q3, %25;\n\t"
      "mul.rn.f32x2 q4, q4, %26;\n\t"
      "mul.rn.f32x2 q5, q5, %26;\n\t"
      "mul.rn.f32x2 q6, q6, %27;\n\t"
      "mul.rn.f32x2 q7, q7, %27;\n\t"
      "fma.rn.f32x2 %0, q0, %28, %0;\n\t"
      "fma.rn.f32x2 %1, q1, %29, %1;\n\t"
      "fma.rn.f32x2 %2, q2, %28, %2;\n\t"
      "fma.rn.f32x2 %3, q3, %29, %3;\n\t"
      "fma.rn.f32x2 %4, q4, %28, %4;\n\t"
      "fma.rn.f32x2 %5, q5, %29, %5;\n\t"
      "fma.rn.f32x2 %6, q6, %28, %6;\n\t"
      "fma.rn.f32x2 %7, q7, %29, %7;\n\t"
      "}"
      : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]),
        "+l"(acc[7])
      : "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), "r"(p[8]),
        "r"(p[9]), "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15]), "l"(sb[0]),
        "l"(sb[1]), "l"(sb[2]), "l"(sb[3]), "l"(sa_lo), "l"(sa_hi));
}

// ---- CTA pairs (tcgen05 cta_group::2) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Relaxed arrives hand an accumulator back: the TMEM loads they follow have
// completed (tcgen05.wait::ld) and nothing else needs ordering, so the arrive
// does not wait for the thread's other memory operations in flight.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// Issued by the leader CTA of a pair: M = 256 rows, 128 from each CTA's
// shared memory (same offsets), B halves from both; each CTA's TMEM receives
// its own 128 rows.
__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrives once on the barrier at this shared-memory offset in both CTAs when
// the MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}


template <int BN_, bool COLS, int G, bool PAIR>
__device__ __forceinline__ void gemm_body(const KParams<G>& kp) {
  using C = Cfg<BN_, PAIR>;
  constexpr int BN = C::BN, STAGES = C::STAGES, ACC_BUFS = C::ACC_BUFS;
  constexpr int EPI_COLS = C::EPI_COLS, CHUNKS = C::CHUNKS;
  static_assert(!COLS || BN >= 128, "column-scale promotion needs 128- or 256-wide tiles");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + STAGES * C::STAGE_BYTES);
  // column mode: [SRING][SSLOT_F] scale ring; uniform mode: [8 promotion warps][1 KB] code staging
  uint8_t* aux = smem + STAGES * C::STAGE_BYTES + 1024;
  // [8 promotion warps][32 rows][32 bf16] output staging
  uint8_t* outbuf = aux + C::AUX_BYTES;
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = kp.tile_end[G - 1];
  // A CTA pair is a cluster of two sharing one 256-row tile (rank 0, the
  // leader, issues the MMAs); a single CTA is a "cluster" of one.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int cl = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  constexpr int TILE_M = PAIR ? 2 * BM : BM;
  // records the error and stops every role of this CTA (and of the peer)
  auto fail = [&]() {
    record_abort(abort_flag, kp.p[0].err);
    if constexpr (PAIR) st_cluster_u32(mapa_shared(smem_u32((const void*)&bars->abort_flag), rank ^ 1u), 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(&bars->tfull[b], 1);
      // a pair's accumulators are handed back to the leader by both CTAs; with
      // uniform scales a single CTA's also by the stage forwarder
      mbar_init(&bars->tempty[b], PAIR ? 2 * EPI_WARPS : (COLS ? EPI_WARPS : EPI_WARPS + 1));
    }
    for (int s = 0; s < SRING; ++s) {
      mbar_init(&bars->sfull[s], 1);
      mbar_init(&bars->sempty[s], EPI_WARPS);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      // one warp of each CTA of the pair allocates, collectively, the same columns in both
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(&bars->tmem_base)),
                   "r"(C::TMEM_ALLOC));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(&bars->tmem_base)),
                   "r"(C::TMEM_ALLOC));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  tc_fence_before();
  // (a pair: both CTAs' barriers are initialised before either signals the other's)
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
    if (warp == 0 && PAIR) {
      // ---------------- TMA producer (both CTAs of a pair) ----------------
      // Each CTA loads its 128 rows of A and its half of B; every copy counts
      // on the leader's full barrier, which expects both CTAs' bytes.
      // (32-bit shared-memory addresses, as in the single-CTA producer)
      if (lane == 0) {
        const uint32_t full0 = smem_u32(&bars->full[0]);
        const uint32_t full_leader0 = mapa_shared(full0, 0);
        constexpr uint32_t STAGE0_OFF = STAGES * C::STAGE_BYTES + offsetof(Barriers, full);
        constexpr uint32_t EMPTY_OFF = offsetof(Barriers, empty) - offsetof(Barriers, full);
        constexpr uint32_t ABORT_OFF = offsetof(Barriers, abort_flag) - offsetof(Barriers, full);
        const int row_off = (int)rank * BM, col_off = (int)rank * (BN / 2);
        uint32_t it = 0;
        bool ok = true;
        for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
          int local, mt, nt;
          const int g = problem_of(kp, tile, local);
          tile_coords_of(kp, g, local, mt, nt);
          const int nkb = kp.nkb;
          const CUtensorMap* const mA = &kp.tmA[g];   // tmB[g] lies G maps after it
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            const uint32_t full = full0 + 8 * s;
            if (!mbar_wait_s(full + EMPTY_OFF, ph ^ 1u, full0 + ABORT_OFF)) {
              fail();
              ok = false;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(full, 2 * C::STAGE_BYTES);
            const uint32_t st = full0 - STAGE0_OFF + s * C::STAGE_BYTES;
            tma_load_2d_pair(st, mA, full_leader0 + 8 * s, kb * BK, mt * TILE_M + row_off);
            tma_load_2d_pair(st + C::A_BYTES, mA + G, full_leader0 + 8 * s, kb * BK, nt * BN + col_off);
          }
        }
        // the leader sees every copy of both CTAs land before the pair exits
        if (rank == 0) {
          const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
          for (uint32_t j = first; j < it; ++j)
            mbar_wait(&bars->full[j % STAGES], (j / STAGES) & 1u, abort_flag, false);
        }
      }
    } else if (warp == 0) {
      // ---------------- TMA producer ----------------
      // (32-bit shared-memory addresses throughout: this warp has few registers)
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(&kp.tmA[g]) : "memory");
          asm volatile("prefetch.tensormap [%0];" ::"l"(&kp.tmB[g]) : "memory");
        }
        // the stages sit right below the barriers
        const uint32_t full0 = smem_u32(&bars->full[0]);
        constexpr uint32_t STAGE0_OFF = STAGES * C::STAGE_BYTES + offsetof(Barriers, full);
        constexpr uint32_t EMPTY_OFF = offsetof(Barriers, empty) - offsetof(Barriers, full);
        constexpr uint32_t ABORT_OFF = offsetof(Barriers, abort_flag) - offsetof(Barriers, full);
        uint32_t it = 0;
        bool ok = true;
        static_assert(offsetof(KParams<G>, tmB) == offsetof(KParams<G>, tmA) + G * sizeof(CUtensorMap),
                      "map arrays are contiguous");
        for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
          int local, mt, nt;
          const int g = problem_of(kp, tile, local);
          tile_coords_of(kp, g, local, mt, nt);
          const int nkb = kp.nkb, drop_kb = pick(kp, g, &DevArgs::drop_kb);
          // tmB[g] lies G maps after tmA[g]: one live pointer
          const CUtensorMap* const mA = &kp.tmA[g];
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            // test hook: leave this stage unfilled, so the MMA's bounded wait runs out
            if (kb == drop_kb) continue;
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            const uint32_t full = full0 + 8 * s;
            if (!mbar_wait_s(full + EMPTY_OFF, ph ^ 1u, full0 + ABORT_OFF)) {
              fail();
              ok = false;
              break;
            }
            const uint32_t st = full0 - STAGE0_OFF + s * C::STAGE_BYTES;
            mbar_arrive_expect_tx(full, C::STAGE_BYTES);
            tma_load_2d(st, mA, full, kb * BK, mt * BM);
            tma_load_2d(st + C::A_BYTES, mA + G, full, kb * BK, nt * BN);
          }
        }
        // every copy issued has landed before the CTA's shared memory goes away
        // (after an abort the tensor core may not have consumed the last ones;
        // otherwise these phases are complete and each poll returns at once)
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait(&bars->full[j % STAGES], (j / STAGES) & 1u, abort_flag, false);
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer (a pair's leader) ----------------
      if (lane == 0 && rank == 0) {
        uint32_t it = 0, acc_it = 0;
        bool ok = true;
        // (every tile has kp.nkb blocks: no per-problem lookup on this warp,
        // whose few registers and issue latency the tensor core waits on)
        const int nkb = kp.nkb;
        for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
          for (int kb = 0; kb < nkb; ++kb, ++it, ++acc_it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            const uint32_t b = acc_it % ACC_BUFS, bph = (acc_it / ACC_BUFS) & 1u;
            // a free accumulator and a full operand stage; with uniform scales
            // both are polled at once (each waited for alone only if needed):
            // decode FProp +3 %, FProp and DGrad +0.5 - 1 %, while the
            // promotion-bound WGrad measured 2 % slower that way
            bool e_ok = false, f_ok = false;
            if constexpr (!COLS)
              mbar_try_wait2(smem_u32(&bars->tempty[b]), bph ^ 1u, smem_u32(&bars->full[s]), ph, e_ok, f_ok);
            if (!((e_ok || mbar_wait(&bars->tempty[b], bph ^ 1u, abort_flag, true)) &&
                  (f_ok || mbar_wait(&bars->full[s], ph, abort_flag, true)))) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
            const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              if constexpr (PAIR)
                umma_e4m3_pair(tmem + b * BN, sdesc_sw128(a_addr + 32 * k), sdesc_sw128(b_addr + 32 * k),
                               C::IDESC, k > 0 ? 1u : 0u);
              else
                umma_e4m3(tmem + b * BN, sdesc_sw128(a_addr + 32 * k), sdesc_sw128(b_addr + 32 * k),
                          C::IDESC, k > 0 ? 1u : 0u);
            }
            // (a pair: the commits arrive on these barriers in both CTAs)
            if constexpr (PAIR) {
              umma_commit_pair(&bars->empty[s]);
              umma_commit_pair(&bars->tfull[b]);
            } else if constexpr (!COLS) {
              // uniform scales: one commit per block, the stage goes back to the
              // producer through the stage forwarder (warp 2) once the block's
              // accumulator is complete (an extra commit per block measured 2.5 %
              // on FProp and DGrad; with the forwarder they run 3-4 % faster)
              umma_commit(&bars->tfull[b]);
            } else {
              // column scales (promotion-bound): the stage as soon as the MMAs are
              // done (the forwarder's later release cost WGrad 2 %)
              umma_commit(&bars->empty[s]);
              umma_commit(&bars->tfull[b]);
            }
          }
        }
        // all MMAs issued by this thread complete before TMEM is released
        if constexpr (PAIR) umma_commit_pair(&bars->done);
        else umma_commit(&bars->done);
      }
      if (lane == 0 && !mbar_wait(&bars->done, 0, abort_flag, false) && !*abort_flag) fail();
    } else if (warp == 2 && !PAIR && !COLS) {
      // ---------------- stage forwarder (single CTA, uniform scales) ----------------
      // For every block in order: once its accumulator is complete, its MMAs no
      // longer read its operand stage, which goes back to the producer.  The
      // forwarder also arrives on the accumulator's empty barrier, so the next
      // completion of the same full barrier cannot happen before it has seen
      // this one (no phase passes unseen).
      if (lane == 0) {
        uint32_t it = 0;
        bool ok = true;
        const int nkb = kp.nkb;
        for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const uint32_t b = it % ACC_BUFS, bph = (it / ACC_BUFS) & 1u;
            if (!mbar_wait(&bars->tfull[b], bph, abort_flag, true)) {
              fail();
              ok = false;
              break;
            }
            mbar_arrive(&bars->empty[it % STAGES]);
            mbar_arrive(&bars->tempty[b]);
          }
        }
      }
    } else if (warp == 3 && COLS) {
      // ---------------- scale loader (column mode) ----------------
      // Block by block, in the order the promotion warps take them: once every
      // promotion warp has read slot it mod SRING, the block's BN column scales
      // and this CTA's 128 row scales go there by two bulk copies.  (The host
      // launches column mode only for whole 128-row tiles, BN-wide column
      // tiles and 16-byte aligned scale rows; a pair's second CTA past the
      // last row tile loads no row scales — its rows are never stored.)
      if (lane == 0) {
        const uint32_t sfull0 = smem_u32(&bars->sfull[0]);
        constexpr uint32_t SEMPTY_OFF = offsetof(Barriers, sempty) - offsetof(Barriers, sfull);
        constexpr uint32_t ABORT_OFF = offsetof(Barriers, abort_flag) - offsetof(Barriers, sfull);
        const uint32_t ring0 = smem_u32(aux);
        uint32_t it = 0;
        bool ok = true;
        for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
          int local, mt, nt;
          const int g = problem_of(kp, tile, local);
          tile_coords_of(kp, g, local, mt, nt);
          const int row0 = mt * TILE_M + (int)rank * BM;
          const uint32_t rbytes = row0 < pick(kp, g, &DevArgs::R) ? BM * 4u : 0u;
          const float* sa = pick(kp, g, &DevArgs::sA) + row0;
          const float* sb = pick(kp, g, &DevArgs::sB) + (long long)nt * BN;
          // (strides in elements, 32 bits)
          const uint32_t sa_step = (uint32_t)pick(kp, g, &DevArgs::ld_sA);
          const uint32_t sb_step = (uint32_t)pick(kp, g, &DevArgs::sb_k);
          const int nkb = kp.nkb;
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const uint32_t slot = it % SRING, bar = sfull0 + 8 * slot;
            if (!mbar_wait_s(bar + SEMPTY_OFF, ((it / SRING) & 1u) ^ 1u, sfull0 + ABORT_OFF)) {
              fail();
              ok = false;
              break;
            }
            const uint32_t dst = ring0 + slot * (C::SSLOT_F * 4);
            mbar_arrive_expect_tx(bar, BN * 4u + rbytes);
            bulk_g2s_plain(dst, sb + (size_t)kb * sb_step, BN * 4u, bar);
            if (rbytes != 0) bulk_g2s_plain(dst + BN * 4u, sa + (size_t)kb * sa_step, rbytes, bar);
          }
        }
        // every copy issued has landed before shared memory goes away
        const uint32_t first = it > (uint32_t)SRING ? it - SRING : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait(&bars->sfull[j % SRING], (j / SRING) & 1u, abort_flag, false);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
    // ---------------- promotion + epilogue ----------------
    const int ew = warp - EPI_WARP0;
    const int wg = ew >> 2;                 // column half of the tile
    const int lq = warp & 3;                // TMEM lane quarter this warp may access
    const uint32_t taddr_w = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(wg * EPI_COLS);
    const float* sring = reinterpret_cast<const float*>(aux);
    uint32_t acc_it = 0;
    bool ok = true;
    for (int tile = cl; tile < num_tiles && ok; tile += ncl) {
      const int nkb = kp.nkb;
      // the tile's problem and coordinates (a grouped launch derives them again
      // after the block loop, so that none of them stays live across it: with
      // its problem index known only at run time that spilled)
      int local, mt, nt;
      int g = problem_of(kp, tile, local);
      tile_coords(kp.p[g], local, mt, nt);
      int wrow0 = mt * TILE_M + (int)rank * BM + lq * 32;   // first tile row of this warp
      int row = wrow0 + lane;                                 // the row whose sA this lane fetches
      int col0 = nt * BN + wg * EPI_COLS;
      bool row_ok = row < kp.p[g].R;
      // Uniform mode: the scales are prefetched two blocks ahead into a
      // two-slot register ring; the block loop is unrolled by two so every slot
      // index is a compile-time constant and no register copy waits on a load
      // in flight.  Column mode reads them from the scale ring.
      const float* sa_ptr = kp.p[g].sA + row;
      const float* sb_ptr = kp.p[g].sB + (long long)(col0 / 128) * kp.p[g].sb_j;
      auto load_sa = [&](int kb) {
        return (!COLS && row_ok && kb < nkb) ? __ldg(sa_ptr + (long long)kb * kp.p[g].ld_sA) : 0.0f;
      };
      auto load_sb = [&](int kb) {
        return (!COLS && kb < nkb) ? __ldg(sb_ptr + (long long)kb * kp.p[g].sb_k) : 0.0f;
      };
      float sa_r[2], sb_r[2];
      if (!COLS) {
        sa_r[0] = load_sa(0);
        sa_r[1] = load_sa(1);
        sb_r[0] = load_sb(0);
        sb_r[1] = load_sb(1);
      }
      // uniform mode: acc[c][j] holds row `row`, columns 32c + 2j + {0,1};
      // column mode: acc[cq][8h + 2j + rs] holds row wrow0 + lane/4 + 8rs + 16h,
      // columns 32cq + 8j + 2(lane mod 4) + {0,1}
      uint64_t acc[CHUNKS][16];
#pragma unroll
      for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c][j] = 0ull;

      // one 128-deep block; SL is the ring slot of this block's scales
      auto block = [&](int kb, auto slot) -> bool {
        constexpr int SL = decltype(slot)::value;
        const uint32_t b = acc_it % ACC_BUFS, bph = (acc_it / ACC_BUFS) & 1u;
        const uint32_t ss = acc_it % SRING;
        ++acc_it;
        uint64_t s2u = 0;
        if (!COLS) {
          const float sc = sa_r[SL] * sb_r[SL];
          s2u = pack2(sc, sc);
          sa_r[SL] = load_sa(kb + 2);
          sb_r[SL] = load_sb(kb + 2);
        }
        // column mode: the block's scales must be in their ring slot as well
        // (both barriers polled together; each is waited for alone only if needed)
        bool good;
        if constexpr (COLS) {
          bool s_ok, t_ok;
          const uint32_t sph = ((acc_it - 1) / SRING) & 1u;
          mbar_try_wait2(smem_u32(&bars->sfull[ss]), sph, smem_u32(&bars->tfull[b]), bph, s_ok, t_ok);
          good = (s_ok || mbar_wait(&bars->sfull[ss], sph, abort_flag, true)) &&
                 (t_ok || mbar_wait(&bars->tfull[b], bph, abort_flag, true));
        } else {
          good = mbar_wait(&bars->tfull[b], bph, abort_flag, true);
        }
        if (!good) fail();
        if (__any_sync(0xffffffffu, !good)) return false;
        tc_fence_after();
        const uint32_t tbase = taddr_w + b * BN;
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // (a pair: on the leader's barrier, addressed through the cluster)
            if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->tempty[b]), 0));
            else mbar_arrive_relaxed(&bars->tempty[b]);
            // column mode: the warp's reads of the scale slot are done (this
            // arrive orders them before the slot is refilled)
            if constexpr (COLS) mbar_arrive(&bars->sempty[ss]);
          }
        };
        if (COLS) {
          // fragments i = 2·cq + h: columns 32cq.., lanes 16h..
          constexpr int NF = 2 * CHUNKS;
          uint32_t r[3][16];
          auto load = [&](int i) {
            tmem_ld16x256_x4(tbase + ((uint32_t)(16 * (i & 1)) << 16) + 32 * (i >> 1), r[i % 3]);
          };
          // this lane's scales in the slot: rows lane/4 + 8i of the warp's 32,
          // and per 32-column chunk cq the column pairs 32cq + 8j + 2(lane mod 4)
          const float* sl = sring + ss * C::SSLOT_F;
          const float* colp = sl + wg * EPI_COLS + 2 * (lane & 3);
          uint64_t sbr[CHUNKS][4];
#pragma unroll
          for (int cq = 0; cq < CHUNKS; ++cq)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              sbr[cq][j] = *reinterpret_cast<const uint64_t*>(colp + 32 * cq + 8 * j);
          float sa_raw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) sa_raw[i] = sl[BN + lq * 32 + (lane >> 2) + 8 * i];
          load(0);
          load(1);
          uint64_t sal[2], sah[2];
          sal[0] = pack2(sa_raw[0], sa_raw[0]);
          sah[0] = pack2(sa_raw[1], sa_raw[1]);
          sal[1] = pack2(sa_raw[2], sa_raw[2]);
          sah[1] = pack2(sa_raw[3], sa_raw[3]);
          tmem_wait_ld16(r[0]);
          tmem_tie16(r[1]);
          if (NF <= 2) release();
#pragma unroll
          for (int i = 0; i < NF; ++i) {
            if (i + 2 < NF) load(i + 2);
            promote_cols_frag(&acc[i >> 1][8 * (i & 1)], r[i % 3], sbr[i >> 1], sal[i & 1], sah[i & 1]);
            if ((i & 1) && i + 1 < NF) {
              tmem_wait_ld16(r[(i + 1) % 3]);
              if (i + 2 < NF) tmem_tie16(r[(i + 2) % 3]);
              if (i + 2 >= NF - 1) release();
            }
          }
        } else {
          // 32-column chunks
          uint32_t cur[3][32];
          tmem_ld32_async(tbase, cur[0]);
          if (CHUNKS > 1) tmem_ld32_async(tbase + 32, cur[1]);
          tmem_wait_ld(cur[0]);
          if (CHUNKS > 1) tmem_tie32(cur[1]);
          if (CHUNKS <= 2) release();
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c) {
            if (c + 2 < CHUNKS) tmem_ld32_async(tbase + (c + 2) * 32, cur[(c + 2) % 3]);
            fma32_uniform(acc[c], cur[c % 3], s2u);
            if ((c & 1) && c + 1 < CHUNKS) {
              tmem_wait_ld(cur[(c + 1) % 3]);
              if (c + 2 < CHUNKS) tmem_tie32(cur[(c + 2) % 3]);
              if (c + 2 >= CHUNKS - 1) release();
            }
          }
        }
        return true;
      };
      for (int kb = 0; kb < nkb; kb += 2) {
        if (!block(kb, std::integral_constant<int, 0>{}) ||
            (kb + 1 < nkb && !block(kb + 1, std::integral_constant<int, 1>{}))) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      if constexpr (G > 1) {
        g = problem_of(kp, tile, local);
        tile_coords(kp.p[g], local, mt, nt);
        wrow0 = mt * TILE_M + (int)rank * BM + lq * 32;
        row = wrow0 + lane;
        col0 = nt * BN + wg * EPI_COLS;
        row_ok = row < kp.p[g].R;
      }
      const DevArgs& p = kp.p[g];
      if (COLS) {
        const int g2 = 2 * (lane & 3);
        if (p.out_fp32) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int rs = 0; rs < 2; ++rs) {
              const int r = wrow0 + (lane >> 2) + 8 * rs + 16 * h;
              if (r < p.R) {
                float* o = static_cast<float*>(p.out) + (size_t)r * p.C + col0 + g2;
#pragma unroll
                for (int cq = 0; cq < CHUNKS; ++cq)
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<float2*>(o + 32 * cq + 8 * j) = unpack2(acc[cq][8 * h + 2 * j + rs]);
              }
            }
        } else {
          uint8_t* ob = outbuf + ew * OUT_CHUNK_BYTES;
#pragma unroll
          for (int cq = 0; cq < CHUNKS; ++cq) {
            if (lane == 0) tma_store_wait_read();   // the previous chunk has left the buffer
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int rs = 0; rs < 2; ++rs)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  // row lane/4 + 8rs + 16h, granule j, bytes 4·(lane mod 4);
                  // (row/2) mod 4 = (lane/8) mod 4
                  const float2 v = unpack2(acc[cq][8 * h + 2 * j + rs]);
                  *reinterpret_cast<uint32_t*>(ob + ((lane >> 2) + 8 * rs + 16 * h) * 64 +
                                               16 * (j ^ ((lane >> 3) & 3)) + 2 * g2) = f2_to_bf2(v.x, v.y);
                }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && wrow0 < p.R) tma_store_2d(&kp.tmOut[g], smem_u32(ob), col0 + cq * 32, wrow0);
          }
        }
      } else if (p.out_fp32) {
        if (row_ok) {
          float* o = static_cast<float*>(p.out) + (size_t)row * p.C + col0;
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const float2 a = unpack2(acc[c][j]), bq = unpack2(acc[c][j + 1]);
              *reinterpret_cast<float4*>(o + c * 32 + 2 * j) = make_float4(a.x, a.y, bq.x, bq.y);
            }
        }
      } else {
        // bf16: each 32-row × 32-column chunk goes row-major (swizzled) into
        // this warp's staging buffer and leaves with one TMA store (rows >= R
        // are clipped).  With the fused quantiser (256-wide tiles: the thread's
        // 128 columns are exactly one 1×128 group of its row) the group's
        // scale comes from the bf16-rounded values and each chunk's 32 codes
        // per row leave through a 1 KB staging buffer in the (here unused)
        // column-scale ring area, so the codes are those of the 1×128
        // quantiser applied to the bf16 output.
        uint8_t* ob = outbuf + ew * OUT_CHUNK_BYTES;
        uint8_t* qb = aux + ew * 1024;
        const bool fuse_q = !PAIR && EPI_COLS == 128 && p.out_q != nullptr;
        GroupScale gq{};
        if (fuse_q) {
          float amax = 0.0f;
#pragma unroll
          for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 v = unpack2(acc[c][j]);
              const float2 f = bf2_to_f2(f2_to_bf2(v.x, v.y));
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          gq = make_scale(amax);
          if (row_ok) p.out_s[(long long)(col0 / 128) * p.ld_out_s + row] = gq.s;
        }
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
          if (lane == 0) tma_store_wait_read();   // the previous chunk's stores have left the buffers
          __syncwarp();
          uint4* dst = reinterpret_cast<uint4*>(ob + lane * 64);
          uint32_t yb[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 v = unpack2(acc[c][j]);
            yb[j] = f2_to_bf2(v.x, v.y);
          }
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            dst[(j / 4) ^ ((lane >> 1) & 3)] = make_uint4(yb[j], yb[j + 1], yb[j + 2], yb[j + 3]);
          if (fuse_q) {
            float2 f[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) f[j] = bf2_to_f2(yb[j]);
            uint32_t codes[8];
            quant_pairs<16>(f, gq, codes);
            uint4* qd = reinterpret_cast<uint4*>(qb + lane * 32);
            qd[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            qd[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && wrow0 < p.R) {
            if (p.out != nullptr) tma_store_2d(&kp.tmOut[g], smem_u32(ob), col0 + c * 32, wrow0);
            if (fuse_q) tma_store_2d(&kp.tmQ, smem_u32(qb), col0 + c * 32, wrow0);
          }
        }
      }
    }
    // stores must be complete before the CTA (and its shared memory) goes away
    if (lane == 0) tma_store_wait_all();
  }

  // ---------------- teardown ----------------
  // (a pair: neither CTA leaves, or frees TMEM, while the pair's MMAs could
  // still read its shared memory or its TMEM is still being read)
  tc_fence_before();
  if constexpr (PAIR) {
    __syncwarp();
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_ALLOC));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(C::TMEM_ALLOC));
  }
}

template <int BN_, bool COLS, int G>
__global__ void __launch_bounds__(THREADS, 1)
k_gemm_e4m3_blockscaled(const __grid_constant__ KParams<G> kp) {
  gemm_body<BN_, COLS, G, false>(kp);
}

// CTA pairs: 256 × 256 tiles over two SMs.  Per SM that is the MMA work of a
// 128 × 256 tile with half of its B operand loaded into (and read from)
// shared memory, the resource that bounds the single-CTA kernel.
template <bool COLS, int G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
k_gemm_e4m3_blockscaled_pair(const __grid_constant__ KParams<G> kp) {
  gemm_body<256, COLS, G, true>(kp);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Tensor maps go through the library's descriptor cache (a repeated call on
// the same buffers copies cached descriptors instead of encoding them again).
// 2-D bf16 output [rows, cols] stored in boxes of 32 rows × 32 columns from a
// shared-memory buffer in the 64-byte swizzle.
bool make_out_map(CUtensorMap* m, void* ptr, uint64_t cols, uint64_t rows) {
  return encode_map_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cols, rows, cols * 2, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// 2-D E4M3 codes [rows, cols] stored in boxes of 32 rows × 32 bytes, no swizzle.
bool encode_codes_map(CUtensorMap* m, void* ptr, uint64_t cols, uint64_t rows) {
  return encode_map_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_UINT8, cols, rows, cols, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// 2-D E4M3 tensor [outer, inner] (row-major, inner contiguous) loaded in
// boxes of box_outer rows × 128 bytes with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  return encode_map_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_UINT8, inner, outer, inner, (uint32_t)BK, box_outer,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Column mode reads each block's scales with bulk copies of whole 128-row and
// BN-column runs: rows and columns must fill their tiles and every scale row
// must start on a 16-byte boundary.
bool scale_ring_ok(const GemmArgs& x, int bn) {
  return x.R % BM == 0 && x.C % bn == 0 && ((uintptr_t)x.sA & 15u) == 0 && ((uintptr_t)x.sB & 15u) == 0 &&
         x.ld_sA % 4 == 0 && x.sb_k % 4 == 0;
}

}  // namespace

namespace {

template <int BN, bool COLS, int G>
cudaError_t launch_cfg(const GemmArgs* a, int count, int dev, cudaStream_t st) {
  using C = Cfg<BN>;
  auto kern = k_gemm_e4m3_blockscaled<BN, COLS, G>;
  static int ready[64] = {0};   // 0 = unchecked, 1 = ok, -1 = unusable
  if (ready[dev] == 0) {
    // The setmaxnreg split assumes the kernel launches with LAUNCH_REGS
    // registers per thread; with fewer, the promotion warps could never get theirs.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != LAUNCH_REGS) {
      ready[dev] = -1;
    } else {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      ready[dev] = 1;
    }
  }
  if (ready[dev] != 1) return cudaErrorInvalidConfiguration;
  if (count < 1 || count > G || (count > 1 && a[0].out_q != nullptr)) return cudaErrorInvalidValue;
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  KParams<G> kp;
  memset(&kp, 0, sizeof(kp));
  kp.nkb = (int)(a[0].Kc / BK);
  int tiles = 0;
  for (int g = 0; g < G; ++g) {
    if (g >= count) {
      // unused slots own no tiles
      kp.tmA[g] = kp.tmA[0];
      kp.tmB[g] = kp.tmB[0];
      kp.tmOut[g] = kp.tmOut[0];
      kp.p[g] = kp.p[0];
      kp.tile_end[g] = tiles;
      continue;
    }
    const GemmArgs& x = a[g];
    if (COLS && !scale_ring_ok(x, BN)) return cudaErrorInvalidValue;
    if (!make_map(&kp.tmA[g], x.A, (uint64_t)x.Kc, (uint64_t)x.R, BM) ||
        !make_map(&kp.tmB[g], x.B, (uint64_t)x.Kc, (uint64_t)x.C, BN))
      return cudaErrorInvalidValue;
    if (x.out_fp32 || x.out == nullptr) {
      kp.tmOut[g] = kp.tmA[g];   // unused: fp32 epilogue, or no bf16 output
    } else if (!make_out_map(&kp.tmOut[g], x.out, (uint64_t)x.C, (uint64_t)x.R)) {
      return cudaErrorInvalidValue;
    }
    DevArgs& d = kp.p[g];
    d.sA = x.sA;
    d.ld_sA = x.ld_sA;
    d.sB = x.sB;
    d.sb_j = x.sb_j;
    d.sb_k = x.sb_k;
    d.out = x.out;
    d.R = (int)x.R;
    d.C = (int)x.C;
    d.nKB = (int)(x.Kc / BK);
    if (x.Kc != a[0].Kc) return cudaErrorInvalidValue;   // one block count per launch
    d.tiles_m = (int)((x.R + BM - 1) / BM);
    d.tiles_n = (int)(x.C / BN);
    d.m_fastest = x.R <= x.C ? 1 : 0;
    d.out_fp32 = x.out_fp32 ? 1 : 0;
    d.out_q = x.out_q;
    d.out_s = x.out_s;
    d.ld_out_s = x.ld_out_s;
    d.err = err;
    d.drop_kb = x.drop_kb;
    tiles += d.tiles_m * d.tiles_n;
    kp.tile_end[g] = tiles;
  }
  if (a[0].out_q == nullptr) {
    kp.tmQ = kp.tmA[0];   // unused
  } else if (!encode_codes_map(&kp.tmQ, a[0].out_q, (uint64_t)a[0].C, (uint64_t)a[0].R)) {
    return cudaErrorInvalidValue;
  }
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  kern<<<grid, THREADS, C::SMEM_BYTES, st>>>(kp);
  return cudaGetLastError();
}


// CTA-pair launch: 256 × 256 tiles (see k_gemm_e4m3_blockscaled_pair).
template <bool COLS, int G>
cudaError_t launch_pair(const GemmArgs* a, int count, int dev, cudaStream_t st) {
  using C = Cfg<256, true>;
  auto kern = k_gemm_e4m3_blockscaled_pair<COLS, G>;
  static int ready[64] = {0};   // 0 = unchecked, 1 = ok, -1 = unusable
  if (ready[dev] == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != LAUNCH_REGS) {
      ready[dev] = -1;
    } else {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      ready[dev] = 1;
    }
  }
  if (ready[dev] != 1) return cudaErrorInvalidConfiguration;
  if (count < 1 || count > G) return cudaErrorInvalidValue;
  unsigned* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  KParams<G> kp;
  memset(&kp, 0, sizeof(kp));
  kp.nkb = (int)(a[0].Kc / BK);
  int tiles = 0;
  for (int g = 0; g < G; ++g) {
    if (g >= count) {
      kp.tmA[g] = kp.tmA[0];
      kp.tmB[g] = kp.tmB[0];
      kp.tmOut[g] = kp.tmOut[0];
      kp.p[g] = kp.p[0];
      kp.tile_end[g] = tiles;
      continue;
    }
    const GemmArgs& x = a[g];
    if (x.out_q != nullptr || x.drop_kb >= 0 || x.C % C::BN != 0) return cudaErrorInvalidValue;
    if (COLS && !scale_ring_ok(x, C::BN)) return cudaErrorInvalidValue;
    if (!make_map(&kp.tmA[g], x.A, (uint64_t)x.Kc, (uint64_t)x.R, BM) ||
        !make_map(&kp.tmB[g], x.B, (uint64_t)x.Kc, (uint64_t)x.C, C::BN / 2))
      return cudaErrorInvalidValue;
    if (x.out_fp32 || x.out == nullptr) {
      kp.tmOut[g] = kp.tmA[g];
    } else if (!make_out_map(&kp.tmOut[g], x.out, (uint64_t)x.C, (uint64_t)x.R)) {
      return cudaErrorInvalidValue;
    }
    DevArgs& d = kp.p[g];
    d.sA = x.sA;
    d.ld_sA = x.ld_sA;
    d.sB = x.sB;
    d.sb_j = x.sb_j;
    d.sb_k = x.sb_k;
    d.out = x.out;
    d.R = (int)x.R;
    d.C = (int)x.C;
    d.nKB = (int)(x.Kc / BK);
    if (x.Kc != a[0].Kc) return cudaErrorInvalidValue;   // one block count per launch
    d.tiles_m = (int)((x.R + 2 * BM - 1) / (2 * BM));
    d.tiles_n = (int)(x.C / C::BN);
    d.m_fastest = x.R <= x.C ? 1 : 0;
    d.out_fp32 = x.out_fp32 ? 1 : 0;
    d.err = err;
    d.drop_kb = -1;
    tiles += d.tiles_m * d.tiles_n;
    kp.tile_end[g] = tiles;
  }
  kp.tmQ = kp.tmA[0];
  if (tiles == 0) return cudaSuccess;
  const int pairs = num_sms() / 2;
  const int grid = 2 * (tiles < pairs ? tiles : pairs);
  kern<<<grid, THREADS, C::SMEM_BYTES, st>>>(kp);
  return cudaGetLastError();
}

// Kernel choice.  The single-CTA kernel runs every GEMM by default.  CTA
// pairs load half as much of B per SM, but on GB300 that does not raise the
// rate: with the promotion removed (a timing-only variant) both kernels run
// the 8192 x 28672 x 4096 FProp at about 2900 TFLOP/s, and with it the pair
// is slower (1950 vs 2400 FProp, 1680 vs 1880 WGrad), because each 256-column
// accumulator is handed back only when both CTAs have promoted it.
// g_gemm_path = 2 runs every GEMM the pair kernel can take on CTA pairs
// (testing and diagnosis); every output element's arithmetic (its MMA
// blocks, promotion order and rounding) is the same on either kernel.
int g_gemm_path = 0;
bool pair_possible(const GemmArgs& a) {
  return a.out_q == nullptr && a.drop_kb < 0 && a.C % 256 == 0 && a.R >= 2 * BM;
}
bool use_pair(const GemmArgs& a) { return g_gemm_path == 2 && pair_possible(a); }

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  // Column scales: 128×256 tiles (two TMEM accumulators) where the output width
  // allows, else 128×128.  Uniform scales: the tile width (256, 128 or 64
  // columns) with the fewest waves of tiles over the SMs, the narrowest of equals
  // — each CTA runs its tiles' K loops one after another, and narrower tiles put
  // more SMs on the weights.  At the training shapes that is always 256 (the
  // widest tiles read the fewest operand bytes per FLOP); a decode batch of 64
  // rows takes 64 columns on the 6144-wide QKV projection (96 tiles) but 256 on
  // the 24576-wide gate/up (96 tiles, where 128 would need two waves).  The
  // arithmetic of every output element (its MMA blocks and promotion order) does
  // not depend on the tile width.
  const bool cols = a.b_mode == BScale::kColumn;
  if (use_pair(a)) return cols ? launch_pair<true, 1>(&a, 1, dev, st) : launch_pair<false, 1>(&a, 1, dev, st);
  if (cols)
    return a.C % 256 == 0 ? launch_cfg<256, true, 1>(&a, 1, dev, st) : launch_cfg<128, true, 1>(&a, 1, dev, st);
  // the fused quantiser needs a thread's 128 columns to be a whole 1×128 group
  if (a.out_q != nullptr)
    return a.C % 256 == 0 ? launch_cfg<256, false, 1>(&a, 1, dev, st) : cudaErrorInvalidValue;
  const int64_t tiles_m = (a.R + BM - 1) / BM, sms = num_sms();
  auto waves = [&](int64_t bn) { return (tiles_m * (a.C / bn) + sms - 1) / sms; };
  int64_t bn = 128;   // C is a multiple of 128
  if (a.C % 64 == 0 && waves(64) <= waves(bn)) bn = 64;
  if (a.C % 256 == 0 && waves(256) < waves(bn)) bn = 256;
  if (bn == 256) return launch_cfg<256, false, 1>(&a, 1, dev, st);
  if (bn == 128) return launch_cfg<128, false, 1>(&a, 1, dev, st);
  return launch_cfg<64, false, 1>(&a, 1, dev, st);
}

void set_gemm_path(int mode) { g_gemm_path = (mode == 1 || mode == 2) ? mode : 0; }

cudaError_t launch_gemm_grouped(const GemmArgs* a, int count, cudaStream_t st) {
  if (count < 1 || count > MAX_GROUP) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  // one tile configuration for all problems: 256-wide tiles when every output
  // width allows, else 128-wide (an element's arithmetic does not depend on
  // the tile width, so each problem's result equals its single launch's)
  bool all256 = true, pair = true;
  for (int g = 0; g < count; ++g) {
    if (a[g].b_mode != BScale::kColumn || a[g].out_q != nullptr || a[g].out_fp32 != a[0].out_fp32)
      return cudaErrorInvalidValue;
    all256 = all256 && a[g].C % 256 == 0;
    pair = pair && pair_possible(a[g]);
  }
  if (pair && g_gemm_path == 2) return launch_pair<true, MAX_GROUP>(a, count, dev, st);
  return all256 ? launch_cfg<256, true, MAX_GROUP>(a, count, dev, st)
                : launch_cfg<128, true, MAX_GROUP>(a, count, dev, st);
}

}  // namespace jetfp8
