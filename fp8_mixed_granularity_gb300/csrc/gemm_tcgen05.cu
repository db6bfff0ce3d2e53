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
// CTA organisation (persistent, one CTA per SM, 384 threads):
//   warp 0      TMA producer: A tile 128×128 B and B tile 256×128 B per stage,
//               128-byte swizzle, 4-stage shared-memory ring.
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma
//               (M=128, N=256, K=32, E4M3×E4M3→FP32) four times per block into
//               one of two 256-column TMEM accumulators, then commits.
//   warps 2-3   idle (they complete the control warpgroup, which gives up
//               registers with setmaxnreg.dec).
//   warps 4-11  two warpgroups; warpgroup w owns output columns [128w, 128w+128)
//               of the tile and each thread one row (its TMEM lane).  They
//               tcgen05.ld the block partial, release the TMEM buffer, promote
//               it into 128 FP32 registers, and after the last block write the
//               row out as bf16 or fp32.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records an
// error word, lets copies and MMAs in flight land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"

namespace jetfp8 {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;   // 512
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                     // warps 0-3: control warpgroup
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // 384
// Register split.  The kernel is launched with LAUNCH_REGS per thread
// (384 × 168 = 64512); the control warpgroup gives registers back and the two
// promotion warpgroups take them: 128·CTRL_REGS + 256·EPI_REGS must not exceed
// the launch total, or setmaxnreg.inc would wait forever.
constexpr int LAUNCH_REGS = 168;
constexpr int CTRL_REGS = 56;
constexpr int EPI_REGS = 224;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= THREADS * LAUNCH_REGS, "register split");
constexpr uint64_t WAIT_NS = 2000000000ull;

// UMMA instruction descriptor: D = F32 (bits 4-5 = 1), A = B = E4M3 (format 0),
// both K-major, N/8 at bits 17-22, M/16 at bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct Barriers {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[ACC_BUFS];
  uint64_t tempty[ACC_BUFS];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + 1024 /*barriers*/ +
                           EPI_WARPS * 2 * 128 * 4 /*column scales*/;

struct DevArgs {
  const float* sA;
  long long ld_sA;
  const float* sB;
  long long sb_j, sb_k;
  void* out;
  int R, C, nKB, tiles_m, tiles_n;
  int b_col_mode, out_fp32;
  unsigned* err;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
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

__device__ __forceinline__ void record_abort(volatile int* abort_flag, unsigned* err) {
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
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
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate));
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
k_gemm_e4m3_blockscaled(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const DevArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + STAGES * STAGE_BYTES);
  float* colbuf = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 1024);  // [8 warps][2][128]
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_m * p.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(&bars->tfull[b], 1);
      mbar_init(&bars->tempty[b], EPI_WARPS);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&bars->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
          const int mt = tile % p.tiles_m, nt = tile / p.tiles_m;
          for (int kb = 0; kb < p.nKB; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort_flag, true)) {
              record_abort(abort_flag, p.err);
              ok = false;
              break;
            }
            uint8_t* st = smem + s * STAGE_BYTES;
            mbar_arrive_expect_tx(&bars->full[s], STAGE_BYTES);
            tma_load_2d(smem_u32(st), &tmA, &bars->full[s], kb * BK, mt * BM);
            tma_load_2d(smem_u32(st + A_BYTES), &tmB, &bars->full[s], kb * BK, nt * BN);
          }
        }
        if (!ok) {
          // let the copies still in flight land before the CTA's shared memory goes away
          const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
          for (uint32_t j = first; j < it; ++j)
            mbar_wait(&bars->full[j % STAGES], (j / STAGES) & 1u, abort_flag, false);
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        uint32_t it = 0, acc_it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
          for (int kb = 0; kb < p.nKB; ++kb, ++it, ++acc_it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            const uint32_t b = acc_it % ACC_BUFS, bph = (acc_it / ACC_BUFS) & 1u;
            if (!mbar_wait(&bars->tempty[b], bph ^ 1u, abort_flag, true) ||
                !mbar_wait(&bars->full[s], ph, abort_flag, true)) {
              record_abort(abort_flag, p.err);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_BYTES;
  #pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              umma_e4m3(tmem + b * BN, sdesc_sw128(a_addr + 32 * k), sdesc_sw128(b_addr + 32 * k),
                        k > 0 ? 1u : 0u);
            umma_commit(&bars->empty[s]);
            umma_commit(&bars->tfull[b]);
          }
        }
        // all MMAs issued by this thread complete before TMEM is released
        umma_commit(&bars->done);
        if (!mbar_wait(&bars->done, 0, abort_flag, false)) record_abort(abort_flag, p.err);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
    // ---------------- promotion + epilogue ----------------
    const int ew = warp - EPI_WARP0;
    const int wg = ew >> 2;                 // column half of the tile
    const int lq = warp & 3;                // TMEM lane quarter this warp may access
    const int row_in_tile = lq * 32 + lane;
    const uint32_t taddr_row = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(wg * 128);
    // per-warp double buffer of this half-tile's 128 column scales (column mode)
    float* cbuf = colbuf + ew * 256;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      const int mt = tile % p.tiles_m, nt = tile / p.tiles_m;
      const int row = mt * BM + row_in_tile;
      const int col0 = nt * BN + wg * 128;
      const bool row_ok = row < p.R, cols_ok = col0 < p.C;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      float4 cs_next = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.b_col_mode && cols_ok) cs_next = __ldg(reinterpret_cast<const float4*>(p.sB + col0) + lane);
      for (int kb = 0; kb < p.nKB; ++kb, ++acc_it) {
        const uint32_t b = acc_it % ACC_BUFS, bph = (acc_it / ACC_BUFS) & 1u;
        const float sa = row_ok ? __ldg(p.sA + (long long)kb * p.ld_sA + row) : 0.0f;
        float scale = sa;
        if (p.b_col_mode) {
          reinterpret_cast<float4*>(cbuf + (kb & 1) * 128)[lane] = cs_next;
          if (cols_ok && kb + 1 < p.nKB)
            cs_next = __ldg(reinterpret_cast<const float4*>(p.sB + (long long)(kb + 1) * p.sb_k + col0) + lane);
          __syncwarp();
        } else {
          const float sb = cols_ok ? __ldg(p.sB + (long long)(col0 / 128) * p.sb_j +
                                           (long long)kb * p.sb_k)
                                   : 0.0f;
          scale = sa * sb;
        }
        if (!mbar_wait(&bars->tfull[b], bph, abort_flag, true)) {
          record_abort(abort_flag, p.err);
          ok = false;
        }
        if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
        tc_fence_after();
        const float* cb = cbuf + (kb & 1) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr_row + b * BN + c * 32, r);
          tmem_wait_ld();
          if (p.b_col_mode) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c * 32 + j] = fmaf(__uint_as_float(r[j]), sa * cb[c * 32 + j], acc[c * 32 + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c * 32 + j] = fmaf(__uint_as_float(r[j]), scale, acc[c * 32 + j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tempty[b]);
      }
      if (!ok) break;
      if (row_ok && cols_ok) {
        if (p.out_fp32) {
          float* o = static_cast<float*>(p.out) + (size_t)row * p.C + col0;
#pragma unroll
          for (int j = 0; j < 128; j += 4)
            *reinterpret_cast<float4*>(o + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        } else {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (size_t)row * p.C + col0;
#pragma unroll
          for (int j = 0; j < 128; j += 8)
            *reinterpret_cast<uint4*>(o + j) =
                make_uint4(f2_to_bf2(acc[j], acc[j + 1]), f2_to_bf2(acc[j + 2], acc[j + 3]),
                           f2_to_bf2(acc[j + 4], acc[j + 5]), f2_to_bf2(acc[j + 6], acc[j + 7]));
        }
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D E4M3 tensor [outer, inner] (row-major, inner contiguous) loaded in
// boxes of box_outer rows × 128 bytes with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_gemm_e4m3_blockscaled, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  CUtensorMap ta, tb;
  if (!make_map(&ta, a.A, (uint64_t)a.Kc, (uint64_t)a.R, BM) ||
      !make_map(&tb, a.B, (uint64_t)a.Kc, (uint64_t)a.C, BN))
    return cudaErrorInvalidValue;
  DevArgs d;
  d.sA = a.sA;
  d.ld_sA = a.ld_sA;
  d.sB = a.sB;
  d.sb_j = a.sb_j;
  d.sb_k = a.sb_k;
  d.out = a.out;
  d.R = (int)a.R;
  d.C = (int)a.C;
  d.nKB = (int)(a.Kc / BK);
  d.tiles_m = (int)((a.R + BM - 1) / BM);
  d.tiles_n = (int)((a.C + BN - 1) / BN);
  d.b_col_mode = a.b_mode == BScale::kColumn ? 1 : 0;
  d.out_fp32 = a.out_fp32 ? 1 : 0;
  d.err = device_error_word();
  if (d.err == nullptr) return cudaErrorInvalidValue;
  // The setmaxnreg split assumes the kernel launches with LAUNCH_REGS registers
  // per thread; with fewer, the promotion warpgroups could never get theirs.
  static int regs_checked[64] = {0};
  if (dev < 64 && regs_checked[dev] == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, k_gemm_e4m3_blockscaled);
    if (e != cudaSuccess) return e;
    regs_checked[dev] = fa.numRegs == LAUNCH_REGS ? 1 : -1;
  }
  if (dev >= 64 || regs_checked[dev] != 1) return cudaErrorInvalidConfiguration;
  const int tiles = d.tiles_m * d.tiles_n;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  k_gemm_e4m3_blockscaled<<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, d);
  return cudaGetLastError();
}

}  // namespace jetfp8
