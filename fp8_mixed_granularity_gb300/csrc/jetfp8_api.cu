// C ABI of the jetfp8 library: argument validation, per-device set-up and the
// dispatch of each entry point to its kernel.  Declarations and the contract
// of every function are in include/jetfp8.h.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "jetfp8_common.cuh"
#include "jetfp8_internal.h"
#include "jetfp8_tma.cuh"

namespace jetfp8 {

// One error word per device, written by kernels whose bounded waits expire.
__device__ unsigned g_device_error_word;

// Scratch of jetfp8_rmsnorm_bwd_noalloc: a fixed device array (one per device,
// created with the module), so that entry point allocates nothing.  Every
// call uses the same array: calls that overlap in time (other streams, other
// host threads) race on it.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  unsigned* err_word = nullptr;
  void* scratch = nullptr;   // this device's g_noalloc_scratch
  int sms = 0;
  bool sm103 = false;
  bool ok = false;
};
DeviceInfo g_devices[kMaxDevices];

DeviceInfo* current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo* d = &g_devices[dev];
  std::call_once(d->once, [d, dev]() {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return;
    d->sms = prop.multiProcessorCount;
    d->sm103 = prop.major == 10 && prop.minor == 3;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return;
    d->err_word = static_cast<unsigned*>(p);
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_noalloc_scratch) != cudaSuccess) return;
    d->scratch = sp;
    d->ok = true;
  });
  return d->ok ? d : nullptr;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

jetfp8_status from_cuda(cudaError_t e) { return e == cudaSuccess ? JETFP8_OK : JETFP8_ERR_CUDA; }

// Validation helpers ---------------------------------------------------------
struct Check {
  jetfp8_status st = JETFP8_OK;
  // E4M3 / FP32 arrays: 16-byte aligned
  Check& ptr(const void* p, bool required = true) { return ptr_aligned(p, 16, required); }
  // bf16 tensors: 32-byte aligned
  Check& bf(const void* p, bool required = true) { return ptr_aligned(p, 32, required); }
  Check& ptr_aligned(const void* p, uintptr_t a, bool required) {
    if (st != JETFP8_OK) return *this;
    if (p == nullptr) {
      if (required) st = JETFP8_ERR_INVALID_ARG;
    } else if (!aligned(p, a)) {
      st = JETFP8_ERR_MISALIGNED;
    }
    return *this;
  }
  Check& positive(int64_t v) {
    if (st == JETFP8_OK && v <= 0) st = JETFP8_ERR_INVALID_ARG;
    return *this;
  }
  Check& mult(int64_t v, int64_t m) {
    if (st == JETFP8_OK && (v <= 0 || v % m != 0)) st = (v <= 0) ? JETFP8_ERR_INVALID_ARG : JETFP8_ERR_UNSUPPORTED_SHAPE;
    return *this;
  }
  Check& mult128(int64_t v) {
    if (st == JETFP8_OK && (v <= 0 || v % 128 != 0)) st = (v <= 0) ? JETFP8_ERR_INVALID_ARG : JETFP8_ERR_UNSUPPORTED_SHAPE;
    return *this;
  }
  // keep 32-bit index arithmetic inside the kernels safe
  Check& fits(int64_t a, int64_t b) {
    if (st == JETFP8_OK && (a > (int64_t(1) << 31) / (b > 0 ? b : 1) || a * b >= (int64_t(1) << 40)))
      st = JETFP8_ERR_UNSUPPORTED_SHAPE;
    return *this;
  }
  Check& device() {
    if (st != JETFP8_OK) return *this;
    DeviceInfo* d = current_device();
    if (d == nullptr) st = JETFP8_ERR_CUDA;
    else if (!d->sm103) st = JETFP8_ERR_UNSUPPORTED;
    return *this;
  }
};

}  // namespace

// ---------------------------------------------------------------------------
// Tensor-map encoding with a cache.  A descriptor is a pure function of its
// arguments, so a cached copy is always valid (even if the memory it names
// was freed and allocated again with the same shape).  64 entries, replaced
// round-robin, under a mutex.
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

struct MapKey {
  const void* ptr;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int dtype, swizzle, promo;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

constexpr int kMapCache = 64;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  bool used[kMapCache] = {};
  int next = 0;
};
MapCache g_map_cache;

}  // namespace

bool encode_map_2d(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));   // padding bytes take part in the comparison
  k.ptr = ptr;
  k.inner = inner;
  k.outer = outer;
  k.row_bytes = row_bytes;
  k.box_inner = box_inner;
  k.box_outer = box_outer;
  k.dtype = (int)dtype;
  k.swizzle = (int)swizzle;
  k.promo = (int)promo;
  {
    std::lock_guard<std::mutex> lock(g_map_cache.mu);
    for (int i = 0; i < kMapCache; ++i)
      if (g_map_cache.used[i] && g_map_cache.key[i] == k) {
        *out = g_map_cache.map[i];
        return true;
      }
  }
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  if (enc(out, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_cache.mu);
  const int i = g_map_cache.next;
  g_map_cache.next = (i + 1) % kMapCache;
  g_map_cache.key[i] = k;
  g_map_cache.map[i] = *out;
  g_map_cache.used[i] = true;
  return true;
}

unsigned* device_error_word() {
  DeviceInfo* d = current_device();
  return d ? d->err_word : nullptr;
}

int num_sms() {
  DeviceInfo* d = current_device();
  return (d && d->sms > 0) ? d->sms : 1;
}

bool device_is_sm103() {
  DeviceInfo* d = current_device();
  return d && d->sm103;
}

}  // namespace jetfp8

using namespace jetfp8;

namespace {

// JETFP8_LOG set to anything but "" or "0": every entry point prints its name and
// sizes to stderr when called (before its arguments are checked).
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("JETFP8_LOG");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

void log_call(const char* name, int64_t a, int64_t b = -1, int64_t c = -1) {
  if (!log_enabled()) return;
  if (c >= 0) std::fprintf(stderr, "jetfp8: %s %lld %lld %lld\n", name, (long long)a, (long long)b, (long long)c);
  else if (b >= 0) std::fprintf(stderr, "jetfp8: %s %lld %lld\n", name, (long long)a, (long long)b);
  else std::fprintf(stderr, "jetfp8: %s %lld\n", name, (long long)a);
}

}  // namespace

extern "C" {

const char* jetfp8_status_string(jetfp8_status st) {
  switch (st) {
    case JETFP8_OK: return "JETFP8_OK";
    case JETFP8_ERR_INVALID_ARG: return "JETFP8_ERR_INVALID_ARG";
    case JETFP8_ERR_UNSUPPORTED_SHAPE: return "JETFP8_ERR_UNSUPPORTED_SHAPE";
    case JETFP8_ERR_MISALIGNED: return "JETFP8_ERR_MISALIGNED";
    case JETFP8_ERR_CUDA: return "JETFP8_ERR_CUDA";
    case JETFP8_ERR_TIMEOUT: return "JETFP8_ERR_TIMEOUT";
    case JETFP8_ERR_UNSUPPORTED: return "JETFP8_ERR_UNSUPPORTED";
  }
  return "JETFP8_ERR_UNKNOWN";
}

jetfp8_status jetfp8_get_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return JETFP8_ERR_CUDA;
  if (current_device() == nullptr) return JETFP8_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word)) != cudaSuccess)
    return JETFP8_ERR_CUDA;
  if (word == 0) return JETFP8_OK;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return JETFP8_ERR_CUDA;
  return JETFP8_ERR_TIMEOUT;
}

jetfp8_status jetfp8_quant_act_1x128(const void* x_bf16, int64_t M, int64_t K, uint8_t* q,
                                     float* s, cudaStream_t stream) {
  log_call("jetfp8_quant_act_1x128", M, K);
  Check c;
  c.bf(x_bf16).ptr(q).ptr(s).positive(M).mult128(K).fits(M, K).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_quant_rowgroups(x_bf16, M, K, q, s, stream));
}

jetfp8_status jetfp8_quant_weight_128x128(const void* w_bf16, int64_t N, int64_t K, uint8_t* q,
                                          float* s, uint8_t* qT, cudaStream_t stream) {
  log_call("jetfp8_quant_weight_128x128", N, K);
  Check c;
  c.bf(w_bf16).ptr(q).ptr(s).ptr(qT, false).mult128(N).mult128(K).fits(N, K).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_quant_weight(w_bf16, N, K, q, s, qT, stream));
}

jetfp8_status jetfp8_quant_weight_grouped(int count, const void* const* w_bf16, const int64_t* N,
                                          const int64_t* K, uint8_t* const* q, float* const* s,
                                          uint8_t* const* qT, cudaStream_t stream) {
  log_call("jetfp8_quant_weight_grouped", count, 0);
  if (count < 1 || count > JETFP8_MAX_GROUP || w_bf16 == nullptr || N == nullptr || K == nullptr ||
      q == nullptr || s == nullptr)
    return JETFP8_ERR_INVALID_ARG;
  Check c;
  for (int i = 0; i < count; ++i) {
    // as jetfp8_quant_weight_128x128, problem by problem
    c.bf(w_bf16[i]).ptr(q[i]).ptr(s[i]).ptr(qT == nullptr ? nullptr : qT[i], false).mult128(N[i])
        .mult128(K[i]).fits(N[i], K[i]);
    if (c.st != JETFP8_OK) return c.st;
  }
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_quant_weight_grouped(count, w_bf16, N, K, q, s, qT, stream));
}

jetfp8_status jetfp8_requant_rowgrp_to_colgrp(const uint8_t* q, const float* s, int64_t M,
                                              int64_t K, uint8_t* qT, float* sT,
                                              cudaStream_t stream) {
  log_call("jetfp8_requant_rowgrp_to_colgrp", M, K);
  Check c;
  c.ptr(q).ptr(s).ptr(qT).ptr(sT).mult128(M).mult128(K).fits(M, K).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_requant_row2col(q, s, M, K, qT, sT, stream));
}

jetfp8_status jetfp8_quant_grad_dual(const void* dy_bf16, int64_t M, int64_t N, uint8_t* q_row,
                                     float* s_row, uint8_t* qT_col, float* sT_col,
                                     cudaStream_t stream) {
  log_call("jetfp8_quant_grad_dual", M, N);
  Check c;
  c.bf(dy_bf16).ptr(q_row).ptr(s_row).ptr(qT_col, false).ptr(sT_col, false).positive(M)
      .mult128(N).fits(M, N).device();
  if (c.st != JETFP8_OK) return c.st;
  if ((qT_col == nullptr) != (sT_col == nullptr)) return JETFP8_ERR_INVALID_ARG;
  if (qT_col != nullptr && M % 128 != 0) return JETFP8_ERR_UNSUPPORTED_SHAPE;
  return from_cuda(launch_quant_grad_dual(dy_bf16, M, N, q_row, s_row, qT_col, sT_col, stream));
}

jetfp8_status jetfp8_rmsnorm_quant(const void* x_bf16, const void* gamma_bf16, float eps,
                                   int64_t M, int64_t H, uint8_t* q, float* s, float* rstd,
                                   void* y_bf16, cudaStream_t stream) {
  log_call("jetfp8_rmsnorm_quant", M, H);
  Check c;
  c.bf(x_bf16).bf(gamma_bf16).ptr(q).ptr(s).ptr(rstd).bf(y_bf16, false).positive(M)
      .mult128(H).fits(M, H).device();
  if (c.st != JETFP8_OK) return c.st;
  if (!(eps >= 0.0f)) return JETFP8_ERR_INVALID_ARG;
  return from_cuda(launch_rmsnorm_quant(x_bf16, gamma_bf16, eps, M, H, q, s, rstd, y_bf16, stream));
}

static jetfp8_status gemm_common(const GemmArgs& g, jetfp8_out_dtype dt, cudaStream_t stream) {
  if (dt != JETFP8_OUT_BF16 && dt != JETFP8_OUT_FP32) return JETFP8_ERR_INVALID_ARG;
  return from_cuda(launch_gemm(g, stream));
}

jetfp8_status jetfp8_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream) {
  log_call("jetfp8_gemm_fprop", M, N, K);
  Check c;
  c.ptr(xq).ptr(sx).ptr(wq).ptr(sw).bf(y).positive(M).mult128(N).mult128(K).fits(M, K)
      .fits(N, K).fits(M, N).device();
  if (c.st != JETFP8_OK) return c.st;
  GemmArgs g{xq, wq, sx, round_up4(M), sw, K / 128, 1, BScale::kBlock,
             y, out_dtype == JETFP8_OUT_FP32, M, N, K};
  return gemm_common(g, out_dtype, stream);
}

jetfp8_status jetfp8_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT,
                                const float* sw, int64_t M, int64_t N, int64_t K, void* dx,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream) {
  log_call("jetfp8_gemm_dgrad", M, N, K);
  Check c;
  c.ptr(dyq).ptr(sdy).ptr(wqT).ptr(sw).bf(dx).positive(M).mult128(N).mult128(K).fits(M, N)
      .fits(N, K).fits(M, K).device();
  if (c.st != JETFP8_OK) return c.st;
  // contraction over N (block kb = n/128), output columns over K (block j/128)
  GemmArgs g{dyq, wqT, sdy, round_up4(M), sw, 1, K / 128, BScale::kBlock,
             dx, out_dtype == JETFP8_OUT_FP32, M, K, N};
  return gemm_common(g, out_dtype, stream);
}

jetfp8_status jetfp8_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                const float* sxT, int64_t M, int64_t N, int64_t K, void* dw,
                                jetfp8_out_dtype out_dtype, cudaStream_t stream) {
  log_call("jetfp8_gemm_wgrad", M, N, K);
  Check c;
  c.ptr(dyqT).ptr(sdyT).ptr(xqT).ptr(sxT).bf(dw).mult128(M).mult128(N).mult128(K).fits(M, N)
      .fits(M, K).fits(N, K).device();
  if (c.st != JETFP8_OK) return c.st;
  // contraction over tokens (block kb = m/128); per-row scale sdyT[kb][n], per-column sxT[kb][k]
  GemmArgs g{dyqT, xqT, sdyT, N, sxT, 0, K, BScale::kColumn,
             dw, out_dtype == JETFP8_OUT_FP32, N, K, M};
  return gemm_common(g, out_dtype, stream);
}

jetfp8_status jetfp8_gemm_wgrad_grouped(int count, const uint8_t* const* dyqT,
                                        const float* const* sdyT, const uint8_t* const* xqT,
                                        const float* const* sxT, int64_t M, const int64_t* N,
                                        const int64_t* K, void* const* dw,
                                        jetfp8_out_dtype out_dtype, cudaStream_t stream) {
  log_call("jetfp8_gemm_wgrad_grouped", count, M);
  if (count < 1 || count > JETFP8_MAX_GROUP || dyqT == nullptr || sdyT == nullptr ||
      xqT == nullptr || sxT == nullptr || N == nullptr || K == nullptr || dw == nullptr ||
      (out_dtype != JETFP8_OUT_BF16 && out_dtype != JETFP8_OUT_FP32))
    return JETFP8_ERR_INVALID_ARG;
  GemmArgs g[JETFP8_MAX_GROUP];
  Check c;
  c.mult128(M);
  for (int i = 0; i < count; ++i) {
    c.ptr(dyqT[i]).ptr(sdyT[i]).ptr(xqT[i]).ptr(sxT[i]).bf(dw[i]).mult128(N[i]).mult128(K[i])
        .fits(M, N[i]).fits(M, K[i]).fits(N[i], K[i]);
    if (c.st != JETFP8_OK) return c.st;
    // as jetfp8_gemm_wgrad, problem by problem
    g[i] = GemmArgs{dyqT[i], xqT[i], sdyT[i], N[i], sxT[i], 0, K[i], BScale::kColumn,
                    dw[i], out_dtype == JETFP8_OUT_FP32, N[i], K[i], M};
  }
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_gemm_grouped(g, count, stream));
}

jetfp8_status jetfp8_gemm_fprop_quant(const uint8_t* xq, const float* sx, const uint8_t* wq,
                                      const float* sw, int64_t M, int64_t N, int64_t K,
                                      void* y_bf16, uint8_t* yq, float* ys, cudaStream_t stream) {
  log_call("jetfp8_gemm_fprop_quant", M, N, K);
  Check c;
  c.ptr(xq).ptr(sx).ptr(wq).ptr(sw).bf(y_bf16, false).ptr(yq).ptr(ys).positive(M).mult128(N)
      .mult128(K).fits(M, K).fits(N, K).fits(M, N);
  // the fused quantiser needs whole 1×128 groups per 256-wide output tile
  if (c.st == JETFP8_OK && N % 256 != 0) c.st = JETFP8_ERR_UNSUPPORTED_SHAPE;
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  GemmArgs g{xq, wq, sx, round_up4(M), sw, K / 128, 1, BScale::kBlock, y_bf16, false, M, N, K};
  g.out_q = yq;
  g.out_s = ys;
  g.ld_out_s = round_up4(M);
  return from_cuda(launch_gemm(g, stream));
}

jetfp8_status jetfp8_gemm_dgrad_quant(const uint8_t* dyq, const float* sdy, const uint8_t* wqT,
                                      const float* sw, int64_t M, int64_t N, int64_t K,
                                      void* dx_bf16, uint8_t* dxq, float* dxs, cudaStream_t stream) {
  log_call("jetfp8_gemm_dgrad_quant", M, N, K);
  Check c;
  c.ptr(dyq).ptr(sdy).ptr(wqT).ptr(sw).bf(dx_bf16, false).ptr(dxq).ptr(dxs).positive(M).mult128(N)
      .mult128(K).fits(M, N).fits(N, K).fits(M, K);
  // the fused quantiser needs whole 1×128 groups per 256-wide output tile
  if (c.st == JETFP8_OK && K % 256 != 0) c.st = JETFP8_ERR_UNSUPPORTED_SHAPE;
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  GemmArgs g{dyq, wqT, sdy, round_up4(M), sw, 1, K / 128, BScale::kBlock, dx_bf16, false, M, K, N};
  g.out_q = dxq;
  g.out_s = dxs;
  g.ld_out_s = round_up4(M);
  return from_cuda(launch_gemm(g, stream));
}

jetfp8_status jetfp8_test_gemm_fprop_drop_block(const uint8_t* xq, const float* sx,
                                               const uint8_t* wq, const float* sw, int64_t M,
                                               int64_t N, int64_t K, void* y, int drop_kb,
                                               cudaStream_t stream) {
  log_call("jetfp8_test_gemm_fprop_drop_block", M, N, K);
  Check c;
  c.ptr(xq).ptr(sx).ptr(wq).ptr(sw).bf(y).positive(M).mult128(N).mult128(K).fits(M, K)
      .fits(N, K).fits(M, N);
  if (c.st == JETFP8_OK && (drop_kb < 0 || drop_kb >= K / 128)) c.st = JETFP8_ERR_INVALID_ARG;
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  GemmArgs g{xq, wq, sx, round_up4(M), sw, K / 128, 1, BScale::kBlock, y, false, M, N, K};
  g.drop_kb = drop_kb;
  return from_cuda(launch_gemm(g, stream));
}

jetfp8_status jetfp8_test_set_gemm_path(int mode) {
  log_call("jetfp8_test_set_gemm_path", mode);
  if (mode < 0 || mode > 2) return JETFP8_ERR_INVALID_ARG;
  set_gemm_path(mode);
  return JETFP8_OK;
}

size_t jetfp8_nvfp4_scale_bytes(int64_t R, int64_t K) {
  if (R <= 0 || K <= 0 || K % 64 != 0) return 0;
  return nvfp4_scale_bytes(R, K);
}

jetfp8_status jetfp8_quant_nvfp4(const void* x_bf16, int64_t R, int64_t K, uint8_t* q, uint8_t* sf,
                                 float* g, cudaStream_t stream) {
  log_call("jetfp8_quant_nvfp4", R, K);
  Check c;
  c.bf(x_bf16).ptr(q).ptr(sf).ptr(g).positive(R).mult(K, 64).fits(R, K).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_quant_nvfp4(x_bf16, R, K, q, sf, g, stream));
}

jetfp8_status jetfp8_gemm_fprop_nvfp4(const uint8_t* xq, const uint8_t* xsf, const float* gx,
                                      const uint8_t* wq, const uint8_t* wsf, const float* gw, int64_t M,
                                      int64_t N, int64_t K, void* y_bf16, cudaStream_t stream) {
  log_call("jetfp8_gemm_fprop_nvfp4", M, N, K);
  Check c;
  c.ptr(xq).ptr(xsf).ptr(gx).ptr(wq).ptr(wsf).ptr(gw).ptr(y_bf16).positive(M).mult(N, 256).mult(K, 256)
      .fits(M, K).fits(N, K).fits(M, N).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_gemm_nvfp4(xq, xsf, gx, wq, wsf, gw, M, N, K, y_bf16, stream));
}

size_t jetfp8_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t H) {
  if (M <= 0 || H <= 0) return 0;
  return rmsnorm_bwd_workspace_bytes(M, H);
}

jetfp8_status jetfp8_rmsnorm_bwd(const void* x_bf16, const void* gamma_bf16, const float* rstd,
                                 const void* dy_bf16, int64_t M, int64_t H, void* dx_bf16,
                                 float* dgamma, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  log_call("jetfp8_rmsnorm_bwd", M, H);
  Check c;
  c.bf(x_bf16).bf(gamma_bf16).ptr(rstd).bf(dy_bf16).bf(dx_bf16).ptr(dgamma).ptr(workspace)
      .positive(M).mult128(H).fits(M, H);
  if (c.st == JETFP8_OK && workspace_bytes < rmsnorm_bwd_workspace_bytes(M, H))
    c.st = JETFP8_ERR_INVALID_ARG;
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_rmsnorm_bwd(x_bf16, gamma_bf16, rstd, dy_bf16, M, H, dx_bf16, dgamma,
                                      static_cast<float*>(workspace), stream));
}

jetfp8_status jetfp8_rmsnorm_bwd_noalloc(const void* x_bf16, const void* gamma_bf16, const float* rstd,
                                         const void* dy_bf16, int64_t M, int64_t H, void* dx_bf16,
                                         float* dgamma, cudaStream_t stream) {
  log_call("jetfp8_rmsnorm_bwd_noalloc", M, H);
  Check c;
  c.bf(x_bf16).bf(gamma_bf16).ptr(rstd).bf(dy_bf16).bf(dx_bf16).ptr(dgamma).positive(M).mult128(H)
      .fits(M, H);
  if (c.st == JETFP8_OK && rmsnorm_bwd_workspace_bytes(M, H) > kNoAllocScratchBytes)
    c.st = JETFP8_ERR_UNSUPPORTED_SHAPE;
  c.device();
  if (c.st != JETFP8_OK) return c.st;
  // every partial sum the kernels read is written first in the same call, so
  // nothing in the scratch needs clearing
  DeviceInfo* d = current_device();
  if (d == nullptr || d->scratch == nullptr) return JETFP8_ERR_CUDA;
  return from_cuda(launch_rmsnorm_bwd(x_bf16, gamma_bf16, rstd, dy_bf16, M, H, dx_bf16, dgamma,
                                      static_cast<float*>(d->scratch), stream));
}

jetfp8_status jetfp8_swiglu_quant(const void* gu_bf16, int64_t M, int64_t I, uint8_t* q, float* s,
                                  void* h_bf16, cudaStream_t stream) {
  log_call("jetfp8_swiglu_quant", M, I);
  Check c;
  c.bf(gu_bf16).ptr(q).ptr(s).bf(h_bf16, false).positive(M).mult128(I).fits(M, 2 * I).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_swiglu_quant(gu_bf16, M, I, q, s, h_bf16, stream));
}

jetfp8_status jetfp8_swiglu_bwd(const void* gu_bf16, const void* dh_bf16, int64_t M, int64_t I,
                                void* dgu_bf16, cudaStream_t stream) {
  log_call("jetfp8_swiglu_bwd", M, I);
  Check c;
  c.bf(gu_bf16).bf(dh_bf16).bf(dgu_bf16).positive(M).mult128(I).fits(M, 2 * I).device();
  if (c.st != JETFP8_OK) return c.st;
  return from_cuda(launch_swiglu_bwd(gu_bf16, dh_bf16, M, I, dgu_bf16, stream));
}

}  // extern "C"
